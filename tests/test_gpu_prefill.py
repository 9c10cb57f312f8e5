"""GPU parity of kda_chunk_fwd against the fp64 oracle (through the C ABI).

Sizes span several 64-token chunks and ragged tails; the full-size workloads
(B=4,H=32,T=8192 and B=1,H=96,T=131072) are checked on sampled heads the
oracle computes one by one."""
import numpy as np
import pytest
import torch

from kda_testutil import assert_close, batch_heads, errors, np64
from oracle import oracle

pytestmark = pytest.mark.gpu
CHUNKS = [64, 1]


def _ref(x, pairs):
    S0 = None if x["init_state"] is None else np.stack([np64(x["init_state"][b, h]) for b, h in pairs])
    return oracle.recurrent(batch_heads(x["q"], pairs), batch_heads(x["k"], pairs), batch_heads(x["v"], pairs),
                            batch_heads(x["log_alpha"], pairs), batch_heads(x["beta"], pairs), S0)


def _check(x, out, fin, pairs, what):
    ro, rs = _ref(x, pairs)
    eo = assert_close(batch_heads(out, pairs), ro, what + " out")
    es = assert_close(np.stack([np64(fin[b, h]) for b, h in pairs]), rs, what + " state")
    return eo, es


@pytest.mark.parametrize("chunk", CHUNKS)
def test_tiny_fp32(chunk):
    """B=1, H=2, T=256, fp32 everything, zero initial state (the oracle-sized case)."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(1, 256, 2, seed=synth.SEED_BASE + 0, device="cuda", in_dtype=torch.float32)
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, chunk=chunk)
    torch.cuda.synchronize()
    _check(x, out, fin, [(0, 0), (0, 1)], "tiny")
    assert kda.kda_get_device_status() == 0


@pytest.mark.parametrize("chunk", CHUNKS)
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 333])
def test_ragged_lengths(chunk, T):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(2, T, 3, seed=1000 + T, device="cuda", init="normal")
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"], chunk=chunk)
    torch.cuda.synchronize()
    _check(x, out, fin, [(b, h) for b in range(2) for h in range(3)], f"T={T}")


@pytest.mark.parametrize("chunk", CHUNKS)
def test_slow_decay_carry(chunk):
    """Slow gates keep the initial state and the inter-chunk carry visible for thousands of tokens."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(1, 4096, 4, seed=77, device="cuda", init="normal", gate="slow")
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"], chunk=chunk)
    torch.cuda.synchronize()
    _check(x, out, fin, [(0, h) for h in range(4)], "slow")


@pytest.mark.parametrize("chunk", CHUNKS)
def test_bf16_output(chunk):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(2, 512, 2, seed=5, device="cuda", init="normal")
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"], chunk=chunk,
                                 out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16
    _check(x, out, fin, [(b, h) for b in range(2) for h in range(2)], "bf16 out")


@pytest.mark.parametrize("chunk", CHUNKS)
def test_empty_and_aliasing(chunk):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(2, 0, 3, seed=9, device="cuda", init="normal")
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"], chunk=chunk)
    torch.cuda.synchronize()
    assert out.shape == (2, 0, 3, 128) and torch.equal(fin, x["init_state"])
    # init_state aliasing final_state: the state is advanced in place
    x = synth.prefill_inputs(1, 130, 2, seed=10, device="cuda", init="normal")
    ref_out, ref_fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                                         chunk=chunk)
    st = x["init_state"].clone()
    out2, fin2 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], st, final_state=st,
                                   chunk=chunk)
    torch.cuda.synchronize()
    assert torch.equal(out2, ref_out) and torch.equal(st, ref_fin)


@pytest.mark.parametrize("chunk", CHUNKS)
def test_deterministic_and_split_resume(chunk):
    """Bit-reproducible, and resuming at a chunk-aligned split equals the unsplit run bit for bit."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(2, 384, 3, seed=11, device="cuda", init="normal")
    args = (x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"])
    o1, f1 = kda.kda_chunk_fwd(*args, chunk=chunk)
    o2, f2 = kda.kda_chunk_fwd(*args, chunk=chunk)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    cut = 192
    part = lambda t, a, b: t[:, a:b].contiguous()
    oa, fa = kda.kda_chunk_fwd(*(part(t, 0, cut) for t in args[:5]), x["init_state"], chunk=chunk)
    ob, fb = kda.kda_chunk_fwd(*(part(t, cut, 384) for t in args[:5]), fa, chunk=chunk)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([oa, ob], dim=1), o1) and torch.equal(fb, f1)


@pytest.mark.parametrize("chunk", CHUNKS)
def test_mid_prefill_full_size_sampled(chunk):
    """B=4, H=32, T=8192, bf16 q/k/v, N(0,0.02) initial states: 12 sampled heads."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(4, 8192, 32, seed=synth.SEED_BASE + 1, device="cuda", init="normal")
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"], chunk=chunk)
    torch.cuda.synchronize()
    pairs = [(0, 0), (3, 31), (1, 7), (2, 16), (0, 30), (3, 1), (1, 25), (2, 2), (0, 13), (1, 19), (2, 28), (3, 9)]
    _check(x, out, fin, pairs, "mid")


@pytest.mark.parametrize("chunk", [64])
def test_long_prefill_full_size_sampled(chunk):
    """B=1, H=96, T=131072 (128K), zero initial state, in the launch configuration the bench times:
    4 sampled heads over the whole sequence, plus a property that holds at any size
    (finite outputs everywhere)."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(1, 131072, 96, seed=synth.SEED_BASE + 2, device="cuda")
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, chunk=chunk)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(fin).all())
    x["init_state"] = None
    _check(x, out, fin, [(0, 0), (0, 95), (0, 42), (0, 61)], "long")
    assert kda.kda_get_device_status() == 0


def test_steep_decay_is_recomputed():
    """A decay too steep for the fp16 operands of the chunk = 64 path (log alpha = -1 per
    token: -31 over a half chunk) needs no status and no chunk = 1 from the caller: the
    units are recomputed by the token-serial pass inside the same call."""
    import kda_recurrent_state_gb300 as kda

    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(1, 128, 2, seed=synth.SEED_BASE + 9, device="cuda")
    steep = torch.full_like(x["log_alpha"], -1.0)
    assert kda.kda_get_device_status() == 0
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], steep, x["beta"], None, chunk=64)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    pairs = [(0, 0), (0, 1)]
    ro, rs = oracle.recurrent(batch_heads(x["q"], pairs), batch_heads(x["k"], pairs), batch_heads(x["v"], pairs),
                              batch_heads(steep, pairs), batch_heads(x["beta"], pairs), None)
    assert_close(batch_heads(out, pairs), ro, "steep decay, out")
    assert_close(np.stack([np64(fin[b, h]) for b, h in pairs]), rs, "steep decay, state")