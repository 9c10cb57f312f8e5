"""GPU parity of the backward (the gradients for training) against the fp64 oracle's reverse
mode, through the C ABI: the chunked kda_chunk_bwd (chunk = 64) and the token-serial
kda_bwd (chunk = 1).

The loss is L = sum_t <do_t, o_t> + <dS_T, S_T> with random cotangents.  Tolerance, per
gradient: rel-L2 <= 2e-3 (the forward's bar) and max-abs <= 1e-2 of the gradient's own
largest magnitude (gradients are not O(1) like the outputs: they sum over many tokens)."""
import numpy as np
import pytest
import torch

from kda_testutil import REL_L2, batch_heads, errors, np64, packed_heads
from oracle import oracle

pytestmark = pytest.mark.gpu


def _close(got, ref, what):
    rel, mx = errors(got, ref)
    scale = max(1.0, float(np.abs(ref).max()) if np.size(ref) else 1.0)
    assert rel <= REL_L2 and mx <= 1e-2 * scale, f"{what}: rel-L2 {rel:.3e}, max-abs {mx:.3e} (scale {scale:.2f})"


def _bcast(la_h, dk=128):
    return la_h.unsqueeze(-1).expand(*la_h.shape, dk).contiguous()


def _oracle_grads(x, la_full, do, dSf, pairs):
    S0 = None if x["init_state"] is None else np.stack([np64(x["init_state"][b, h]) for b, h in pairs])
    dsf = None if dSf is None else np.stack([np64(dSf[b, h]) for b, h in pairs])
    return oracle.recurrent_bwd(batch_heads(x["q"], pairs), batch_heads(x["k"], pairs), batch_heads(x["v"], pairs),
                                batch_heads(la_full, pairs), batch_heads(x["beta"], pairs), S0,
                                batch_heads(do, pairs), dsf)


CHUNKS = pytest.mark.parametrize("chunk", [64, 1])


@CHUNKS
@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T", [1, 7, 64, 65, 200])
def test_bwd_parity(T, in_dtype, chunk):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, H = 2, 2
    x = synth.prefill_inputs(B, T, H, seed=5100 + T, device="cuda", init="normal", in_dtype=in_dtype)
    g = torch.Generator(device="cuda").manual_seed(5200 + T)
    do = torch.randn(B, T, H, 128, generator=g, device="cuda")
    dSf = torch.randn(B, H, 128, 128, generator=g, device="cuda")
    got = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], dSf, chunk=chunk)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    pairs = [(b, h) for b in range(B) for h in range(H)]
    ref = _oracle_grads(x, x["log_alpha"], do, dSf, pairs)
    for name in ("dq", "dk", "dv", "dlog_alpha", "dbeta"):
        _close(batch_heads(got[name], pairs), ref[name], name)
    _close(np.stack([np64(got["d_init"][b, h]) for b, h in pairs]), ref["dS0"], "d_init")


@CHUNKS
@pytest.mark.parametrize("gate", [1, 2], ids=["head", "none"])
def test_bwd_scalar_and_no_gate(gate, chunk):
    """Gated DeltaNet's per-head gate gets the sum over key channels of the per-channel
    gradient of the broadcast gate; DeltaNet has no gate gradient."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, T, H = 1, 300, 3
    x = synth.prefill_inputs(B, T, H, seed=5301, device="cuda", init="normal")
    la_h = synth.head_gates((B, T), H, seed=5302, device="cuda") if gate == 1 else None
    g = torch.Generator(device="cuda").manual_seed(5303)
    do = torch.randn(B, T, H, 128, generator=g, device="cuda")
    got = kda.kda_bwd(x["q"], x["k"], x["v"], la_h, x["beta"], do, x["init_state"], None, gate=gate, chunk=chunk)
    torch.cuda.synchronize()
    pairs = [(0, h) for h in range(H)]
    la_full = _bcast(la_h) if gate == 1 else torch.zeros_like(x["log_alpha"])
    ref = _oracle_grads(x, la_full, do, None, pairs)
    for name in ("dq", "dk", "dv", "dbeta"):
        _close(batch_heads(got[name], pairs), ref[name], name)
    _close(np.stack([np64(got["d_init"][b, h]) for b, h in pairs]), ref["dS0"], "d_init")
    if gate == 1:
        _close(batch_heads(got["dlog_alpha"], pairs), ref["dlog_alpha"].sum(axis=-1), "dlog_alpha (per head)")
    else:
        assert got["dlog_alpha"] is None


@CHUNKS
def test_bwd_varlen(chunk):
    """Packed sequences (one empty, ragged tails): each sequence's gradients against the oracle;
    an empty sequence passes its final-state cotangent through to its initial state."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    lengths, H = [300, 0, 65, 513], 2
    xv = synth.varlen_inputs(lengths, H, seed=5401, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(5402)
    do = torch.randn(xv["q"].shape[0], H, 128, generator=g, device="cuda")
    dSf = torch.randn(len(lengths), H, 128, 128, generator=g, device="cuda")
    got = kda.kda_bwd(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], do, xv["init_states"], dSf,
                      cu_seqlens=xv["cu_seqlens"], chunk=chunk)
    torch.cuda.synchronize()
    cu = xv["cu_seqlens"].tolist()
    heads = [0, 1]
    for s in range(len(lengths)):
        a, b = cu[s], cu[s + 1]
        if a == b:
            assert torch.equal(got["d_init"][s], dSf[s])
            continue
        ref = oracle.recurrent_bwd(packed_heads(xv["q"], a, b, heads), packed_heads(xv["k"], a, b, heads),
                                   packed_heads(xv["v"], a, b, heads), packed_heads(xv["log_alpha"], a, b, heads),
                                   packed_heads(xv["beta"], a, b, heads), np64(xv["init_states"][s]),
                                   packed_heads(do, a, b, heads), np64(dSf[s]))
        for name in ("dq", "dk", "dv", "dlog_alpha", "dbeta"):
            _close(packed_heads(got[name], a, b, heads), ref[name], f"seq {s} {name}")
        _close(np64(got["d_init"][s]), ref["dS0"], f"seq {s} d_init")


@CHUNKS
def test_bwd_slow_gates_long(chunk):
    """Slow gates keep gradients flowing back over thousands of tokens and across many
    checkpoint segments: B=1, H=2, T=2048."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(1, 2048, 2, seed=5501, device="cuda", init="normal", gate="slow")
    g = torch.Generator(device="cuda").manual_seed(5502)
    do = torch.randn(1, 2048, 2, 128, generator=g, device="cuda")
    got = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], chunk=chunk)
    torch.cuda.synchronize()
    pairs = [(0, 0), (0, 1)]
    ref = _oracle_grads(x, x["log_alpha"], do, None, pairs)
    for name in ("dq", "dk", "dv", "dlog_alpha", "dbeta"):
        _close(batch_heads(got[name], pairs), ref[name], name)
    _close(np.stack([np64(got["d_init"][b, h]) for b, h in pairs]), ref["dS0"], "d_init")


@CHUNKS
def test_bwd_deterministic(chunk):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(2, 333, 3, seed=5601, device="cuda", init="normal")
    do = torch.randn(2, 333, 3, 128, generator=torch.Generator(device="cuda").manual_seed(1), device="cuda")
    g1 = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], chunk=chunk)
    g2 = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], chunk=chunk)
    torch.cuda.synchronize()
    for name in g1:
        assert torch.equal(g1[name], g2[name]), name


def test_chunk_bwd_beyond_the_fp32_bound():
    """A half-chunk whose summed log-decay is below -80 cannot be factored in fp32: the chunked
    backward flags the unit and recomputes it with the token-serial backward inside the same call
    (no status), and the result matches the oracle and the chunk = 1 call."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(1, 64, 1, seed=5701, device="cuda", init="normal")
    la = x["log_alpha"].clone()
    la[0, 40:44] = -30.0  # rows 32..63 of the chunk sum to about -120
    do = torch.randn(1, 64, 1, 128, generator=torch.Generator(device="cuda").manual_seed(5702), device="cuda")
    assert kda.kda_get_device_status() == 0
    got = kda.kda_bwd(x["q"], x["k"], x["v"], la, x["beta"], do, x["init_state"], chunk=64)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    one = kda.kda_bwd(x["q"], x["k"], x["v"], la, x["beta"], do, x["init_state"], chunk=1)
    torch.cuda.synchronize()
    ref = _oracle_grads(dict(x, log_alpha=la), la, do, None, [(0, 0)])
    for name in ("dq", "dk", "dv", "dbeta"):
        _close(batch_heads(got[name], [(0, 0)]), ref[name], name)
        assert torch.equal(got[name], one[name]), name  # the same token-serial kernel computed both


def test_chunk_bwd_workspace_and_bad_chunk():
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(1, 100, 1, seed=5801, device="cuda")
    do = torch.zeros(1, 100, 1, 128, device="cuda")
    with pytest.raises(kda.KdaError):
        kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, chunk=16)
    need = kda.kda_workspace_size(kda.KDA_OP_CHUNK_BWD, 1, 100, 1, chunk=64)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError):
        kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, chunk=64, workspace=small)


def test_chunk_bwd_full_size_sampled():
    """The timed backward configuration (B=4, H=32, T=8192, bf16 inputs, S0 ~ N(0,0.02), chunk 64):
    two sampled (sequence, head) pairs over all 8192 tokens against the oracle."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, T, H = 4, 8192, 32
    x = synth.prefill_inputs(B, T, H, seed=synth.SEED_BASE + 1, device="cuda", init="normal")
    do = torch.randn(B, T, H, 128, generator=torch.Generator(device="cuda").manual_seed(7), device="cuda")
    got = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], chunk=64)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    pairs = [(1, 5), (3, 30)]
    ref = _oracle_grads(x, x["log_alpha"], do, None, pairs)
    for name in ("dq", "dk", "dv", "dlog_alpha", "dbeta"):
        _close(batch_heads(got[name], pairs), ref[name], name)
    _close(np.stack([np64(got["d_init"][b, h]) for b, h in pairs]), ref["dS0"], "d_init")


@CHUNKS
def test_bwd_no_tokens(chunk):
    """T = 0: no gradient but the initial state's, which equals the final state's cotangent."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(2, 0, 3, seed=5901, device="cuda", init="normal")
    dSf = torch.randn(2, 3, 128, 128, generator=torch.Generator(device="cuda").manual_seed(5902), device="cuda")
    do = torch.zeros(2, 0, 3, 128, device="cuda")
    got = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], dSf, chunk=chunk)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    assert torch.equal(got["d_init"], dSf)
    assert got["dq"].numel() == 0 and got["dbeta"].numel() == 0
