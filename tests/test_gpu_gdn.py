"""GPU parity of the scalar-gate entry points (kda_gdn_chunk_fwd, kda_gdn_varlen_fwd,
kda_gdn_decode_step) against the fp64 oracle, through the C ABI.

Gated DeltaNet decays a head's whole state by one scalar per token; DeltaNet has no
decay.  Both are the KDA recurrence with the per-channel gate replaced by a constant
across key channels, so the oracle is the same per-token recurrence fed the scalar
broadcast over the channels (or zeros).  The same broadcast fed to the per-channel
entry points must give the scalar entry points' results bit for bit: both evaluate
the same arithmetic on the same values."""
import numpy as np
import pytest
import torch

from kda_testutil import assert_close, batch_heads, np64, packed_heads
from oracle import oracle

pytestmark = pytest.mark.gpu
CHUNKS = [64, 1]


def _bcast(la_h, dk=128):
    """[.., H] scalar gates -> [.., H, dk] per-channel gates with equal channels."""
    return la_h.unsqueeze(-1).expand(*la_h.shape, dk).contiguous()


def _inputs(B, T, H, seed, gate, deltanet, init="normal"):
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(B, T, H, seed=seed, device="cuda", init=init, gate=gate)
    la_h = None if deltanet else synth.head_gates((B, T), H, seed=seed + 1, device="cuda", gate=gate)
    return x, la_h


def _oracle(x, la_h, pairs):
    la = torch.zeros_like(x["log_alpha"]) if la_h is None else _bcast(la_h)
    S0 = None if x["init_state"] is None else np.stack([np64(x["init_state"][b, h]) for b, h in pairs])
    return oracle.recurrent(batch_heads(x["q"], pairs), batch_heads(x["k"], pairs), batch_heads(x["v"], pairs),
                            batch_heads(la, pairs), batch_heads(x["beta"], pairs), S0)


@pytest.mark.parametrize("chunk", CHUNKS)
@pytest.mark.parametrize("deltanet", [False, True], ids=["gdn", "deltanet"])
@pytest.mark.parametrize("T", [1, 64, 200, 1000])
def test_chunk_parity(chunk, deltanet, T):
    import kda_recurrent_state_gb300 as kda

    x, la_h = _inputs(2, T, 3, seed=3000 + T, gate="config", deltanet=deltanet)
    out, fin = kda.kda_gdn_chunk_fwd(x["q"], x["k"], x["v"], la_h, x["beta"], x["init_state"], chunk=chunk)
    torch.cuda.synchronize()
    pairs = [(b, h) for b in range(2) for h in range(3)]
    ro, rs = _oracle(x, la_h, pairs)
    assert_close(batch_heads(out, pairs), ro, "out")
    assert_close(np.stack([np64(fin[b, h]) for b, h in pairs]), rs, "state")
    assert kda.kda_get_device_status() == 0


@pytest.mark.parametrize("chunk", CHUNKS)
def test_slow_gate_carry(chunk):
    """Slow scalar gates keep the initial state and the chunk carry visible for thousands of tokens."""
    import kda_recurrent_state_gb300 as kda

    x, la_h = _inputs(1, 4096, 2, seed=91, gate="slow", deltanet=False)
    out, fin = kda.kda_gdn_chunk_fwd(x["q"], x["k"], x["v"], la_h, x["beta"], x["init_state"], chunk=chunk)
    torch.cuda.synchronize()
    pairs = [(0, 0), (0, 1)]
    ro, rs = _oracle(x, la_h, pairs)
    assert_close(batch_heads(out, pairs), ro, "out")
    assert_close(np.stack([np64(fin[b, h]) for b, h in pairs]), rs, "state")


@pytest.mark.parametrize("chunk", CHUNKS)
@pytest.mark.parametrize("deltanet", [False, True], ids=["gdn", "deltanet"])
@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
def test_equals_channel_path_with_equal_channels(chunk, deltanet, in_dtype):
    """The scalar-gate path and the per-channel path fed the broadcast gate agree bit for bit."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(2, 777, 3, seed=4242, device="cuda", init="normal", in_dtype=in_dtype)
    la_h = None if deltanet else synth.head_gates((2, 777), 3, seed=4243, device="cuda")
    la_c = torch.zeros_like(x["log_alpha"]) if deltanet else _bcast(la_h)
    o1, f1 = kda.kda_gdn_chunk_fwd(x["q"], x["k"], x["v"], la_h, x["beta"], x["init_state"], chunk=chunk)
    o2, f2 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], la_c, x["beta"], x["init_state"], chunk=chunk)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_varlen_snapshots_and_parity():
    """Packed sequences with scalar gates: every sequence equals its own kda_gdn_chunk_fwd run
    bit for bit, snapshots equal the final states of the prefixes, sampled heads match the oracle."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    lengths = [300, 64, 1, 1000, 0, 513]
    H = 2
    xv = synth.varlen_inputs(lengths, H, seed=515, device="cuda")
    la_h = synth.head_gates((int(sum(lengths)),), H, seed=516, device="cuda")
    out, fin, snaps = kda.kda_gdn_varlen_fwd(xv["q"], xv["k"], xv["v"], la_h, xv["beta"], xv["cu_seqlens"],
                                             xv["init_states"], snapshot_interval=256)
    torch.cuda.synchronize()
    cu = xv["cu_seqlens"].tolist()
    off = kda.kda_snapshot_offsets(cu, 256).tolist()
    for s, L in enumerate(lengths):
        a, b = cu[s], cu[s + 1]
        sl = lambda t: t[a:b].unsqueeze(0).contiguous()
        o1, f1 = kda.kda_gdn_chunk_fwd(sl(xv["q"]), sl(xv["k"]), sl(xv["v"]), sl(la_h), sl(xv["beta"]),
                                       xv["init_states"][s:s + 1].contiguous())
        assert torch.equal(out[a:b], o1[0]) and torch.equal(fin[s], f1[0]), f"sequence {s}"
        for m in range(L // 256):
            _, fp = kda.kda_gdn_chunk_fwd(sl(xv["q"])[:, :256 * (m + 1)].contiguous(),
                                          sl(xv["k"])[:, :256 * (m + 1)].contiguous(),
                                          sl(xv["v"])[:, :256 * (m + 1)].contiguous(),
                                          sl(la_h)[:, :256 * (m + 1)].contiguous(),
                                          sl(xv["beta"])[:, :256 * (m + 1)].contiguous(),
                                          xv["init_states"][s:s + 1].contiguous())
            assert torch.equal(snaps[off[s] + m], fp[0]), f"snapshot {m} of sequence {s}"
    a, b = cu[3], cu[4]
    heads = [0, 1]
    la = _bcast(la_h)
    ro, rs = oracle.recurrent(packed_heads(xv["q"], a, b, heads), packed_heads(xv["k"], a, b, heads),
                              packed_heads(xv["v"], a, b, heads), packed_heads(la, a, b, heads),
                              packed_heads(xv["beta"], a, b, heads), np64(xv["init_states"][3]))
    assert_close(packed_heads(out, a, b, heads), ro, "varlen out")
    assert_close(np64(fin[3]), rs, "varlen state")
    assert kda.kda_get_device_status() == 0


@pytest.mark.parametrize("deltanet", [False, True], ids=["gdn", "deltanet"])
def test_decode(deltanet):
    """Decode steps with a scalar gate (or none) against the oracle, and bit for bit against the
    per-channel decode fed the broadcast gate."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, H, steps = 4, 3, 5
    d = synth.decode_inputs(B, H, seed=613, steps=steps, device="cuda")
    la_h = None if deltanet else synth.head_gates((steps, B), H, seed=614, device="cuda")
    s1, s2 = d["state"].clone(), d["state"].clone()
    outs = []
    for s in range(steps):
        g = None if deltanet else la_h[s]
        gc = torch.zeros_like(d["log_alpha"][s]) if deltanet else _bcast(la_h[s])
        o1 = kda.kda_gdn_decode_step(d["q"][s], d["k"][s], d["v"][s], g, d["beta"][s], s1)
        o2 = kda.kda_decode_step(d["q"][s], d["k"][s], d["v"][s], gc, d["beta"][s], s2)
        outs.append(o1)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
    assert torch.equal(s1, s2)
    pairs = [(b, h) for b in range(B) for h in range(H)]
    la = torch.zeros(steps, B, H, 128, device="cuda") if deltanet else _bcast(la_h)
    col = lambda t, b, h: np64(t[:steps, b, h])
    ro, rs = oracle.recurrent(np.stack([col(d["q"], b, h) for b, h in pairs]),
                              np.stack([col(d["k"], b, h) for b, h in pairs]),
                              np.stack([col(d["v"], b, h) for b, h in pairs]),
                              np.stack([col(la, b, h) for b, h in pairs]),
                              np.stack([col(d["beta"], b, h) for b, h in pairs]),
                              np.stack([np64(d["state"][b, h]) for b, h in pairs]))
    got = np.stack([np.stack([np64(outs[s][b, h]) for s in range(steps)]) for b, h in pairs])
    assert_close(got, ro, "decode out")
    assert_close(np.stack([np64(s1[b, h]) for b, h in pairs]), rs, "decode state")


def test_full_size_sampled():
    """B=1, H=96, T=131072 with scalar gates (the long-prefill shape): the first 4096 outputs of
    two heads, and one head's whole sequence (outputs of its last 4096 tokens, final state),
    against the oracle."""
    import kda_recurrent_state_gb300 as kda

    x, la_h = _inputs(1, 131072, 96, seed=7001, gate="config", deltanet=False, init="zero")
    out, fin = kda.kda_gdn_chunk_fwd(x["q"], x["k"], x["v"], la_h, x["beta"], None)
    torch.cuda.synchronize()
    t_s = 4096
    xs = {k: (v[:, :t_s] if v is not None else v) for k, v in x.items()}
    pairs = [(0, 0), (0, 95)]
    ro, _ = _oracle(xs, la_h[:, :t_s], pairs)
    assert_close(batch_heads(out[:, :t_s], pairs), ro, "prefix out")
    ro_all, rs_all = _oracle(x, la_h, [(0, 17)])
    assert_close(batch_heads(out[:, -t_s:], [(0, 17)]), ro_all[:, -t_s:], "tail out")
    assert_close(np64(fin[0, 17])[None], rs_all, "final state")
    assert kda.kda_get_device_status() == 0


@pytest.mark.parametrize("deltanet", [False, True], ids=["gdn", "deltanet"])
def test_decode_bf16state(deltanet):
    """Scalar-gate decode on a bf16-stored state: bit for bit the per-channel bf16-state decode
    fed the broadcast gate, and against the rounding oracle."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, H, steps = 4, 3, 5
    d = synth.decode_inputs(B, H, seed=631, steps=steps, device="cuda")
    la_h = None if deltanet else synth.head_gates((steps, B), H, seed=632, device="cuda")
    s1 = d["state"].to(torch.bfloat16)
    s0, s2 = s1.clone(), s1.clone()
    outs = []
    for s in range(steps):
        g = None if deltanet else la_h[s]
        gc = torch.zeros_like(d["log_alpha"][s]) if deltanet else _bcast(la_h[s])
        o1 = kda.kda_gdn_decode_step_bf16state(d["q"][s], d["k"][s], d["v"][s], g, d["beta"][s], s1)
        o2 = kda.kda_decode_step_bf16state(d["q"][s], d["k"][s], d["v"][s], gc, d["beta"][s], s2)
        outs.append(o1)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
    assert torch.equal(s1, s2)
    pairs = [(b, h) for b in range(B) for h in range(H)]
    la = torch.zeros(steps, B, H, 128, device="cuda") if deltanet else _bcast(la_h)
    col = lambda t, b, h: np64(t[:steps, b, h])
    ro, rs = oracle.recurrent_bf16state(np.stack([col(d["q"], b, h) for b, h in pairs]),
                                        np.stack([col(d["k"], b, h) for b, h in pairs]),
                                        np.stack([col(d["v"], b, h) for b, h in pairs]),
                                        np.stack([col(la, b, h) for b, h in pairs]),
                                        np.stack([col(d["beta"], b, h) for b, h in pairs]),
                                        np.stack([np64(s0[b, h]) for b, h in pairs]))
    got = np.stack([np.stack([np64(outs[s][b, h]) for s in range(steps)]) for b, h in pairs])
    assert_close(got, ro, "decode out")
    assert_close(np.stack([np64(s1[b, h]) for b, h in pairs]), rs, "decode state")
