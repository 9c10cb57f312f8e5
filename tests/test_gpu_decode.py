"""GPU parity of kda_decode_step and kda_decode_step_bf16state against the fp64 oracle
(through the C ABI)."""
import numpy as np
import pytest
import torch

from kda_testutil import assert_close, errors, np64
from oracle import oracle

pytestmark = pytest.mark.gpu


def _oracle_steps(d, pairs, steps, fn=oracle.recurrent, state=None):
    """Oracle over `steps` tokens for the listed (b,h) pairs, starting from `state`
    (default d['state'])."""
    state = d["state"] if state is None else state
    col = lambda t, b, h: np64(t[:steps, b, h])
    q = np.stack([col(d["q"], b, h) for b, h in pairs])
    k = np.stack([col(d["k"], b, h) for b, h in pairs])
    v = np.stack([col(d["v"], b, h) for b, h in pairs])
    la = np.stack([col(d["log_alpha"], b, h) for b, h in pairs])
    be = np.stack([col(d["beta"], b, h) for b, h in pairs])
    S0 = np.stack([np64(state[b, h]) for b, h in pairs])
    return fn(q, k, v, la, be, S0)


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_small(in_dtype, out_dtype):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, H, steps = 5, 3, 6
    d = synth.decode_inputs(B, H, seed=101, steps=steps, device="cuda", in_dtype=in_dtype)
    state = d["state"].clone()
    outs = []
    for s in range(steps):
        outs.append(kda.kda_decode_step(d["q"][s], d["k"][s], d["v"][s], d["log_alpha"][s], d["beta"][s], state,
                                        out_dtype=out_dtype))
    torch.cuda.synchronize()
    pairs = [(b, h) for b in range(B) for h in range(H)]
    ro, rs = _oracle_steps(d, pairs, steps)
    got_o = np.stack([np.stack([np64(outs[s][b, h]) for s in range(steps)]) for b, h in pairs])
    assert_close(got_o, ro, "decode outputs")
    assert_close(np.stack([np64(state[b, h]) for b, h in pairs]), rs, "decode state")
    assert kda.kda_get_device_status() == 0


def test_decode_full_size_sampled():
    """256 sessions x 96 heads, 64 successive steps with the state updated in place (the
    batched-decode workload); sampled (session, head) pairs are checked against the oracle."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    Bs, H, steps = 256, 96, 64
    d = synth.decode_inputs(Bs, H, seed=synth.SEED_BASE + 3, steps=steps, device="cuda")
    state = d["state"].clone()
    pairs = [(0, 0), (255, 95), (17, 40), (128, 3), (200, 77), (63, 64)]
    outs = torch.empty(steps, len(pairs), 128, device="cuda")
    for s in range(steps):
        o = kda.kda_decode_step(d["q"][s], d["k"][s], d["v"][s], d["log_alpha"][s], d["beta"][s], state)
        for i, (b, h) in enumerate(pairs):
            outs[s, i] = o[b, h]
    torch.cuda.synchronize()
    ro, rs = _oracle_steps(d, pairs, steps)
    assert_close(np64(outs).transpose(1, 0, 2), ro, "decode outputs")
    assert_close(np.stack([np64(state[b, h]) for b, h in pairs]), rs, "decode state")


def test_decode_empty_is_noop():
    import kda_recurrent_state_gb300 as kda

    z = torch.empty(0, 4, 128, device="cuda", dtype=torch.bfloat16)
    st = torch.empty(0, 4, 128, 128, device="cuda")
    out = kda.kda_decode_step(z, z, z, z.float(), torch.empty(0, 4, device="cuda"), st)
    assert out.shape == (0, 4, 128)


# ---- bf16-stored state -------------------------------------------------------------


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
def test_decode_bf16state_small(in_dtype):
    """Several steps on a bf16 state against the oracle that rounds its fp64 state to bf16
    after every token (the output is read before the rounding)."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, H, steps = 5, 3, 6
    d = synth.decode_inputs(B, H, seed=211, steps=steps, device="cuda", in_dtype=in_dtype)
    state = d["state"].to(torch.bfloat16)
    s0 = state.clone()
    outs = [kda.kda_decode_step_bf16state(d["q"][s], d["k"][s], d["v"][s], d["log_alpha"][s], d["beta"][s], state)
            for s in range(steps)]
    torch.cuda.synchronize()
    pairs = [(b, h) for b in range(B) for h in range(H)]
    ro, rs = _oracle_steps(d, pairs, steps, oracle.recurrent_bf16state, s0)
    got_o = np.stack([np.stack([np64(outs[s][b, h]) for s in range(steps)]) for b, h in pairs])
    assert_close(got_o, ro, "bf16-state decode outputs")
    assert_close(np.stack([np64(state[b, h]) for b, h in pairs]), rs, "bf16-state decode state")
    assert kda.kda_get_device_status() == 0


def test_decode_bf16state_rounding_one_step():
    """One step from a bf16 state: the stored state is the fp32 update rounded to nearest
    bf16, so it equals the oracle's rounded fp64 update except where the two sides'
    unrounded values straddle a rounding boundary (then they differ by one bf16 unit, or
    by the fp32 rounding of the update's terms where an entry cancels to near zero).
    Truncation instead of rounding would change about half of the elements."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, H = 8, 16
    d = synth.decode_inputs(B, H, seed=223, steps=1, device="cuda")
    state = d["state"].to(torch.bfloat16)
    s0 = state.clone()
    kda.kda_decode_step_bf16state(d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0], d["beta"][0], state)
    torch.cuda.synchronize()
    pairs = [(b, h) for b in range(B) for h in range(H)]
    _, rs = _oracle_steps(d, pairs, 1, oracle.recurrent_bf16state, s0)
    got = np.stack([np64(state[b, h]) for b, h in pairs])
    diff = got != rs
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(rs), 1e-30))[1] - 8)  # bf16 spacing at |rs|
    # fp32 rounding of the update's terms (a few units of 2^-24 of the head's largest entry)
    # can exceed the bf16 spacing of an entry that cancels to near zero
    slack = ulp + 2.0 ** -19 * np.abs(rs).max(axis=(1, 2), keepdims=True)
    err = np.abs(got - rs)
    w = np.unravel_index(np.argmax(err / slack), err.shape)
    assert np.all(err <= slack), f"stored state at {w}: {got[w]!r} vs {rs[w]!r} (bf16 unit {ulp[w]:.3e})"
    assert diff.mean() < 1e-3, f"{diff.mean():.2e} of the stored elements differ from round-to-nearest"


def test_decode_bf16state_full_size_sampled():
    """256 sessions x 96 heads with a bf16 state, 64 successive in-place steps; sampled
    (session, head) pairs against the rounding oracle, and the drift from the fp64-state
    recurrence stays within what bf16 storage implies."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    Bs, H, steps = 256, 96, 64
    d = synth.decode_inputs(Bs, H, seed=synth.SEED_BASE + 3, steps=steps, device="cuda")
    state = d["state"].to(torch.bfloat16)
    s0 = state.clone()
    pairs = [(0, 0), (255, 95), (17, 40), (128, 3), (200, 77), (63, 64)]
    outs = torch.empty(steps, len(pairs), 128, device="cuda")
    for s in range(steps):
        o = kda.kda_decode_step_bf16state(d["q"][s], d["k"][s], d["v"][s], d["log_alpha"][s], d["beta"][s], state)
        for i, (b, h) in enumerate(pairs):
            outs[s, i] = o[b, h]
    torch.cuda.synchronize()
    got_o = np64(outs).transpose(1, 0, 2)
    got_s = np.stack([np64(state[b, h]) for b, h in pairs])
    ro, rs = _oracle_steps(d, pairs, steps, oracle.recurrent_bf16state, s0)
    assert_close(got_o, ro, "bf16-state decode outputs")
    assert_close(got_s, rs, "bf16-state decode state")
    fo, fs = _oracle_steps(d, pairs, steps, oracle.recurrent, s0)  # same start, state kept in fp64
    rel_o, _ = errors(got_o, fo)
    rel_s, _ = errors(got_s, fs)
    assert rel_o < 3e-2 and rel_s < 3e-2, (rel_o, rel_s)
    assert kda.kda_get_device_status() == 0


def test_decode_bf16state_rejects_fp32_state():
    import kda_recurrent_state_gb300 as kda

    z = torch.zeros(1, 1, 128, device="cuda")
    with pytest.raises(TypeError):
        kda.kda_decode_step_bf16state(z, z, z, z, torch.zeros(1, 1, device="cuda"), torch.zeros(1, 1, 128, 128,
                                                                                                  device="cuda"))


@pytest.mark.parametrize("bf16state", [False, True], ids=["fp32_state", "bf16_state"])
def test_decode_continues_prefill(bf16state):
    """A prefill of 300 tokens followed by 20 decode steps on its final state equals the
    per-token recurrence over all 320 tokens (outputs of the decoded tokens and the final
    state).  With a bf16-stored state the prefill's state is rounded once before decoding
    and every decode step rounds again, which the oracle reproduces."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    T0, n, H = 300, 20, 3
    x = synth.prefill_inputs(2, T0 + n, H, seed=707, device="cuda", init="normal")
    pre = lambda t: t[:, :T0].contiguous()
    _, fin = kda.kda_chunk_fwd(pre(x["q"]), pre(x["k"]), pre(x["v"]), pre(x["log_alpha"]), pre(x["beta"]),
                               x["init_state"])
    state = fin.to(torch.bfloat16) if bf16state else fin.clone()
    step = kda.kda_decode_step_bf16state if bf16state else kda.kda_decode_step
    outs = [step(x["q"][:, t].contiguous(), x["k"][:, t].contiguous(), x["v"][:, t].contiguous(),
                 x["log_alpha"][:, t].contiguous(), x["beta"][:, t].contiguous(), state) for t in range(T0, T0 + n)]
    torch.cuda.synchronize()
    pairs = [(b, h) for b in range(2) for h in range(H)]
    col = lambda t, b, h: np64(t[b, :, h])
    S0 = np.stack([np64(x["init_state"][b, h]) for b, h in pairs])
    args = [np.stack([col(x[nm], b, h) for b, h in pairs]) for nm in ("q", "k", "v", "log_alpha", "beta")]
    if bf16state:  # fp64 prefill, state rounded once, then the rounding decode steps
        _, s_mid = oracle.recurrent(*[a[:, :T0] for a in args], S0)
        ro, rs = oracle.recurrent_bf16state(*[a[:, T0:] for a in args], oracle.round_bf16(s_mid))
    else:
        ro_all, rs = oracle.recurrent(*args, S0)
        ro = ro_all[:, T0:]
    got = np.stack([np.stack([np64(outs[t][b, h]) for t in range(n)]) for b, h in pairs])
    assert_close(got, ro, "decoded outputs")
    assert_close(np.stack([np64(state[b, h]) for b, h in pairs]), rs, "state after decoding")
    assert kda.kda_get_device_status() == 0
