"""GPU parity of the chunked backward's tcgen05 serial passes.

The chunked backward runs its two serial recurrences (chunk-start states, state gradients) on
tcgen05 with one CTA per (sequence, head) whenever the units fill more than a quarter of the
SMs, and in a warp-level form split over value columns below that.  The shapes here have 40 or
more units, so on a 152-SM GB300 they take the tcgen05 form (the other tests in
test_gpu_bwd.py use a few units and take the warp-level one).  Sampled heads are checked
against the fp64 oracle's reverse mode at the backward's bar; every head is checked against the
independent token-serial fp32 backward (chunk = 1) at a tighter tolerance."""
import numpy as np
import pytest
import torch

from kda_testutil import batch_heads, errors, np64, packed_heads
from oracle import oracle
from test_gpu_bwd import _bcast, _close, _oracle_grads

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dlog_alpha", "dbeta", "d_init")
SERIAL_REL = 1e-4  # chunked (split-bf16 products) against the token-serial fp32 path


def _against_serial(got, one, names=GRADS):
    for name in names:
        if got[name] is None:
            assert one[name] is None, name
            continue
        rel, _ = errors(np64(got[name]), np64(one[name]))
        assert rel <= SERIAL_REL, f"{name}: rel-L2 {rel:.3e} against the token-serial backward"


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T", [65, 300])
def test_tc_serial_parity(T, in_dtype):
    """B=1, H=40 (40 units), ragged T, resumed from a state and with a final-state cotangent."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, H = 1, 40
    x = synth.prefill_inputs(B, T, H, seed=6100 + T, device="cuda", init="normal", in_dtype=in_dtype)
    g = torch.Generator(device="cuda").manual_seed(6200 + T)
    do = torch.randn(B, T, H, 128, generator=g, device="cuda")
    dSf = torch.randn(B, H, 128, 128, generator=g, device="cuda")
    got = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], dSf, chunk=64)
    one = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], dSf, chunk=1)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    pairs = [(0, 0), (0, 21), (0, 39)]
    ref = _oracle_grads(x, x["log_alpha"], do, dSf, pairs)
    for name in ("dq", "dk", "dv", "dlog_alpha", "dbeta"):
        _close(batch_heads(got[name], pairs), ref[name], name)
    _close(np.stack([np64(got["d_init"][b, h]) for b, h in pairs]), ref["dS0"], "d_init")
    _against_serial(got, one)


def test_tc_serial_varlen():
    """Packed sequences with 8 heads (48 units): an empty sequence passes its final-state
    cotangent through exactly; the others match the oracle on sampled heads."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    lengths, H = [300, 0, 65, 513, 1, 64], 8
    xv = synth.varlen_inputs(lengths, H, seed=6301, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(6302)
    do = torch.randn(xv["q"].shape[0], H, 128, generator=g, device="cuda")
    dSf = torch.randn(len(lengths), H, 128, 128, generator=g, device="cuda")
    got = kda.kda_bwd(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], do, xv["init_states"], dSf,
                      cu_seqlens=xv["cu_seqlens"], chunk=64)
    one = kda.kda_bwd(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], do, xv["init_states"], dSf,
                      cu_seqlens=xv["cu_seqlens"], chunk=1)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    cu = xv["cu_seqlens"].tolist()
    heads = [0, 7]
    for s in range(len(lengths)):
        a, b = cu[s], cu[s + 1]
        if a == b:
            assert torch.equal(got["d_init"][s], dSf[s])
            continue
        ref = oracle.recurrent_bwd(packed_heads(xv["q"], a, b, heads), packed_heads(xv["k"], a, b, heads),
                                   packed_heads(xv["v"], a, b, heads), packed_heads(xv["log_alpha"], a, b, heads),
                                   packed_heads(xv["beta"], a, b, heads), np64(xv["init_states"][s][heads]),
                                   packed_heads(do, a, b, heads), np64(dSf[s][heads]))
        for name in ("dq", "dk", "dv", "dlog_alpha", "dbeta"):
            _close(packed_heads(got[name], a, b, heads), ref[name], f"seq {s} {name}")
        _close(np64(got["d_init"][s][heads]), ref["dS0"], f"seq {s} d_init")
    _against_serial(got, one)


@pytest.mark.parametrize("gate", [1, 2], ids=["head", "none"])
def test_tc_serial_scalar_and_no_gate(gate):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, T, H = 1, 200, 40
    x = synth.prefill_inputs(B, T, H, seed=6401, device="cuda", init="normal")
    la_h = synth.head_gates((B, T), H, seed=6402, device="cuda") if gate == 1 else None
    do = torch.randn(B, T, H, 128, generator=torch.Generator(device="cuda").manual_seed(6403), device="cuda")
    got = kda.kda_bwd(x["q"], x["k"], x["v"], la_h, x["beta"], do, x["init_state"], None, gate=gate, chunk=64)
    one = kda.kda_bwd(x["q"], x["k"], x["v"], la_h, x["beta"], do, x["init_state"], None, gate=gate, chunk=1)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    pairs = [(0, 3), (0, 36)]
    la_full = _bcast(la_h) if gate == 1 else torch.zeros_like(x["log_alpha"])
    ref = _oracle_grads(x, la_full, do, None, pairs)
    for name in ("dq", "dk", "dv", "dbeta"):
        _close(batch_heads(got[name], pairs), ref[name], name)
    _against_serial(got, one)


def test_tc_serial_deterministic_and_redo():
    """Two calls give the same bits; a unit with a half-chunk beyond the fp32 bound is recomputed
    by the token-serial backward (bit-equal to chunk = 1) while the other units keep the tcgen05
    result."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, T, H = 1, 192, 40
    x = synth.prefill_inputs(B, T, H, seed=6501, device="cuda", init="normal")
    la = x["log_alpha"].clone()
    la[0, 100:104, 5] = -30.0  # head 5: rows 32..63 of chunk 1 sum to about -120
    do = torch.randn(B, T, H, 128, generator=torch.Generator(device="cuda").manual_seed(6502), device="cuda")
    g1 = kda.kda_bwd(x["q"], x["k"], x["v"], la, x["beta"], do, x["init_state"], chunk=64)
    g2 = kda.kda_bwd(x["q"], x["k"], x["v"], la, x["beta"], do, x["init_state"], chunk=64)
    one = kda.kda_bwd(x["q"], x["k"], x["v"], la, x["beta"], do, x["init_state"], chunk=1)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    for name in GRADS:
        assert torch.equal(g1[name], g2[name]), name
    for name in ("dq", "dk", "dv", "dlog_alpha", "dbeta"):
        assert torch.equal(g1[name][:, :, 5], one[name][:, :, 5]), name
    assert torch.equal(g1["d_init"][:, 5], one["d_init"][:, 5])
    keep = [h for h in range(H) if h != 5]
    _against_serial({n: g1[n][:, :, keep] if n != "d_init" else g1[n][:, keep] for n in GRADS},
                    {n: one[n][:, :, keep] if n != "d_init" else one[n][:, keep] for n in GRADS})
    ref = _oracle_grads(dict(x, log_alpha=la), la, do, None, [(0, 5), (0, 6)])
    for name in ("dq", "dk", "dv", "dbeta"):
        _close(batch_heads(g1[name], [(0, 5), (0, 6)]), ref[name], name)
