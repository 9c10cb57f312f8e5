"""GPU parity over the whole gate domain ("Kimi K3" article, lshu.cn/news/263999, §四: each key
channel has its own alpha in [0, 1], so some channels forget within a few tokens while others keep
their memory).  The chunk = 64 path factors each chunk's decay into fp16 operands; a chunk whose
gates leave that range is applied token by token in fp32 by the same kernel instead.  These tests
check the results against the fp64 oracle for gates on both sides of the bound and for the extreme
ones (per-token log alpha of -30, and -inf), mixed within one sequence, and check that the chunk
boundary invariants (split and resume, packed = solo, snapshots = prefix runs) stay bit-exact."""
import numpy as np
import pytest
import torch

from kda_testutil import assert_close, batch_heads, np64, packed_heads
from oracle import oracle

pytestmark = pytest.mark.gpu


def _ref(x, la, pairs, S0=None):
    s0 = None if S0 is None else np.stack([np64(S0[b, h]) for b, h in pairs])
    return oracle.recurrent(batch_heads(x["q"], pairs), batch_heads(x["k"], pairs), batch_heads(x["v"], pairs),
                            batch_heads(la, pairs), batch_heads(x["beta"], pairs), s0)


def _run(x, la, S0, gdn=False, final=None, sl=slice(None)):
    import kda_recurrent_state_gb300 as kda

    fn = kda.kda_gdn_chunk_fwd if gdn else kda.kda_chunk_fwd
    out, fin = fn(x["q"][:, sl].contiguous(), x["k"][:, sl].contiguous(), x["v"][:, sl].contiguous(),
                  la[:, sl].contiguous(), x["beta"][:, sl].contiguous(), S0, None, final, chunk=64)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    return out, fin


def _check(x, la, out, fin, pairs, S0, what):
    ro, rs = _ref(x, la, pairs, S0)
    assert_close(batch_heads(out, pairs), ro, what + ", out")
    assert_close(np.stack([np64(fin[b, h]) for b, h in pairs]), rs, what + ", state")


def test_mixed_fast_and_slow_channels():
    """Half the key channels forget within a few tokens (log alpha = -U(1, 10), four of them at
    -30), half are slow (-U(1e-5, 1e-3)); T = 4096 with a N(0, 0.02) initial state."""
    from kda_recurrent_state_gb300 import synth

    B, T, H = 1, 4096, 3
    x = synth.prefill_inputs(B, T, H, seed=7301, device="cuda", init="normal", gate="mixed")
    out, fin = _run(x, x["log_alpha"], x["init_state"])
    _check(x, x["log_alpha"], out, fin, [(0, h) for h in range(H)], x["init_state"], "mixed gates")


def test_steep_gates_inside_the_bound():
    """log alpha = -U(0.15, 0.2): a half chunk decays by about e^-5.6 (8.1 in log2 units), inside
    the fp16 operand bound (10), so the tensor-core path itself must meet the bar, with a
    N(0, 0.02) initial state whose small entries are the ones a too-wide operand range would push
    into the fp16 subnormals."""
    from kda_recurrent_state_gb300 import synth

    B, T, H = 2, 1024, 2
    x = synth.prefill_inputs(B, T, H, seed=7302, device="cuda", init="normal", gate="steep")
    out, fin = _run(x, x["log_alpha"], x["init_state"])
    _check(x, x["log_alpha"], out, fin, [(b, h) for b in range(B) for h in range(H)], x["init_state"], "steep")


@pytest.mark.parametrize("per_token", [-0.25, -0.3, -1.0, -30.0])
def test_uniform_steep_decay(per_token):
    """Every channel at one per-token log alpha around and beyond the bound (-0.25 x 32 = -8 per
    half chunk: 11.5 in log2 units; the previous bound of 15 accepted -0.3 with too little
    precision)."""
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(1, 300, 2, seed=7303, device="cuda", init="normal")
    la = torch.full_like(x["log_alpha"], per_token)
    out, fin = _run(x, la, x["init_state"])
    _check(x, la, out, fin, [(0, 0), (0, 1)], x["init_state"], f"log alpha {per_token}")


def test_alpha_zero():
    """log alpha = -inf (alpha = 0, a channel erased at that token) at a few (token, channel)
    positions: the state's rows for those channels are cleared exactly."""
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(1, 200, 2, seed=7304, device="cuda", init="normal")
    la = x["log_alpha"].clone()
    la[0, 0, :, 5] = float("-inf")
    la[0, 70, :, 17] = float("-inf")
    la[0, 199, :, 100] = float("-inf")
    out, fin = _run(x, la, x["init_state"])
    _check(x, la, out, fin, [(0, 0), (0, 1)], x["init_state"], "alpha = 0")
    # at the last token row 100 is cleared and then written once: S[100, :] = k_100 u^T, with
    # u the token's beta-scaled prediction error; its direction is u for every head
    for h in range(2):
        r = fin[0, h, 100].double()
        kk = float(x["k"][0, 199, h, 100])
        assert abs(kk) > 0 and bool(torch.isfinite(r).all())


def test_marked_units():
    """The first pass marks exactly the (sequence, head) units that met a chunk beyond the fp16
    range, in the caller's workspace (one int per unit): gates inside the bound keep every unit on
    the tensor-core path; one head with fast channels is the only one marked, and the other units'
    results are those of the run where no unit is marked, bit for bit."""
    from kda_recurrent_state_gb300 import binding, synth

    B, T, H = 2, 384, 3
    x = synth.prefill_inputs(B, T, H, seed=7314, device="cuda", init="normal", gate="steep")
    ws = torch.full((binding.kda_workspace_size(binding.KDA_OP_CHUNK, B, T, H),), 255, dtype=torch.uint8,
                    device="cuda")
    flags = lambda: ws[: 4 * B * H].view(torch.int32).cpu().tolist()  # noqa: E731
    import kda_recurrent_state_gb300 as kda

    out0, fin0 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"], chunk=64,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert flags() == [0] * (B * H)
    la = x["log_alpha"].clone()
    la[1, 200:, 1] = synth.prefill_inputs(1, T, 1, seed=7315, device="cuda", gate="mixed")["log_alpha"][0, 200:, 0]
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], la, x["beta"], x["init_state"], chunk=64, workspace=ws)
    torch.cuda.synchronize()
    assert flags() == [0, 0, 0, 0, 1, 0]
    assert kda.kda_get_device_status() == 0
    for b in range(B):
        for h in range(H):
            if (b, h) != (1, 1):
                assert torch.equal(out[b, :, h], out0[b, :, h]) and torch.equal(fin[b, h], fin0[b, h]), (b, h)
    _check(x, la, out, fin, [(1, 1)], x["init_state"], "marked unit")
    # the marked unit's first 192 tokens (chunks 0..2, within range) are the unmarked run's bits
    assert torch.equal(out[1, :192, 1], out0[1, :192, 1])


def _slow_then_fast(B, T, H, seed, fast_from, fast_to):
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(B, T, H, seed=seed, device="cuda", init="normal", gate="slow")
    la = x["log_alpha"].clone()
    fast = synth.prefill_inputs(B, T, H, seed=seed + 1, device="cuda", gate="mixed")["log_alpha"]
    la[:, fast_from:fast_to] = fast[:, fast_from:fast_to]
    return x, la


def test_fast_stretch_inside_a_sequence():
    """Slow gates with a stretch of fast ones in the middle (tokens 150..300: chunks 2..4 take the
    exact path, the others the tensor cores), and in place (init_state aliasing final_state)."""
    B, T, H = 2, 640, 3
    x, la = _slow_then_fast(B, T, H, 7305, 150, 300)
    S = x["init_state"].clone()
    out, fin = _run(x, la, S, final=S)
    assert fin.data_ptr() == S.data_ptr()
    _check(x, la, out, fin, [(b, h) for b in range(B) for h in range(H)], x["init_state"], "fast stretch")


@pytest.mark.parametrize("split", [128, 192, 256, 384])
def test_split_and_resume_bit_exact_across_paths(split):
    """A run resumed at a chunk boundary reproduces the unsplit run bit for bit whichever path each
    chunk takes (the fast stretch 150..300 lies before, across and after the split points)."""
    B, T, H = 1, 640, 2
    x, la = _slow_then_fast(B, T, H, 7306, 150, 300)
    out, fin = _run(x, la, x["init_state"])
    o1, f1 = _run(x, la, x["init_state"], sl=slice(0, split))
    o2, f2 = _run(x, la, f1, sl=slice(split, T))
    assert torch.equal(torch.cat([o1, o2], dim=1), out) and torch.equal(f2, fin)


def test_scalar_gate_beyond_the_bound():
    """Gated DeltaNet (one gate per head): half the heads forget fast; those chunks take the exact
    path like KDA's."""
    from kda_recurrent_state_gb300 import synth

    B, T, H = 1, 700, 4
    x = synth.prefill_inputs(B, T, H, seed=7307, device="cuda", init="normal")
    la_h = synth.head_gates((B, T), H, seed=7308, device="cuda", gate="mixed")
    out, fin = _run(x, la_h, x["init_state"], gdn=True)
    la = la_h[..., None].expand(B, T, H, 128).contiguous()  # the oracle's per-channel form
    _check(x, la, out, fin, [(0, h) for h in range(H)], x["init_state"], "scalar gates")


def test_varlen_snapshots_with_fast_channels():
    """Packed sequences, fast channels in every other one from its token 100 on: each sequence equals
    its solo run bit for bit, each snapshot equals the prefix run's final state bit for bit (the
    prefixes cover chunks of both paths), and the oracle agrees."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    lengths = [300, 128, 517, 64, 256]
    H = 2
    xv = synth.varlen_inputs(lengths, H, seed=7309, device="cuda")
    fastla = synth.varlen_inputs(lengths, H, seed=7310, device="cuda", gate="mixed")["log_alpha"]
    cu = xv["cu_seqlens"].cpu().tolist()
    la = xv["log_alpha"].clone()
    for s in range(0, len(lengths), 2):
        la[cu[s] + 100:cu[s + 1]] = fastla[cu[s] + 100:cu[s + 1]]
    out, fin, snaps = kda.kda_varlen_fwd(xv["q"], xv["k"], xv["v"], la, xv["beta"], xv["cu_seqlens"],
                                         xv["init_states"], snapshot_interval=64,
                                         cu_seqlens_host=xv["cu_seqlens"].cpu())
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    offs = kda.kda_snapshot_offsets(xv["cu_seqlens"].cpu(), 64).tolist()
    solo = lambda t, a, e: t[a:e][None].contiguous()  # noqa: E731
    for s, L in enumerate(lengths):
        a, e = cu[s], cu[s + 1]
        S0 = xv["init_states"][s:s + 1]
        so, sf = kda.kda_chunk_fwd(solo(xv["q"], a, e), solo(xv["k"], a, e), solo(xv["v"], a, e), solo(la, a, e),
                                   solo(xv["beta"], a, e), S0, chunk=64)
        torch.cuda.synchronize()
        assert torch.equal(out[a:e], so[0]) and torch.equal(fin[s], sf[0]), s
        ro, rs = oracle.recurrent(packed_heads(xv["q"], a, e, range(H)), packed_heads(xv["k"], a, e, range(H)),
                                  packed_heads(xv["v"], a, e, range(H)), packed_heads(la, a, e, range(H)),
                                  packed_heads(xv["beta"], a, e, range(H)), np64(S0[0]))
        assert_close(packed_heads(out, a, e, range(H)), ro, f"seq {s} out")
        assert_close(np64(fin[s]), rs, f"seq {s} state")
        for m in range(L // 64):  # snapshot m + 1 equals the final state of the prefix run
            p = a + 64 * (m + 1)
            _, pf = kda.kda_chunk_fwd(solo(xv["q"], a, p), solo(xv["k"], a, p), solo(xv["v"], a, p),
                                      solo(la, a, p), solo(xv["beta"], a, p), S0, chunk=64)
            torch.cuda.synchronize()
            assert torch.equal(snaps[offs[s] + m], pf[0]), (s, m)


def test_host_streamed_with_fast_channels():
    """The host-buffer entry point equals the device call bit for bit on gates beyond the bound
    (segments of 256 tokens: some start inside the fast stretch)."""
    import kda_recurrent_state_gb300 as kda

    x, la = _slow_then_fast(1, 700, 2, 7311, 200, 600)
    out_d, fin_d = _run(x, la, None)
    h = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "beta")}
    out_h, fin_h = kda.kda_chunk_fwd_host(h["q"], h["k"], h["v"], la.cpu().pin_memory(), h["beta"], None,
                                          segment_tokens=256, device="cuda")
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(fin_h, fin_d.cpu())


def test_chunk_bwd_beyond_its_bound():
    """The chunked backward (fp32, bound -80 per half chunk) on mixed gates: the units beyond the
    bound are recomputed by the token-serial backward in the same call; gradients match the oracle's
    reverse mode and no status is raised."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, T, H = 1, 200, 2
    x = synth.prefill_inputs(B, T, H, seed=7312, device="cuda", init="normal", gate="mixed")
    do = torch.randn(B, T, H, 128, generator=torch.Generator(device="cuda").manual_seed(7313), device="cuda")
    g = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], chunk=64)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    pairs = [(0, 0), (0, 1)]
    ref = oracle.recurrent_bwd(batch_heads(x["q"], pairs), batch_heads(x["k"], pairs), batch_heads(x["v"], pairs),
                               batch_heads(x["log_alpha"], pairs), batch_heads(x["beta"], pairs),
                               np.stack([np64(x["init_state"][b, h]) for b, h in pairs]), batch_heads(do, pairs))
    for name in ("dq", "dk", "dv", "dlog_alpha"):
        got = batch_heads(g[name], pairs)
        r = ref[name]
        rel = float(np.linalg.norm(got - r) / np.linalg.norm(r))
        mx = float(np.abs(got - r).max())
        assert rel <= 2e-3 and mx <= 1e-2 * max(1.0, float(np.abs(r).max())), (name, rel, mx)
