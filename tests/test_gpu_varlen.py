"""GPU parity of kda_varlen_fwd: packed sequences, per-sequence initial/final
states and state snapshots.  Floating-point results are checked against the
fp64 oracle; indexing (which snapshot lands where, which tokens belong to which
sequence) is checked bit-exactly against single-sequence runs of the GPU path."""
import numpy as np
import pytest
import torch

from kda_testutil import assert_close, np64, packed_heads
from oracle import oracle

pytestmark = pytest.mark.gpu
CHUNKS = [64, 1]


def _run(x, chunk, interval=0, **kw):
    import kda_recurrent_state_gb300 as kda

    return kda.kda_varlen_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"], x["init_states"],
                              chunk=chunk, snapshot_interval=interval, **kw)


def _check_seq(x, s, heads, out, fin, snaps, snap_off, interval, what):
    cu = x["cu_seqlens"].tolist()
    a, b = cu[s], cu[s + 1]
    S0 = np.stack([np64(x["init_states"][s, h]) for h in heads])
    if b == a:
        assert np.array_equal(np.stack([np64(fin[s, h]) for h in heads]), S0)
        return
    res = oracle.recurrent(*(packed_heads(x[n], a, b, heads) for n in ("q", "k", "v", "log_alpha", "beta")), S0,
                           snap_interval=interval)
    assert_close(packed_heads(out, a, b, heads), res[0], f"{what} seq {s} out")
    assert_close(np.stack([np64(fin[s, h]) for h in heads]), res[1], f"{what} seq {s} state")
    if interval and (b - a) >= interval:
        o0 = int(snap_off[s])
        m = (b - a) // interval
        got = np.stack([np64(snaps[o0:o0 + m, h]) for h in heads])
        assert_close(got, res[2], f"{what} seq {s} snapshots")


@pytest.mark.parametrize("chunk", CHUNKS)
def test_varlen_small_with_snapshots(chunk):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    lengths = [1, 63, 64, 65, 200, 0, 128, 257]
    x = synth.varlen_inputs(lengths, 3, seed=21, device="cuda")
    out, fin, snaps = _run(x, chunk, interval=64)
    torch.cuda.synchronize()
    off = kda.kda_snapshot_offsets(x["cu_seqlens"].cpu(), 64)
    for s in range(len(lengths)):
        _check_seq(x, s, [0, 1, 2], out, fin, snaps, off, 64, "small")
    assert kda.kda_get_device_status() == 0


@pytest.mark.parametrize("chunk", CHUNKS)
def test_varlen_equals_single_sequence_runs(chunk):
    """Each packed sequence is bit-identical to running it alone; snapshot m is bit-identical
    to the final state of the length-m*interval prefix; the last snapshot of a sequence whose
    length is a multiple of the interval equals its final state."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    lengths = [300, 128, 77, 512]
    x = synth.varlen_inputs(lengths, 2, seed=22, device="cuda")
    out, fin, snaps = _run(x, chunk, interval=128)
    cu = x["cu_seqlens"].tolist()
    off = kda.kda_snapshot_offsets(cu, 128).tolist()
    for s, L in enumerate(lengths):
        a, b = cu[s], cu[s + 1]
        one = {n: x[n][a:b].contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
        one["cu_seqlens"] = torch.tensor([0, L], dtype=torch.int64, device="cuda")
        one["init_states"] = x["init_states"][s:s + 1].contiguous()
        o1, f1, _ = _run(one, chunk)
        assert torch.equal(o1, out[a:b]) and torch.equal(f1[0], fin[s])
        for m in range(1, L // 128 + 1):
            pre = {n: one[n][:128 * m].contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
            pre["cu_seqlens"] = torch.tensor([0, 128 * m], dtype=torch.int64, device="cuda")
            pre["init_states"] = one["init_states"]
            _, fp, _ = _run(pre, chunk)
            assert torch.equal(snaps[off[s] + m - 1], fp[0]), (s, m)
        if L % 128 == 0:
            assert torch.equal(snaps[off[s + 1] - 1], fin[s])


@pytest.mark.parametrize("chunk", [64])
def test_varlen_full_size_sampled(chunk):
    """16 packed sequences, lengths log-uniform in [1024, 65536], H=64, every other sequence
    resuming from an N(0,0.02) state, snapshots every 16384 tokens: sampled (sequence, head)
    pairs against the oracle, including every snapshot of the sampled heads."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    lengths = synth.varlen_lengths(16, 1024, 65536, seed=synth.SEED_BASE + 4)
    x = synth.varlen_inputs(lengths, 64, seed=synth.SEED_BASE + 4, device="cuda")
    out, fin, snaps = _run(x, chunk, interval=16384)
    torch.cuda.synchronize()
    off = kda.kda_snapshot_offsets(x["cu_seqlens"].cpu(), 16384)
    longest = int(np.argmax(lengths))
    for s, heads in [(longest, [0, 63]), (0, [5]), (1, [17]), (7, [40]), (15, [62])]:
        _check_seq(x, s, heads, out, fin, snaps, off, 16384, "full")


@pytest.mark.parametrize("prefix", [700, 1000])
def test_resume_from_snapshot(prefix):
    """Prefix reuse: the latest snapshot covering a request's prefix, used as the initial
    state of a run over the remaining tokens, reproduces the unsplit run bit for bit
    (outputs after the snapshot and the final state)."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    lengths = [1000, 700, 130]
    x = synth.varlen_inputs(lengths, 3, seed=synth.SEED_BASE + 13, device="cuda", gate="slow")
    out, fin, snaps = _run(x, 64, interval=128)
    off = kda.kda_snapshot_offsets(x["cu_seqlens"].cpu(), 128)
    idx, covered = kda.kda_snapshot_lookup(off, 0, 128, prefix)
    assert covered == (prefix // 128) * 128 and idx == off[0].item() + prefix // 128 - 1
    rest = {n: x[n][covered:lengths[0]].unsqueeze(0).contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
    o2, f2 = kda.kda_chunk_fwd(rest["q"], rest["k"], rest["v"], rest["log_alpha"], rest["beta"],
                               snaps[idx].unsqueeze(0).contiguous(), chunk=64)
    torch.cuda.synchronize()
    assert torch.equal(o2[0], out[covered:lengths[0]])
    assert torch.equal(f2[0], fin[0])
    assert kda.kda_snapshot_lookup(off, 2, 128, 100) == (-1, 0)



def test_many_sequences_beyond_longest_first_ranking():
    """300 packed sequences (more than the kernel ranks for its longest-first order, so CTAs
    take sequences in order), lengths 0..130 with snapshots every 64 tokens: sampled
    sequences against the oracle, and every sequence bit for bit against its own run."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    g = torch.Generator().manual_seed(606)
    lengths = torch.randint(0, 131, (300,), generator=g).tolist()
    x = synth.varlen_inputs(lengths, 1, seed=607, device="cuda", resume_every=3)
    out, fin, snaps = _run(x, 64, 64)
    torch.cuda.synchronize()
    off = kda.kda_snapshot_offsets(x["cu_seqlens"].cpu(), 64)
    for s in (0, 1, 77, 150, 299):
        _check_seq(x, s, [0], out, fin, snaps, off, 64, "many")
    cu = x["cu_seqlens"].tolist()
    for s in range(0, 300, 7):
        a, b = cu[s], cu[s + 1]
        sl = lambda t: t[a:b].unsqueeze(0).contiguous()
        o1, f1 = kda.kda_chunk_fwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["log_alpha"]), sl(x["beta"]),
                                   x["init_states"][s:s + 1].contiguous())
        assert torch.equal(out[a:b], o1[0]) and torch.equal(fin[s], f1[0]), f"sequence {s}"
    assert kda.kda_get_device_status() == 0
