"""GPU tests of kda_varlen_fwd_pool, the packed prefill over a caller-owned state pool
(prefix reuse from state snapshots), through the C ABI.

The pool call must give exactly what kda_varlen_fwd gives with the same states gathered
into packed arrays; snapshots land in the requested slots and nowhere else; a prompt
sharing a prefix resumes from the nearest pooled snapshot and reproduces the unsplit
run bit for bit; out-of-range slots are skipped and reported, never dereferenced."""
import numpy as np
import pytest
import torch

from kda_testutil import assert_close, np64, packed_heads
from oracle import oracle

pytestmark = pytest.mark.gpu

LENGTHS = [700, 64, 0, 1500, 257]
H = 2
INTERVAL = 256


def _gates(xv, gate, seed):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    if gate == kda.KDA_GATE_CHANNEL:
        return xv["log_alpha"]
    if gate == kda.KDA_GATE_HEAD:
        return synth.head_gates((xv["q"].shape[0],), H, seed=seed, device="cuda")
    return None


@pytest.mark.parametrize("chunk", [64, 1])
@pytest.mark.parametrize("gate", [0, 1, 2], ids=["channel", "head", "none"])
def test_pool_equals_packed(chunk, gate):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    xv = synth.varlen_inputs(LENGTHS, H, seed=808, device="cuda")
    la = _gates(xv, gate, 809)
    N = len(LENGTHS)
    init_slots = torch.tensor([5, -1, 2, 7, -1], dtype=torch.int64)
    init_packed = xv["init_states"].clone()
    init_packed[(init_slots < 0).cuda()] = 0.0
    off = kda.kda_snapshot_offsets(xv["cu_seqlens"].cpu(), INTERVAL)
    n_snap = int(off[-1])
    # distinct destination slots, every third snapshot not stored
    free = [i for i in range(16) if i not in (5, 2, 7)]
    snap_slots = torch.tensor([(-1 if k % 3 == 2 else free[k]) for k in range(n_snap)], dtype=torch.int64)

    pool = torch.full((16, H, 128, 128), float("nan"), device="cuda")
    for s in range(N):
        if init_slots[s] >= 0:
            pool[init_slots[s]] = xv["init_states"][s]
    pool0 = pool.clone()

    if gate == kda.KDA_GATE_CHANNEL:
        ref = kda.kda_varlen_fwd
    else:
        ref = kda.kda_gdn_varlen_fwd
    o_p, f_p, snaps = ref(xv["q"], xv["k"], xv["v"], la, xv["beta"], xv["cu_seqlens"], init_packed, chunk=chunk,
                          snapshot_interval=INTERVAL)
    o, f = kda.kda_varlen_fwd_pool(xv["q"], xv["k"], xv["v"], la, xv["beta"], xv["cu_seqlens"], pool,
                                   init_slots.cuda(), snap_slots.cuda(), gate=gate, chunk=chunk,
                                   snapshot_interval=INTERVAL)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    assert torch.equal(o, o_p) and torch.equal(f, f_p)
    written = set()
    for kk in range(n_snap):
        if snap_slots[kk] >= 0:
            assert torch.equal(pool[snap_slots[kk]], snaps[kk]), f"snapshot {kk}"
            written.add(int(snap_slots[kk]))
    for i in range(16):
        if i not in written:  # initial-state slots and unused slots are untouched
            assert torch.equal(pool[i].isnan(), pool0[i].isnan())
            assert torch.equal(torch.nan_to_num(pool[i]), torch.nan_to_num(pool0[i]))


@pytest.mark.parametrize("chunk", [64, 1])
def test_prefix_resume_from_pool(chunk):
    """Request A (3000 tokens) stores its snapshots every 512 tokens in the pool.  Request B
    shares A's first 2000 tokens and then diverges: it resumes from the latest snapshot
    covering at most 2000 tokens (1536) and processes only the rest.  Its outputs and final
    state equal those of B run from the start, bit for bit; sampled heads match the oracle."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    TA, TB, shared, iv = 3000, 3000, 2000, 512
    xa = synth.varlen_inputs([TA], H, seed=901, device="cuda", resume_every=1000)
    xb = synth.varlen_inputs([TB], H, seed=902, device="cuda", resume_every=1000)
    for key in ("q", "k", "v", "log_alpha", "beta"):  # B shares A's prefix
        xb[key][:shared] = xa[key][:shared]
    pool = torch.zeros(8, H, 128, 128, device="cuda")
    n_snap = TA // iv
    cu_a = torch.tensor([0, TA], dtype=torch.int64, device="cuda")
    kda.kda_varlen_fwd_pool(xa["q"], xa["k"], xa["v"], xa["log_alpha"], xa["beta"], cu_a, pool, None,
                            torch.arange(n_snap, dtype=torch.int64, device="cuda"), chunk=chunk,
                            snapshot_interval=iv)
    off = kda.kda_snapshot_offsets([0, TA], iv)
    idx, covered = kda.kda_snapshot_lookup(off, 0, iv, shared)
    assert (idx, covered) == (2, 1536)
    rest = lambda t: t[covered:].contiguous()
    cu_r = torch.tensor([0, TB - covered], dtype=torch.int64, device="cuda")
    o_r, f_r = kda.kda_varlen_fwd_pool(rest(xb["q"]), rest(xb["k"]), rest(xb["v"]), rest(xb["log_alpha"]),
                                       rest(xb["beta"]), cu_r, pool,
                                       torch.tensor([idx], dtype=torch.int64, device="cuda"), chunk=chunk)
    cu_b = torch.tensor([0, TB], dtype=torch.int64, device="cuda")
    o_b, f_b, _ = kda.kda_varlen_fwd(xb["q"], xb["k"], xb["v"], xb["log_alpha"], xb["beta"], cu_b, None,
                                     chunk=chunk)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    assert torch.equal(o_r, o_b[covered:]) and torch.equal(f_r, f_b)
    ro, rs = oracle.recurrent(packed_heads(xb["q"], 0, TB, [0, 1]), packed_heads(xb["k"], 0, TB, [0, 1]),
                              packed_heads(xb["v"], 0, TB, [0, 1]), packed_heads(xb["log_alpha"], 0, TB, [0, 1]),
                              packed_heads(xb["beta"], 0, TB, [0, 1]), None)
    assert_close(packed_heads(o_r, 0, TB - covered, [0, 1]), ro[:, covered:], "resumed out")
    assert_close(np64(f_r[0]), rs, "resumed state")


def test_out_of_range_slots_are_skipped():
    """A slot index past the pool (or below -1) is never dereferenced: the state is taken as
    zero or the snapshot dropped, and KDA_STATUS_SLOT_RANGE is raised."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    xv = synth.varlen_inputs([512, 300], H, seed=77, device="cuda")
    pool = torch.zeros(2, H, 128, 128, device="cuda")
    pool[0] = xv["init_states"][0]
    init_slots = torch.tensor([0, 1000], dtype=torch.int64, device="cuda")
    # three snapshots (two of sequence 0, one of sequence 1): one stored, two out of range
    assert int(kda.kda_snapshot_offsets([0, 512, 812], 256)[-1]) == 3
    snap_slots = torch.tensor([1, -5, 7], dtype=torch.int64, device="cuda")
    o, f = kda.kda_varlen_fwd_pool(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], xv["cu_seqlens"], pool,
                                   init_slots, snap_slots, snapshot_interval=256)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == kda.binding.KDA_STATUS_SLOT_RANGE
    assert kda.kda_get_device_status() == 0  # read and cleared
    init = xv["init_states"].clone()
    init[1] = 0.0
    o_p, f_p, snaps = kda.kda_varlen_fwd(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], xv["cu_seqlens"],
                                         init, snapshot_interval=256)
    torch.cuda.synchronize()
    assert torch.equal(o, o_p) and torch.equal(f, f_p)
    assert torch.equal(pool[1], snaps[0])


@pytest.mark.parametrize("chunk", [64, 1])
def test_bf16_pool(chunk):
    """A bf16 pool: snapshots are the fp32 snapshots rounded to nearest bf16 (bit for bit),
    initial states are widened exactly, and a request resumed from a bf16 snapshot equals a
    run started from that snapshot widened to fp32, bit for bit; sampled against the oracle."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    xv = synth.varlen_inputs(LENGTHS, H, seed=818, device="cuda")
    N = len(LENGTHS)
    off = kda.kda_snapshot_offsets(xv["cu_seqlens"].cpu(), INTERVAL)
    n_snap = int(off[-1])
    init_slots = torch.arange(N, dtype=torch.int64)  # slots 0..N-1: initial states
    snap_slots = torch.arange(N, N + n_snap, dtype=torch.int64)
    pool = torch.zeros(N + n_snap, H, 128, 128, dtype=torch.bfloat16, device="cuda")
    pool[:N] = xv["init_states"].to(torch.bfloat16)
    o, f = kda.kda_varlen_fwd_pool(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], xv["cu_seqlens"], pool,
                                   init_slots.cuda(), snap_slots.cuda(), chunk=chunk, snapshot_interval=INTERVAL)
    o_p, f_p, snaps = kda.kda_varlen_fwd(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], xv["cu_seqlens"],
                                         pool[:N].float(), chunk=chunk, snapshot_interval=INTERVAL)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status() == 0
    assert torch.equal(o, o_p) and torch.equal(f, f_p)
    assert torch.equal(pool[N:], snaps.to(torch.bfloat16))
    assert torch.equal(pool[:N], xv["init_states"].to(torch.bfloat16))  # initial-state slots untouched

    # resume sequence 3 (1500 tokens) from its snapshot after 1024 tokens
    s, covered = 3, 1024
    idx, cov = kda.kda_snapshot_lookup(off, s, INTERVAL, covered + 100)
    assert cov == covered
    a, b = xv["cu_seqlens"][s].item() + covered, xv["cu_seqlens"][s + 1].item()
    rest = lambda t: t[a:b].contiguous()
    cu_r = torch.tensor([0, b - a], dtype=torch.int64, device="cuda")
    o_r, f_r = kda.kda_varlen_fwd_pool(rest(xv["q"]), rest(xv["k"]), rest(xv["v"]), rest(xv["log_alpha"]),
                                       rest(xv["beta"]), cu_r, pool, torch.tensor([N + idx], device="cuda"),
                                       chunk=chunk)
    o_w, f_w, _ = kda.kda_varlen_fwd(rest(xv["q"]), rest(xv["k"]), rest(xv["v"]), rest(xv["log_alpha"]),
                                     rest(xv["beta"]), cu_r, pool[N + idx:N + idx + 1].float(), chunk=chunk)
    torch.cuda.synchronize()
    assert torch.equal(o_r, o_w) and torch.equal(f_r, f_w)
    heads = [0, 1]
    ro, rs = oracle.recurrent(packed_heads(xv["q"], a, b, heads), packed_heads(xv["k"], a, b, heads),
                              packed_heads(xv["v"], a, b, heads), packed_heads(xv["log_alpha"], a, b, heads),
                              packed_heads(xv["beta"], a, b, heads), np64(pool[N + idx]))
    assert_close(packed_heads(o_r, 0, b - a, heads), ro, "resumed from bf16 snapshot: out")
    assert_close(np64(f_r[0]), rs, "resumed from bf16 snapshot: state")


def test_no_snapshot_table_stores_nothing():
    """snapshot_interval > 0 with no slot table (or an empty one, as when no sequence reaches
    the interval) stores no snapshot and leaves the pool untouched."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    xv = synth.varlen_inputs([100, 30], H, seed=4321, device="cuda")
    pool = torch.full((3, H, 128, 128), 7.0, device="cuda")
    pool[0] = xv["init_states"][0]
    before = pool.clone()
    o, f = kda.kda_varlen_fwd_pool(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], xv["cu_seqlens"], pool,
                                   torch.tensor([0, -1], device="cuda"), None, snapshot_interval=128)
    o2, f2 = kda.kda_varlen_fwd_pool(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], xv["cu_seqlens"], pool,
                                     torch.tensor([0, -1], device="cuda"),
                                     torch.empty(0, dtype=torch.int64, device="cuda"), snapshot_interval=128)
    torch.cuda.synchronize()
    assert torch.equal(pool, before)
    assert torch.equal(o, o2) and torch.equal(f, f2)
    assert kda.kda_get_device_status() == 0
