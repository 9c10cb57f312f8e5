"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every entry point declared in include/kda.h, and its host helpers and
argument validation behave as documented.  No call here reaches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from kda_recurrent_state_gb300 import binding, build

    build.build()
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"kda_chunk_fwd", "kda_varlen_fwd", "kda_decode_step"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"libkda.so does not export {n}"


def test_snapshot_helpers(L):
    from kda_recurrent_state_gb300 import binding as b

    assert b.kda_snapshot_count(65536, 16384) == 4
    assert b.kda_snapshot_count(16383, 16384) == 0
    assert b.kda_snapshot_count(100, 0) == 0
    assert b.kda_snapshot_count(-5, 64) == 0
    off = b.kda_snapshot_offsets([0, 100, 300, 300, 1000], 64)
    assert off.tolist() == [0, 1, 4, 4, 14]
    with pytest.raises(b.KdaError):
        b.kda_snapshot_offsets([0, 100, 50], 64)  # decreasing cu_seqlens


def test_snapshot_lookup(L):
    from kda_recurrent_state_gb300 import binding as b

    off = b.kda_snapshot_offsets([0, 1000, 1700, 1830], 128)  # 7, 5 and 1 snapshots
    assert off.tolist() == [0, 7, 12, 13]
    assert b.kda_snapshot_lookup(off, 0, 128, 700) == (4, 640)    # snapshot 5 of sequence 0
    assert b.kda_snapshot_lookup(off, 0, 128, 5000) == (6, 896)   # clamped to its last snapshot
    assert b.kda_snapshot_lookup(off, 1, 128, 256) == (8, 256)    # exactly on an interval
    assert b.kda_snapshot_lookup(off, 2, 128, 100) == (-1, 0)     # shorter than one interval
    assert b.kda_snapshot_lookup(off, 2, 128, 130) == (12, 128)
    for bad in [(3, 128, 10), (-1, 128, 10), (0, 0, 10), (0, 128, -1)]:
        with pytest.raises(b.KdaError):
            b.kda_snapshot_lookup(off, *bad)


def test_status_strings(L):
    from kda_recurrent_state_gb300 import binding as b

    for code in range(10):
        assert b.kda_status_string(code).startswith("KDA_")
    assert "unknown" in b.kda_status_string(99)


def _chunk(L, *, q=16, B=1, T=8, H=1, dk=128, dv=128, chunk=64, in_dt=0, out_dt=1, ws=None, ws_bytes=0):
    P = ctypes.c_void_p
    ptr = P(q) if q else None
    return L.kda_chunk_fwd(ptr, ptr, ptr, ptr, ptr, None, ptr, None, B, T, H, dk, dv, chunk, in_dt, out_dt,
                           P(ws) if ws else None, ws_bytes, None)


def test_argument_validation(L):
    from kda_recurrent_state_gb300 import binding as b

    assert _chunk(L, B=-1) == b.KDA_ERR_INVALID_ARG
    assert _chunk(L, dk=64) == b.KDA_ERR_UNSUPPORTED
    assert _chunk(L, chunk=32) == b.KDA_ERR_UNSUPPORTED
    assert _chunk(L, in_dt=7) == b.KDA_ERR_INVALID_ARG
    assert _chunk(L, q=0) == b.KDA_ERR_INVALID_ARG
    assert _chunk(L, q=0x1008) == b.KDA_ERR_MISALIGNED
    assert _chunk(L, B=0) == b.KDA_OK  # nothing to do
    assert _chunk(L, H=0) == b.KDA_OK
    need = L.kda_workspace_size(0, 1, 8, 1, 128, 128, 64)
    assert need == 512  # one int per (sequence, head), rounded up to 256 bytes, and 256 bytes of unit counters
    assert _chunk(L, ws=0x2000, ws_bytes=need - 1) == b.KDA_ERR_WORKSPACE
    assert _chunk(L, ws=0, ws_bytes=0) == b.KDA_ERR_WORKSPACE
    P = ctypes.c_void_p
    # varlen: interval must be a multiple of the chunk; final_states is required
    assert L.kda_varlen_fwd(P(16), P(16), P(16), P(16), P(16), P(16), 2, 100, 1, 128, 128, 64, None, P(16), 100,
                            P(16), P(16), P(16), 0, 1, None, 0, None) == b.KDA_ERR_INVALID_ARG
    assert L.kda_varlen_fwd(P(16), P(16), P(16), P(16), P(16), P(16), 2, 100, 1, 128, 128, 64, None, None, 0,
                            None, None, P(16), 0, 1, None, 0, None) == b.KDA_ERR_INVALID_ARG
    assert L.kda_decode_step(P(16), P(16), P(16), P(16), P(16), P(16), P(16), 2, 2, 96, 128, 0, 1,
                             None) == b.KDA_ERR_UNSUPPORTED
    assert L.kda_decode_step(P(16), P(16), P(16), P(16), P(16), P(0x1004), P(16), 2, 2, 128, 128, 0, 1,
                             None) == b.KDA_ERR_MISALIGNED
    assert L.kda_decode_step(P(16), P(16), P(16), P(16), P(0x1002), P(16), P(16), 2, 2, 128, 128, 0, 1,
                             None) == b.KDA_ERR_MISALIGNED  # beta needs 4 bytes
    assert L.kda_decode_step_bf16state(P(16), P(16), P(16), P(16), P(16), P(16), P(16), 2, 2, 128, 96, 0, 1,
                                       None) == b.KDA_ERR_UNSUPPORTED
    assert L.kda_decode_step_bf16state(P(16), P(16), P(16), P(16), P(16), P(0x1008), P(16), 2, 2, 128, 128, 0,
                                       1, None) == b.KDA_ERR_MISALIGNED  # the state needs 16 bytes
    assert L.kda_decode_step_bf16state(P(16), P(16), P(16), P(16), P(16), P(16), P(16), 0, 2, 128, 128, 0, 1,
                                       None) == b.KDA_OK  # B = 0: nothing to do


def test_gate_validation(L):
    """Per-channel gates are required and 16-byte aligned; scalar gates (Gated DeltaNet) need
    4 bytes; a null gate selects DeltaNet in the scalar entry points only."""
    from kda_recurrent_state_gb300 import binding as b

    P = ctypes.c_void_p

    def chunk(fn, la, dk=128):
        return fn(P(16), P(16), P(16), la, P(16), None, P(16), None, 1, 8, 1, dk, 128, 64, 0, 1, None, 0, None)

    assert chunk(L.kda_chunk_fwd, None) == b.KDA_ERR_INVALID_ARG
    assert chunk(L.kda_chunk_fwd, P(0x1004)) == b.KDA_ERR_MISALIGNED
    assert chunk(L.kda_gdn_chunk_fwd, P(0x1002)) == b.KDA_ERR_MISALIGNED
    assert chunk(L.kda_gdn_chunk_fwd, None, dk=64) == b.KDA_ERR_UNSUPPORTED
    assert L.kda_gdn_varlen_fwd(P(16), P(16), P(16), P(0x1002), P(16), P(16), 2, 100, 1, 128, 128, 64, None,
                                P(16), 0, None, None, P(16), 0, 1, None, 0, None) == b.KDA_ERR_MISALIGNED
    assert L.kda_gdn_varlen_fwd(P(16), P(16), P(16), None, P(16), P(16), 2, 100, 1, 128, 128, 64, None,
                                None, 0, None, None, P(16), 0, 1, None, 0, None) == b.KDA_ERR_INVALID_ARG
    assert L.kda_gdn_decode_step(P(16), P(16), P(16), P(0x1002), P(16), P(16), P(16), 2, 2, 128, 128, 0, 1,
                                 None) == b.KDA_ERR_MISALIGNED
    assert L.kda_decode_step(P(16), P(16), P(16), None, P(16), P(16), P(16), 2, 2, 128, 128, 0, 1,
                             None) == b.KDA_ERR_INVALID_ARG


def test_pool_validation(L):
    from kda_recurrent_state_gb300 import binding as b

    P, I64 = ctypes.c_void_p, ctypes.c_int64

    def pool(gate=0, la=16, pool_ptr=16, slots=4, init=None, interval=0, snap_off=None, snap_slots=None, pool_dt=1):
        return L.kda_varlen_fwd_pool(P(16), P(16), P(16), P(la) if la else None, gate, P(16), P(16), 2, 100, 1, 128,
                                     128, 64, P(pool_ptr) if pool_ptr else None, slots, pool_dt,
                                     P(init) if init else None,
                                     interval, P(snap_off) if snap_off else None,
                                     P(snap_slots) if snap_slots else None, P(16), P(16), 0, 1, None, 0, None)

    assert pool(gate=5) == b.KDA_ERR_INVALID_ARG
    assert pool(slots=-1) == b.KDA_ERR_INVALID_ARG
    assert pool(pool_dt=7) == b.KDA_ERR_INVALID_ARG                       # fp32 or bf16 pools only
    assert pool(pool_ptr=0, init=16) == b.KDA_ERR_INVALID_ARG             # a pool to read from
    assert pool(gate=b.KDA_GATE_HEAD, la=0) == b.KDA_ERR_INVALID_ARG      # scalar gates required
    assert pool(gate=b.KDA_GATE_NONE, la=16) == b.KDA_ERR_INVALID_ARG     # DeltaNet takes no gates
    assert pool(init=0x1004) == b.KDA_ERR_MISALIGNED
    assert pool(pool_ptr=0x1008, init=16) == b.KDA_ERR_MISALIGNED
    assert pool(interval=96, snap_off=16, snap_slots=16) == b.KDA_ERR_INVALID_ARG  # not a chunk multiple
    del I64


def test_bwd_validation(L):
    from kda_recurrent_state_gb300 import binding as b

    P = ctypes.c_void_p

    def bwd(gate=0, la=16, dla=16, dk=128, ws=None, ws_bytes=0, N=1, T=8, in_dt=0):
        ptr = P(16)
        return L.kda_bwd(ptr, ptr, ptr, P(la) if la else None, gate, ptr, None, ptr, None, None, N, T, 1, dk, 128,
                         ptr, ptr, ptr, P(dla) if dla else None, ptr, None, in_dt, P(ws) if ws else None, ws_bytes,
                         None)

    need = b.kda_workspace_size(b.KDA_OP_BWD, 1, 8, 1)
    assert need > 0
    assert bwd(gate=4, ws=0x10000, ws_bytes=need) == b.KDA_ERR_INVALID_ARG
    assert bwd(dk=64, ws=0x10000, ws_bytes=need) == b.KDA_ERR_UNSUPPORTED
    assert bwd(dla=0, ws=0x10000, ws_bytes=need) == b.KDA_ERR_INVALID_ARG               # gated: dlog_alpha needed
    assert bwd(gate=b.KDA_GATE_NONE, ws=0x10000, ws_bytes=need) == b.KDA_ERR_INVALID_ARG  # DeltaNet: no gates
    assert bwd(ws=None) == b.KDA_ERR_WORKSPACE
    assert bwd(ws=0x10000, ws_bytes=need - 1) == b.KDA_ERR_WORKSPACE
    assert bwd(ws=0x10008, ws_bytes=need) == b.KDA_ERR_MISALIGNED
    assert bwd(N=0) == b.KDA_OK
    # workspace: a 64 KB state per 64 tokens (and per sequence) of every head, plus per-(sequence, head) scratch
    assert b.kda_workspace_size(b.KDA_OP_BWD, 4, 4 * 8192, 32) == (32 * (4 * 8192 // 64 + 4 + 1) + 4 * 32 * 16) * 65536


def test_chunk_bwd_validation(L):
    """kda_chunk_bwd: chunk 64 (chunked) or 1 (token-serial); 16-byte aligned q, k, v, d_out for
    chunk 64; its workspace size, written out from the records it holds."""
    from kda_recurrent_state_gb300 import binding as b

    P = ctypes.c_void_p

    def cbwd(chunk=64, q=16, ws=0x10000, ws_bytes=None, N=1, T=8):
        ptr = P(16)
        if ws_bytes is None:
            ws_bytes = b.kda_workspace_size(b.KDA_OP_CHUNK_BWD, N, N * T, 1, chunk=chunk)
        return L.kda_chunk_bwd(P(q), ptr, ptr, ptr, 0, ptr, None, ptr, None, None, N, T, 1, 128, 128, chunk, ptr, ptr,
                               ptr, ptr, ptr, None, 0, P(ws) if ws else None, ws_bytes, None)

    assert cbwd(chunk=16, ws_bytes=1 << 20) == b.KDA_ERR_UNSUPPORTED
    assert cbwd(chunk=0, ws_bytes=1 << 20) == b.KDA_ERR_UNSUPPORTED
    assert cbwd(q=0x1008) == b.KDA_ERR_MISALIGNED        # 8-byte aligned: enough for chunk 1 only
    assert cbwd(chunk=64, ws=None) == b.KDA_ERR_WORKSPACE
    need = b.kda_workspace_size(b.KDA_OP_CHUNK_BWD, 1, 8, 1, chunk=64)
    assert cbwd(ws_bytes=need - 1) == b.KDA_ERR_WORKSPACE
    assert cbwd(N=0) == b.KDA_OK
    # chunk 1 is kda_bwd, with kda_bwd's workspace
    assert b.kda_workspace_size(b.KDA_OP_CHUNK_BWD, 4, 4 * 8192, 32, chunk=1) == \
        b.kda_workspace_size(b.KDA_OP_BWD, 4, 4 * 8192, 32)
    # chunk 64: per chunk-head W~, U', K^ (C x D), E and dS (D x D), T and P (C x C) and three D-vectors;
    # per (chunk + sequence) and head one D x D state; at most T_total / 64 + N chunks
    C, D, N, Tt, H = 64, 128, 4, 4 * 8192, 32
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    nch = (Tt // C + N) * H
    per = 3 * C * D + 2 * D * D + 2 * C * C + 3 * D
    # plus one int per (sequence, head) flagging the units the token-serial backward recomputes, which
    # reuses everything from the records on (so that part is at least kda_bwd's workspace)
    serial = b.kda_workspace_size(b.KDA_OP_BWD, N, Tt, H)
    tail = max(al(nch * per * 4) + al((Tt // C + N) * H * D * D * 4 + N * H * D * D * 4), al(serial))
    want = al((N + 1) * 8) + al(N * H * 4) + tail
    assert b.kda_workspace_size(b.KDA_OP_CHUNK_BWD, N, Tt, H, chunk=64) == want
    # one-token sequences: the token-serial workspace (a checkpoint and 16 scratch states per unit) is
    # the larger part
    assert b.kda_workspace_size(b.KDA_OP_CHUNK_BWD, 8, 8, 2, chunk=64) == \
        al(9 * 8) + al(8 * 2 * 4) + al(b.kda_workspace_size(b.KDA_OP_BWD, 8, 8, 2))
    assert b.kda_workspace_size(b.KDA_OP_CHUNK_BWD, N, Tt, H, chunk=16) == 0


def test_bwd_noalloc_rejects_oversize(L):
    """A problem whose backward scratch exceeds the static 128 MiB is refused before any CUDA call."""
    from kda_recurrent_state_gb300 import binding as b

    P = ctypes.c_void_p
    assert b.kda_workspace_size(b.KDA_OP_BWD, 4, 4 * 8192, 32) > b.KDA_NOALLOC_SCRATCH_BYTES
    ptr = P(16)
    rc = L.kda_bwd_noalloc(ptr, ptr, ptr, ptr, 0, ptr, None, ptr, None, None, 4, 8192, 32, 128, 128, ptr, ptr, ptr,
                           ptr, ptr, None, 0, None)
    assert rc == b.KDA_ERR_SCRATCH_TOO_SMALL
    assert "static" in b.kda_status_string(rc)


def test_host_fwd_validation(L):
    from kda_recurrent_state_gb300 import binding as b

    P = ctypes.c_void_p
    need = L.kda_host_fwd_workspace_size(1, 2, 128, 128, 256, 0, 1)
    # two segments of staging (bf16 q, k, v; fp32 gates, beta, out), two fp32 states and the
    # prefill's own workspace (one int per (sequence, head), rounded up to 256 bytes, and 256 bytes
    # of unit counters)
    assert need == 2 * (256 * 2 * (3 * 256 + 512 + 4 + 512)) + 2 * 2 * 65536 + 512
    ptr = P(16)

    def call(seg=256, ws=0x10000, ws_bytes=need, T=100):
        return L.kda_chunk_fwd_host(ptr, ptr, ptr, ptr, ptr, None, ptr, None, 1, T, 2, 128, 128, 0, 1, seg,
                                    P(ws) if ws else None, ws_bytes, None)

    assert call(seg=100) == b.KDA_ERR_INVALID_ARG       # not a multiple of the chunk
    assert call(ws=None) == b.KDA_ERR_WORKSPACE
    assert call(ws_bytes=need - 1) == b.KDA_ERR_WORKSPACE
    assert call(ws=0x10008) == b.KDA_ERR_MISALIGNED


def test_workspace_size(L):
    from kda_recurrent_state_gb300 import binding as b

    assert b.kda_workspace_size(b.KDA_OP_DECODE, 256, 1, 96) == 0
    # chunk 64: one int per (sequence, head), rounded up to 256 bytes, marking the units the exact
    # pass recomputes, and 256 bytes of unit counters; chunk 1 needs none
    assert b.kda_workspace_size(b.KDA_OP_CHUNK, 1, 131072, 96) == 512 + 256
    assert b.kda_workspace_size(b.KDA_OP_CHUNK, 4, 8192, 32) == 512 + 256
    assert b.kda_workspace_size(b.KDA_OP_VARLEN, 16, 262144, 64) == 4096 + 256
    assert b.kda_workspace_size(b.KDA_OP_CHUNK, 1, 131072, 96, chunk=1) == 0
