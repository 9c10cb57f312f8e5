"""Thin Python binding of libkda (include/kda.h), same names as the C ABI.

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, outputs are allocated with torch when the caller passes none, and
the raw device pointers go to the C entry points on the current CUDA stream.
Every step of the computation runs inside libkda's kernels.  If the shared
library is missing the import of this module's functions fails loudly; there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_BF16, KDA_F32 = 0, 1
KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_MISALIGNED = 0, 1, 2, 3
KDA_ERR_CUDA, KDA_ERR_TIMEOUT, KDA_ERR_WORKSPACE, KDA_STATUS_GATE_RANGE = 4, 5, 6, 7
KDA_STATUS_SLOT_RANGE, KDA_ERR_SCRATCH_TOO_SMALL = 8, 9
KDA_NOALLOC_SCRATCH_BYTES = 128 << 20
KDA_OP_CHUNK, KDA_OP_VARLEN, KDA_OP_DECODE, KDA_OP_BWD, KDA_OP_CHUNK_BWD = 0, 1, 2, 3, 4
KDA_GATE_CHANNEL, KDA_GATE_HEAD, KDA_GATE_NONE = 0, 1, 2

_lib = None


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {kda_status_string(code)} (code {code})")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded libkda.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkda.so not found at {LIB_PATH}; build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        L.kda_chunk_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I64, I, I, I, I, I, I, P, SZ, P]
        L.kda_varlen_fwd.argtypes = [P, P, P, P, P, P, I, I64, I, I, I, I, P, P, I64, P, P, P, I, I, P, SZ, P]
        L.kda_decode_step.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P]
        L.kda_decode_step_bf16state.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P]
        L.kda_gdn_chunk_fwd.argtypes = L.kda_chunk_fwd.argtypes
        L.kda_gdn_varlen_fwd.argtypes = L.kda_varlen_fwd.argtypes
        L.kda_gdn_decode_step.argtypes = L.kda_decode_step.argtypes
        L.kda_gdn_decode_step_bf16state.argtypes = L.kda_decode_step.argtypes
        L.kda_chunk_fwd_host.argtypes = [P, P, P, P, P, P, P, P, I, I64, I, I, I, I, I, I64, P, SZ, P]
        L.kda_host_fwd_workspace_size.argtypes = [I, I, I, I, I64, I, I]
        L.kda_host_fwd_workspace_size.restype = SZ
        L.kda_bwd.argtypes = [P, P, P, P, I, P, P, P, P, P, I, I64, I, I, I, P, P, P, P, P, P, I, P, SZ, P]
        L.kda_bwd_noalloc.argtypes = [P, P, P, P, I, P, P, P, P, P, I, I64, I, I, I, P, P, P, P, P, P, I, P]
        L.kda_chunk_bwd.argtypes = [P, P, P, P, I, P, P, P, P, P, I, I64, I, I, I, I, P, P, P, P, P, P, I, P, SZ,
                                    P]
        L.kda_varlen_fwd_pool.argtypes = [P, P, P, P, I, P, P, I, I64, I, I, I, I, P, I64, I, P, I64, P, P, P, P, I,
                                          I, P, SZ, P]
        L.kda_snapshot_count.argtypes = [I64, I64]
        L.kda_snapshot_count.restype = I64
        L.kda_snapshot_offsets.argtypes = [P, I, I64, P]
        L.kda_snapshot_lookup.argtypes = [P, I, I, I64, I64, P]
        L.kda_snapshot_lookup.restype = I64
        L.kda_workspace_size.argtypes = [I, I, I64, I, I, I, I]
        L.kda_workspace_size.restype = SZ
        L.kda_status_string.argtypes = [I]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_get_device_status.argtypes = [P]
        L.kda_selftest_bounded_wait.argtypes = [P]
        for f in (L.kda_chunk_fwd, L.kda_varlen_fwd, L.kda_decode_step, L.kda_decode_step_bf16state,
                  L.kda_gdn_chunk_fwd, L.kda_gdn_varlen_fwd, L.kda_gdn_decode_step, L.kda_varlen_fwd_pool, L.kda_bwd,
                  L.kda_bwd_noalloc, L.kda_chunk_bwd, L.kda_selftest_bounded_wait, L.kda_gdn_decode_step_bf16state,
                  L.kda_chunk_fwd_host,
                  L.kda_snapshot_offsets,
                  L.kda_get_device_status):
            f.restype = I
        _lib = L
    return _lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use bfloat16 or float32")


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libkda must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(rc: int, where: str):
    if rc != KDA_OK:
        raise KdaError(rc, where)


def _dtype_of(code: int):
    return torch.bfloat16 if code == KDA_BF16 else torch.float32


def kda_status_string(code: int) -> str:
    return lib().kda_status_string(int(code)).decode()


def kda_snapshot_count(seqlen: int, interval: int) -> int:
    return int(lib().kda_snapshot_count(int(seqlen), int(interval)))


def kda_snapshot_offsets(cu_seqlens_host, interval: int) -> torch.Tensor:
    """HOST int64 [N+1] snapshot offsets for HOST cu_seqlens (a list or CPU tensor)."""
    cu = torch.as_tensor(cu_seqlens_host, dtype=torch.int64).cpu().contiguous()
    N = cu.numel() - 1
    off = torch.empty(N + 1, dtype=torch.int64)
    _check(lib().kda_snapshot_offsets(_ptr(cu), N, int(interval), _ptr(off)), "kda_snapshot_offsets")
    return off


def kda_snapshot_lookup(offsets_host, seq: int, interval: int, prefix_len: int):
    """(index, covered): the latest snapshot of sequence `seq` covering at most `prefix_len`
    tokens (index into the packed snapshots, tokens it covers), or (-1, 0) if there is none."""
    off = torch.as_tensor(offsets_host, dtype=torch.int64).cpu().contiguous()
    cov = ctypes.c_int64(0)
    idx = lib().kda_snapshot_lookup(_ptr(off), off.numel() - 1, int(seq), int(interval), int(prefix_len),
                                    ctypes.byref(cov))
    if idx == -2:
        raise KdaError(KDA_ERR_INVALID_ARG, "kda_snapshot_lookup")
    return int(idx), int(cov.value)


def kda_workspace_size(op: int, B: int, T: int, H: int, dk: int = 128, dv: int = 128, chunk: int = 64) -> int:
    return int(lib().kda_workspace_size(int(op), int(B), int(T), int(H), int(dk), int(dv), int(chunk)))


def kda_selftest_bounded_wait(stream=None) -> None:
    """Launch the bounded-wait diagnostic (about 2 s; afterwards the device status reads
    KDA_ERR_TIMEOUT)."""
    st = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream(None)
    _check(lib().kda_selftest_bounded_wait(st), "kda_selftest_bounded_wait")


def kda_get_device_status(stream=None) -> int:
    st = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream(None)
    return int(lib().kda_get_device_status(st))


def _workspace(op, B, T, H, dk, dv, chunk, device, workspace):
    need = kda_workspace_size(op, B, T, H, dk, dv, chunk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace, (workspace.numel() * workspace.element_size() if workspace is not None else 0)


def _chunk(name, q, k, v, log_alpha, beta, init_state, out, final_state, chunk, out_dtype, return_final_state,
           workspace):
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(B, T, H, dv, dtype=out_dtype, device=q.device)
    if final_state is None and return_final_state:
        final_state = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    ws, ws_bytes = _workspace(KDA_OP_CHUNK, B, T, H, dk, dv, chunk, q.device, workspace)
    rc = getattr(lib(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(init_state), _ptr(out),
                              _ptr(final_state), B, T, H, dk, dv, int(chunk), _dt(q), _dt(out), _ptr(ws), ws_bytes,
                              _stream(q.device))
    _check(rc, name)
    return out, final_state


def kda_chunk_fwd(q, k, v, log_alpha, beta, init_state=None, out=None, final_state=None, *, chunk: int = 64,
                  out_dtype=torch.float32, return_final_state: bool = True, workspace=None):
    """Batched prefill.  q,k [B,T,H,dk], v [B,T,H,dv] (bf16/fp32), log_alpha [B,T,H,dk] fp32,
    beta [B,T,H] fp32, init_state [B,H,dk,dv] fp32 or None.  Returns (out, final_state)."""
    return _chunk("kda_chunk_fwd", q, k, v, log_alpha, beta, init_state, out, final_state, chunk, out_dtype,
                  return_final_state, workspace)


def kda_chunk_fwd_host(q, k, v, log_alpha, beta, init_state=None, out=None, final_state=None, *,
                       out_dtype=torch.float32, segment_tokens: int = 0, workspace=None, device=None):
    """kda_chunk_fwd on HOST tensors (CPU; page-locked for overlap), streamed through the GPU
    in segments.  init_state is a device tensor or None; out and final_state are host tensors
    (allocated pinned if None).  Returns (out, final_state) once the call is enqueued on the
    current stream of `device` (cuda:0 by default); synchronise before reading them."""
    for t in (q, k, v, log_alpha, beta):
        if t.is_cuda:
            raise ValueError("kda_chunk_fwd_host takes host tensors")
    dev = torch.device(device or "cuda")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(B, T, H, dv, dtype=out_dtype, pin_memory=True)
    if final_state is None:
        final_state = torch.empty(B, H, dk, dv, dtype=torch.float32, pin_memory=True)
    if workspace is None:
        need = lib().kda_host_fwd_workspace_size(B, H, dk, dv, int(segment_tokens), _dt(q), _dt(out))
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=dev)
    rc = lib().kda_chunk_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(init_state), _ptr(out),
                                  _ptr(final_state), B, T, H, dk, dv, _dt(q), _dt(out), int(segment_tokens),
                                  _ptr(workspace), workspace.numel(), _stream(dev))
    _check(rc, "kda_chunk_fwd_host")
    return out, final_state


def kda_gdn_chunk_fwd(q, k, v, log_alpha, beta, init_state=None, out=None, final_state=None, *, chunk: int = 64,
                      out_dtype=torch.float32, return_final_state: bool = True, workspace=None):
    """kda_chunk_fwd with one log-decay per (token, head): log_alpha [B,T,H] fp32 (Gated
    DeltaNet), or None for no decay (DeltaNet)."""
    return _chunk("kda_gdn_chunk_fwd", q, k, v, log_alpha, beta, init_state, out, final_state, chunk, out_dtype,
                  return_final_state, workspace)


def _varlen(name, q, k, v, log_alpha, beta, cu_seqlens, init_states, chunk, snapshot_interval, cu_seqlens_host,
            out, final_states, snapshots, out_dtype, workspace):
    Ttot, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty(Ttot, H, dv, dtype=out_dtype, device=q.device)
    if final_states is None:
        final_states = torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device)
    snap_off = None
    if snapshot_interval:
        cu_h = cu_seqlens.cpu() if cu_seqlens_host is None else torch.as_tensor(cu_seqlens_host)
        off_h = kda_snapshot_offsets(cu_h, snapshot_interval)
        snap_off = off_h.to(q.device)
        if snapshots is None:
            snapshots = torch.empty(max(int(off_h[-1]), 1), H, dk, dv, dtype=torch.float32, device=q.device)
    ws, ws_bytes = _workspace(KDA_OP_VARLEN, N, Ttot, H, dk, dv, chunk, q.device, workspace)
    rc = getattr(lib(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(cu_seqlens), N, Ttot,
                              H, dk, dv, int(chunk), _ptr(init_states), _ptr(final_states), int(snapshot_interval),
                              _ptr(snap_off), _ptr(snapshots) if snapshot_interval else None, _ptr(out), _dt(q),
                              _dt(out), _ptr(ws), ws_bytes, _stream(q.device))
    _check(rc, name)
    if snapshot_interval and snapshots is not None:
        snapshots = snapshots[: int(snap_off[-1].item())] if snapshots.shape[0] > 0 else snapshots
    return out, final_states, (snapshots if snapshot_interval else None)


def kda_varlen_fwd(q, k, v, log_alpha, beta, cu_seqlens, init_states=None, *, chunk: int = 64,
                   snapshot_interval: int = 0, cu_seqlens_host=None, out=None, final_states=None,
                   snapshots=None, out_dtype=torch.float32, workspace=None):
    """Packed sequences.  q,k [Ttot,H,dk], v [Ttot,H,dv], log_alpha [Ttot,H,dk], beta [Ttot,H];
    cu_seqlens int64 [N+1] on the device.  Returns (out, final_states, snapshots or None)."""
    return _varlen("kda_varlen_fwd", q, k, v, log_alpha, beta, cu_seqlens, init_states, chunk, snapshot_interval,
                   cu_seqlens_host, out, final_states, snapshots, out_dtype, workspace)


def kda_varlen_fwd_pool(q, k, v, log_alpha, beta, cu_seqlens, pool, init_slots=None, snap_slots=None, *,
                        gate: int = KDA_GATE_CHANNEL, chunk: int = 64, snapshot_interval: int = 0,
                        cu_seqlens_host=None, out=None, final_states=None, out_dtype=torch.float32, workspace=None):
    """Packed sequences over a state pool [pool_slots,H,dk,dv] (fp32, or bf16 storage with fp32
    arithmetic): sequence s starts from slot
    init_slots[s] (-1: zeros; None: all zeros) and snapshot m of sequence s goes to slot
    snap_slots[offsets[s] + m - 1] (-1: not stored).  log_alpha's layout is given by `gate`.
    Returns (out, final_states); the snapshots are in the pool."""
    Ttot, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty(Ttot, H, dv, dtype=out_dtype, device=q.device)
    if final_states is None:
        final_states = torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device)
    if pool.dtype not in (torch.float32, torch.bfloat16) or tuple(pool.shape[1:]) != (H, dk, dv):
        raise ValueError(f"pool must be float32 or bfloat16 [slots, {H}, {dk}, {dv}]")
    snap_off = None
    if snapshot_interval:
        cu_h = cu_seqlens.cpu() if cu_seqlens_host is None else torch.as_tensor(cu_seqlens_host)
        snap_off = kda_snapshot_offsets(cu_h, snapshot_interval).to(q.device)
    for name, t in (("init_slots", init_slots), ("snap_slots", snap_slots)):
        if t is not None and t.dtype != torch.int64:
            raise TypeError(f"{name} must be int64")
    ws, ws_bytes = _workspace(KDA_OP_VARLEN, N, Ttot, H, dk, dv, chunk, q.device, workspace)
    rc = lib().kda_varlen_fwd_pool(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), int(gate), _ptr(beta),
                                   _ptr(cu_seqlens), N, Ttot, H, dk, dv, int(chunk), _ptr(pool), pool.shape[0],
                                   _dt(pool), _ptr(init_slots), int(snapshot_interval), _ptr(snap_off),
                                   _ptr(snap_slots),
                                   _ptr(final_states), _ptr(out), _dt(q), _dt(out), _ptr(ws), ws_bytes,
                                   _stream(q.device))
    _check(rc, "kda_varlen_fwd_pool")
    return out, final_states


def kda_gdn_varlen_fwd(q, k, v, log_alpha, beta, cu_seqlens, init_states=None, *, chunk: int = 64,
                       snapshot_interval: int = 0, cu_seqlens_host=None, out=None, final_states=None,
                       snapshots=None, out_dtype=torch.float32, workspace=None):
    """kda_varlen_fwd with log_alpha [Ttot,H] (Gated DeltaNet) or None (DeltaNet)."""
    return _varlen("kda_gdn_varlen_fwd", q, k, v, log_alpha, beta, cu_seqlens, init_states, chunk,
                   snapshot_interval, cu_seqlens_host, out, final_states, snapshots, out_dtype, workspace)


def _decode(fn, name, state_dtype, q, k, v, log_alpha, beta, state, out, out_dtype):
    if state.dtype != state_dtype:
        raise TypeError(f"{name}: state must be {state_dtype}, got {state.dtype}")
    B, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(B, H, dv, dtype=out_dtype, device=q.device)
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(state), _ptr(out), B, H, dk, dv, _dt(q),
            _dt(out), _stream(q.device))
    _check(rc, name)
    return out


def kda_decode_step(q, k, v, log_alpha, beta, state, out=None, *, out_dtype=torch.float32):
    """One token per session: q,k [B,H,dk], v [B,H,dv], log_alpha [B,H,dk], beta [B,H];
    state [B,H,dk,dv] fp32 is updated in place.  Returns out [B,H,dv]."""
    return _decode(lib().kda_decode_step, "kda_decode_step", torch.float32, q, k, v, log_alpha, beta, state, out,
                   out_dtype)


def kda_decode_step_bf16state(q, k, v, log_alpha, beta, state, out=None, *, out_dtype=torch.float32):
    """kda_decode_step with a bf16-stored state [B,H,dk,dv] (updated in place; the step
    itself runs in fp32 and the output is read before the state is rounded)."""
    return _decode(lib().kda_decode_step_bf16state, "kda_decode_step_bf16state", torch.bfloat16, q, k, v, log_alpha,
                   beta, state, out, out_dtype)


def kda_gdn_decode_step_bf16state(q, k, v, log_alpha, beta, state, out=None, *, out_dtype=torch.float32):
    """kda_gdn_decode_step with a bf16-stored state (fp32 arithmetic)."""
    return _decode(lib().kda_gdn_decode_step_bf16state, "kda_gdn_decode_step_bf16state", torch.bfloat16, q, k, v,
                   log_alpha, beta, state, out, out_dtype)


def kda_gdn_decode_step(q, k, v, log_alpha, beta, state, out=None, *, out_dtype=torch.float32):
    """kda_decode_step with log_alpha [B,H] (Gated DeltaNet) or None (DeltaNet); fp32 state."""
    return _decode(lib().kda_gdn_decode_step, "kda_gdn_decode_step", torch.float32, q, k, v, log_alpha, beta, state,
                   out, out_dtype)


def kda_bwd(q, k, v, log_alpha, beta, d_out, init_state=None, d_final_state=None, *, gate: int = KDA_GATE_CHANNEL,
            cu_seqlens=None, return_d_init: bool = True, chunk: int = 64, workspace=None,
            no_alloc: bool = False) -> dict:
    """Gradients of L = sum <d_out, o> + <d_final_state, S_final> through the forward of
    kda_chunk_fwd (batched q [B,T,H,dk] when cu_seqlens is None, else packed [Ttot,H,dk]).
    log_alpha's layout follows `gate`.  Returns dict(dq, dk, dv, dlog_alpha, dbeta, d_init).
    chunk=64 calls kda_chunk_bwd (chunked), chunk=1 the token-serial kda_bwd; no_alloc=True
    calls kda_bwd_noalloc (token-serial, the library's static scratch, no workspace)."""
    if cu_seqlens is None:
        N, T, H, dk = q.shape
        t_arg, t_total = T, N * T
    else:
        t_total, H, dk = q.shape
        N = cu_seqlens.numel() - 1
        t_arg = t_total
    dv = v.shape[-1]
    f32 = dict(dtype=torch.float32, device=q.device)
    g = {"dq": torch.empty(q.shape, **f32), "dk": torch.empty(k.shape, **f32), "dv": torch.empty(v.shape, **f32),
         "dlog_alpha": None if gate == KDA_GATE_NONE else torch.empty(log_alpha.shape, **f32),
         "dbeta": torch.empty(beta.shape, **f32),
         "d_init": torch.empty(N, H, dk, dv, **f32) if return_d_init else None}
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), int(gate), _ptr(beta), _ptr(init_state), _ptr(d_out),
            _ptr(d_final_state), _ptr(cu_seqlens), N, t_arg, H, dk, dv)
    grads = (_ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dlog_alpha"]), _ptr(g["dbeta"]),
             _ptr(g["d_init"]), _dt(q))
    if no_alloc:
        _check(lib().kda_bwd_noalloc(*head, *grads, _stream(q.device)), "kda_bwd_noalloc")
        return g
    if workspace is None:
        need = kda_workspace_size(KDA_OP_CHUNK_BWD, N, t_total, H, dk, dv, chunk)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if chunk == 1:
        rc, name = lib().kda_bwd(*head, *grads, _ptr(workspace), workspace.numel(), _stream(q.device)), "kda_bwd"
    else:
        rc = lib().kda_chunk_bwd(*head, int(chunk), *grads, _ptr(workspace), workspace.numel(), _stream(q.device))
        name = "kda_chunk_bwd"
    _check(rc, name)
    return g
