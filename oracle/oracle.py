"""Python wrapper of the fp64 CPU oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The product
library never loads it and it never loads the product library.

What it computes is the Kimi Delta Attention recurrence of the "Kimi K3"
article (lshu.cn/news/263999), §四, with the delta-rule expansion of §三 and
the read of §二.1, in fp64:

    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = S_t^T q_t,          alpha_t = exp(log_alpha_t) per key channel.

``recurrent`` runs it token by token; ``chunked`` runs the naive chunked
rewrite of §六 (recurrent between chunks of C tokens, WY form inside);
``recurrent_bwd`` is the reverse mode of ``recurrent`` (the pages give no
backward; it is derived step by step from the forward definition).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(out_path: str = _LIB_PATH, mutant: int | None = None) -> str:
    """Compile the oracle with gcc (plain -O2, portable: no -march flags)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", out_path, "-lm"]
    if mutant is not None:
        cmd.insert(1, f"-DORACLE_MUTANT={int(mutant)}")
    subprocess.run(cmd, check=True)
    return out_path


def _bind(path: str):
    lib = ctypes.CDLL(path)
    f, d, i64, i32 = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.kda_oracle_recurrent.argtypes = [i64, i64, i32, i32, f, f, f, f, f, d, d, d, i64, d, i32]
    lib.kda_oracle_recurrent.restype = ctypes.c_int
    lib.kda_oracle_chunked.argtypes = [i64, i64, i32, i32, i32, f, f, f, f, f, d, d, d, i64, d, i32]
    lib.kda_oracle_chunked.restype = ctypes.c_int
    lib.kda_oracle_recurrent_bf16state.argtypes = [i64, i64, i32, i32, f, f, f, f, f, d, d, d, i32]
    lib.kda_oracle_recurrent_bf16state.restype = ctypes.c_int
    lib.kda_oracle_round_bf16.argtypes = [d, d, i64]
    lib.kda_oracle_round_bf16.restype = None
    lib.kda_oracle_recurrent_bwd.argtypes = [i64, i64, i32, i32, f, f, f, f, f, d, d, d, d, d, d, d, d, d, i32]
    lib.kda_oracle_recurrent_bwd.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
                build()
            _lib = _bind(_LIB_PATH)
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _run(which, q, k, v, log_alpha, beta, S0, chunk, snap_interval, threads, lib):
    """Shared marshalling. Arrays: q,k,log_alpha [n,T,dk]; v [n,T,dv]; beta [n,T]; S0 [n,dk,dv]."""
    lib = lib or load()
    q, k, v, la, be = _f64(q), _f64(k), _f64(v), _f64(log_alpha), _f64(beta)
    n, T, dk = q.shape
    dv = v.shape[2]
    assert k.shape == (n, T, dk) and la.shape == (n, T, dk) and v.shape == (n, T, dv) and be.shape == (n, T)
    s0 = None if S0 is None else np.ascontiguousarray(np.asarray(S0, dtype=np.float64))
    if s0 is not None:
        assert s0.shape == (n, dk, dv)
    out = np.zeros((n, T, dv), dtype=np.float64)
    Sf = np.zeros((n, dk, dv), dtype=np.float64)
    nsnap = T // snap_interval if snap_interval else 0
    snaps = np.zeros((n, nsnap, dk, dv), dtype=np.float64) if nsnap else None
    threads = threads or os.cpu_count() or 1
    if which == "recurrent":
        rc = lib.kda_oracle_recurrent(n, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(be), _ptr(s0),
                                      _ptr(out), _ptr(Sf), int(snap_interval), _ptr(snaps), int(threads))
    else:
        rc = lib.kda_oracle_chunked(n, T, dk, dv, int(chunk), _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(be),
                                    _ptr(s0), _ptr(out), _ptr(Sf), int(snap_interval), _ptr(snaps), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle {which} failed (rc={rc})")
    return (out, Sf, snaps) if snap_interval else (out, Sf)


def recurrent(q, k, v, log_alpha, beta, S0=None, snap_interval: int = 0, threads: int | None = None, lib=None):
    """Per-token fp64 recurrence.  Returns (out [n,T,dv], S_final [n,dk,dv][, snaps])."""
    return _run("recurrent", q, k, v, log_alpha, beta, S0, 0, snap_interval, threads, lib)


def recurrent_bf16state(q, k, v, log_alpha, beta, S0=None, threads: int | None = None, lib=None):
    """Per-token recurrence (fp64 arithmetic) with the state rounded to bf16 after every token,
    as stored by a decode step that keeps its state in bf16.  Returns (out, S_final)."""
    lib = lib or load()
    q, k, v, la, be = _f64(q), _f64(k), _f64(v), _f64(log_alpha), _f64(beta)
    n, T, dk = q.shape
    dv = v.shape[2]
    s0 = None if S0 is None else np.ascontiguousarray(np.asarray(S0, dtype=np.float64))
    out = np.zeros((n, T, dv), dtype=np.float64)
    Sf = np.zeros((n, dk, dv), dtype=np.float64)
    rc = lib.kda_oracle_recurrent_bf16state(n, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(be), _ptr(s0),
                                            _ptr(out), _ptr(Sf), int(threads or os.cpu_count() or 1))
    if rc != 0:
        raise RuntimeError(f"oracle recurrent_bf16state failed (rc={rc})")
    return out, Sf


def round_bf16(x, lib=None) -> np.ndarray:
    """The oracle's bf16 rounding (to nearest, ties to even) of fp64 values."""
    lib = lib or load()
    x = _f64(x)
    y = np.empty_like(x)
    lib.kda_oracle_round_bf16(_ptr(x), _ptr(y), x.size)
    return y


def chunked(q, k, v, log_alpha, beta, S0=None, chunk: int = 64, snap_interval: int = 0,
            threads: int | None = None, lib=None):
    """Naive chunked rewrite (WY form) in fp64.  Same returns as ``recurrent``."""
    return _run("chunked", q, k, v, log_alpha, beta, S0, chunk, snap_interval, threads, lib)


def recurrent_bwd(q, k, v, log_alpha, beta, S0, dout, dS_final=None, threads: int | None = None, lib=None,
                  mem_budget: int = 2 << 30) -> dict:
    """Gradients of L = sum_t <dout_t, o_t> + <dS_final, S_T> through the per-token recurrence,
    in fp64: dict with dq, dk, dv, dlog_alpha, dbeta (the inputs' layouts) and dS0 [n,dk,dv].
    Each head keeps its T states in memory; threads are capped to stay near ``mem_budget`` bytes."""
    lib = lib or load()
    q, k, v, la, be, do = _f64(q), _f64(k), _f64(v), _f64(log_alpha), _f64(beta), _f64(dout)
    n, T, dk = q.shape
    dv = v.shape[2]
    assert do.shape == (n, T, dv)
    s0 = None if S0 is None else _f64(S0)
    dsf = None if dS_final is None else _f64(dS_final)
    g = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v), "dlog_alpha": np.zeros_like(la),
         "dbeta": np.zeros_like(be), "dS0": np.zeros((n, dk, dv), dtype=np.float64)}
    per_head = max(1, T) * dk * dv * 8
    threads = max(1, min(threads or os.cpu_count() or 1, mem_budget // per_head or 1))
    rc = lib.kda_oracle_recurrent_bwd(n, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(be), _ptr(s0), _ptr(do),
                                      _ptr(dsf), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dlog_alpha"]),
                                      _ptr(g["dbeta"]), _ptr(g["dS0"]), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle recurrent_bwd failed (rc={rc})")
    return g
