"""fp64 CPU oracle for the Kimi-K3 shared-expert SwiGLU MLP (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
library never loads it, and it shares no code with the CUDA path: the C source
next to this file is the whole implementation, this module only marshals numpy
arrays into it.

Functions and the passages they follow are documented in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, F32 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (plain C11, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                                  os.path.getmtime(os.path.join(_HERE, "oracle.h"))))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               "-Wall", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            ci = ctypes.c_int
            L.oracle_bf16_to_f64.restype = ctypes.c_double
            L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
            L.oracle_f64_to_bf16_rne.argtypes = [ctypes.c_double]
            L.oracle_silu.restype = ctypes.c_double
            L.oracle_silu.argtypes = [ctypes.c_double]
            L.oracle_swiglu_hidden.restype = None
            L.oracle_swiglu_hidden.argtypes = [P, i64, i64, i64, P, i64, i64, P, i64, P, P, P, ci]
            L.oracle_mlp_forward.restype = None
            L.oracle_mlp_forward.argtypes = [P, i64, i64, i64, P, P, P, i64, P, P, P, ci]
            L.oracle_shard_partial.restype = ci
            L.oracle_shard_partial.argtypes = [P, i64, i64, i64, P, P, ci, ci, P, i64, P, P, ci, ci]
            L.oracle_shard_group_sum.restype = ci
            L.oracle_shard_group_sum.argtypes = [P, i64, i64, i64, P, P, ci, ci, ci, P, i64, P, P, ci, ci]
            L.oracle_shard_sum.restype = None
            L.oracle_shard_sum.argtypes = [P, ci, ci, i64, i64, P]
            L.oracle_rank_major_to_logical.restype = ci
            L.oracle_rank_major_to_logical.argtypes = [i64, i64, ci, P]
            L.oracle_merged_proj.restype = ci
            L.oracle_merged_proj.argtypes = [P, i64, i64, P, i64, i64, ci, P, i64, P, P, P, ci]
            L.oracle_reorder.restype = ci
            L.oracle_reorder.argtypes = [P, P, i64, i64, i64, ci]
            _lib = L
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint16)


def _rows(rows, T):
    if rows is None:
        return None, T
    r = np.ascontiguousarray(rows, dtype=np.int64)
    if r.size and (r.min() < 0 or r.max() >= T):
        raise ValueError("row index out of range")
    return r, int(r.size)


# ---------------------------------------------------------------------------------------
# scalar helpers
# ---------------------------------------------------------------------------------------

def bf16_to_f64(b: int) -> float:
    return lib().oracle_bf16_to_f64(int(b) & 0xFFFF)


def f64_to_bf16(d: float) -> int:
    return int(lib().oracle_f64_to_bf16_rne(float(d)))


def silu(z: float) -> float:
    return lib().oracle_silu(float(z))


def bf16_array_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact decode of bf16 bit patterns (a bit shift; no arithmetic)."""
    b = _u16(b)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------------------
# array entry points
# ---------------------------------------------------------------------------------------

def swiglu_hidden(x, w_gate_up, I, j_begin=0, j_end=None, rows=None, nthreads=None,
                  want_gu=False):
    x = _u16(x); w = _u16(w_gate_up)
    T, H = x.shape
    j_end = I if j_end is None else j_end
    r, n = _rows(rows, T)
    width = j_end - j_begin
    h = np.empty((n, width), dtype=np.uint16)
    g = np.empty((n, width), dtype=np.float64) if want_gu else None
    u = np.empty((n, width), dtype=np.float64) if want_gu else None
    lib().oracle_swiglu_hidden(_p(x), T, H, I, _p(w), j_begin, j_end, _p(r), n, _p(h), _p(g), _p(u),
                               nthreads or default_threads())
    return (h, g, u) if want_gu else h


def mlp_forward(x, w_gate_up, w_down, rows=None, nthreads=None):
    """Replicated layer -> (y bf16 bits [n x H], y fp64 pre-rounding, h bf16 bits [n x I])."""
    x = _u16(x); wgu = _u16(w_gate_up); wd = _u16(w_down)
    T, H = x.shape
    I = wgu.shape[0] // 2
    assert wgu.shape == (2 * I, H) and wd.shape == (H, I)
    r, n = _rows(rows, T)
    y = np.empty((n, H), dtype=np.uint16)
    yf = np.empty((n, H), dtype=np.float64)
    h = np.empty((n, I), dtype=np.uint16)
    lib().oracle_mlp_forward(_p(x), T, H, I, _p(wgu), _p(wd), _p(r), n, _p(y), _p(yf), _p(h),
                             nthreads or default_threads())
    return y, yf, h


def shard_partial(x, w_gate_up, w_down, tp, rank, dtype=BF16, rows=None, nthreads=None):
    """Partial of one shard -> (p fp64 [n x H], p rounded: uint16 bf16 bits or float32)."""
    x = _u16(x); wgu = _u16(w_gate_up); wd = _u16(w_down)
    T, H = x.shape
    I = wgu.shape[0] // 2
    r, n = _rows(rows, T)
    pf = np.empty((n, H), dtype=np.float64)
    pr = np.empty((n, H), dtype=np.uint16 if dtype == BF16 else np.float32)
    rc = lib().oracle_shard_partial(_p(x), T, H, I, _p(wgu), _p(wd), tp, rank, _p(r), n,
                                    _p(pf), _p(pr), dtype, nthreads or default_threads())
    if rc != 0:
        raise ValueError("invalid shard geometry")
    return pf, pr


def shard_group_sum(x, w_gate_up, w_down, tp, rank_first=0, rank_count=None, dtype=BF16, rows=None,
                    nthreads=None):
    """Sum of shards rank_first.. fp64 partials, rounded once -> (sum fp64 [n x H], rounded)."""
    x = _u16(x); wgu = _u16(w_gate_up); wd = _u16(w_down)
    T, H = x.shape
    I = wgu.shape[0] // 2
    rank_count = tp - rank_first if rank_count is None else rank_count
    r, n = _rows(rows, T)
    sf = np.empty((n, H), dtype=np.float64)
    sr = np.empty((n, H), dtype=np.uint16 if dtype == BF16 else np.float32)
    rc = lib().oracle_shard_group_sum(_p(x), T, H, I, _p(wgu), _p(wd), tp, rank_first, rank_count, _p(r), n,
                                      _p(sf), _p(sr), dtype, nthreads or default_threads())
    if rc != 0:
        raise ValueError("invalid shard geometry")
    return sf, sr


def shard_sum(partials, dtype=BF16):
    p = np.ascontiguousarray(partials, dtype=np.uint16 if dtype == BF16 else np.float32)
    n, T, H = p.shape
    out = np.empty((T, H), dtype=np.uint16)
    lib().oracle_shard_sum(_p(p), dtype, n, T, H, _p(out))
    return out


def rank_major_to_logical(q_dim, kv_dim, tp):
    m = np.empty(q_dim + kv_dim, dtype=np.int64)
    if lib().oracle_rank_major_to_logical(q_dim, kv_dim, tp, _p(m)) != 0:
        raise ValueError("q_dim and kv_dim must be divisible by tp")
    return m


def merged_proj(x, w, q_dim, kv_dim, tp, rows=None, nthreads=None):
    """-> (logical bf16 bits, rank-major bf16 bits, logical fp64)."""
    x = _u16(x); w = _u16(w)
    T, H = x.shape
    C = q_dim + kv_dim
    assert w.shape == (C, H)
    r, n = _rows(rows, T)
    lo = np.empty((n, C), dtype=np.uint16)
    rm = np.empty((n, C), dtype=np.uint16)
    f = np.empty((n, C), dtype=np.float64)
    rc = lib().oracle_merged_proj(_p(x), T, H, _p(w), q_dim, kv_dim, tp, _p(r), n, _p(lo), _p(rm),
                                  _p(f), nthreads or default_threads())
    if rc != 0:
        raise ValueError("q_dim and kv_dim must be divisible by tp")
    return lo, rm, f


def reorder(rank_major, q_dim, kv_dim, tp):
    rm = _u16(rank_major)
    T, C = rm.shape
    out = np.empty_like(rm)
    if lib().oracle_reorder(_p(rm), _p(out), T, q_dim, kv_dim, tp) != 0:
        raise ValueError("q_dim and kv_dim must be divisible by tp")
    return out
