"""GB300 (sm_103a) Kimi-K3 shared-expert SwiGLU MLP: thin Python binding of ``libmse.so``.

Every step of the computation runs in the CUDA library behind the C ABI of
``include/mse.h``; this module only marshals torch tensors (device memory and
streams) into pointers and sizes and turns status codes into exceptions.  There
is no CPU or PyTorch fallback: if the library is missing, every call raises.

Functions carry the C-ABI names:
    mlp_swiglu_forward, mlp_swiglu_shard_partial, mlp_swiglu_shard_forward, shard_sum,
    merged_proj_forward, merged_proj_reorder, shard_sequence_parallel_mlp
plus the workspace queries, the device-error poll and the settings, and
``sequence_parallel_mlp``, which takes the sharding decision and makes the matching call.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "MSEError", "lib", "library_path", "mlp_swiglu_forward", "mlp_swiglu_shard_partial", "shard_sum",
    "mlp_swiglu_shard_forward", "shard_sequence_parallel_mlp", "sequence_parallel_mlp",
    "merged_proj_forward", "merged_proj_reorder", "mlp_swiglu_workspace_bytes", "merged_proj_workspace_bytes",
    "poll_device_error", "set_wait_limit_ns", "get_wait_limit_ns", "set_kernel_path", "selftest_wait_timeout",
    "set_phase_events", "set_prefill_kernel", "set_tuning", "BF16", "F32", "PATH_AUTO", "PATH_GENERIC", "PATH_TENSORCORE",
    "PREFILL_AUTO", "PREFILL_SINGLE", "PREFILL_PAIR", "STATUS",
]

BF16, F32 = 0, 1
PATH_AUTO, PATH_GENERIC, PATH_TENSORCORE = 0, 1, 2
PREFILL_AUTO, PREFILL_SINGLE, PREFILL_PAIR = 0, 1, 2
TUNE_ISSUE_GROUP, TUNE_STAGES, TUNE_CACHE_HINTS, TUNE_GRID, TUNE_SPIN_WAIT, TUNE_ONE_LAUNCH, TUNE_PDL = \
    1, 2, 3, 4, 6, 7, 8
TUNE_COOP_FINISH, TUNE_PAIR_MIN_T, TUNE_GRID_DOWN, TUNE_CLUSTER_FINISH = 9, 10, 11, 12
TUNE_L2_PREFETCH, TUNE_SWAPAB_MAX_T, TUNE_X_EARLY, TUNE_DOWN_FLAGS = 14, 15, 16, 17
TUNE_HOST_X_COPIERS, TUNE_PAIR_SPLIT = 18, 19
STATUS = {
    0: "MSE_OK", 1: "MSE_ERR_INVALID_ARG", 2: "MSE_ERR_NOT_DIVISIBLE", 3: "MSE_ERR_GEOMETRY",
    4: "MSE_ERR_WORKSPACE", 5: "MSE_ERR_UNSUPPORTED_DEVICE", 6: "MSE_ERR_CUDA", 7: "MSE_ERR_TIMEOUT",
    8: "MSE_ERR_UNSUPPORTED_SHAPE",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


class MSEError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = int(status)
        self.name = STATUS.get(self.status, f"status {status}")
        super().__init__(f"{func}: {self.name}")


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded C library (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libmse.so not built ({_build.LIB}); run __graft_entry__.build() first")
            L = ctypes.CDLL(_build.LIB)
            P, i64, ci, sz, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64
            sig = {
                "mlp_swiglu_workspace_bytes": (sz, [i64, i64, i64]),
                "merged_proj_workspace_bytes": (sz, [i64, i64, i64, i64]),
                "mlp_swiglu_workspace_sync_range": (ci, [i64, i64, i64, sz, P, P]),
                "merged_proj_workspace_sync_range": (ci, [i64, i64, i64, i64, sz, P, P]),
                "mlp_swiglu_forward": (ci, [P, i64, i64, i64, P, P, P, i64, P, sz, P]),
                "mlp_swiglu_shard_partial": (ci, [P, i64, i64, i64, P, P, ci, ci, ci, P, ci, i64, P, sz, P]),
                "mlp_swiglu_shard_forward": (ci, [P, i64, i64, i64, P, P, ci, ci, ci, P, ci, i64, P, sz, P]),
                "mse_shard_sequence_parallel_mlp": (ci, [ci, ci, ci, ci, i64, i64]),
                "shard_sum": (ci, [P, ci, ci, i64, i64, P, i64, P]),
                "merged_proj_forward": (ci, [P, i64, i64, P, i64, i64, ci, P, P, i64, P, sz, P]),
                "merged_proj_reorder": (ci, [P, P, i64, i64, i64, ci, i64, P]),
                "mlp_swiglu_forward_static_scratch": (ci, [P, i64, i64, i64, P, P, P, i64, P]),
                "mlp_swiglu_host_workspace_bytes": (sz, [i64, i64, i64]),
                "mlp_swiglu_forward_host": (ci, [P, i64, i64, i64, P, P, P, i64, P, sz, P]),
                "mse_poll_device_error": (ci, [P]),
                "mse_set_wait_limit_ns": (None, [u64]),
                "mse_get_wait_limit_ns": (u64, []),
                "mse_set_kernel_path": (ci, [ci]),
                "mse_set_prefill_kernel": (ci, [ci]),
                "mse_set_tuning": (ci, [ci, ci]),
                "mse_mlp_launch_plan": (ci, [i64, i64, i64, ci, ci, ci, ci, P]),
                "mse_merged_launch_plan": (ci, [i64, i64, i64, i64, ci, ci, P]),
                "mse_selftest_wait_timeout": (ci, [u64, P]),
                "mse_set_phase_events": (None, [P, P, P]),
                "mse_status_string": (ctypes.c_char_p, [ci]),
                "mse_version": (ctypes.c_char_p, []),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


# ---------------------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(func: str, status: int) -> None:
    if status != 0:
        raise MSEError(func, status)


def _need(t, name: str, dtypes, ndim: int):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or t.dtype not in dtypes or t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name}: need a contiguous {ndim}-d CUDA tensor of {dtypes}, got "
                         f"{t.dtype} {tuple(t.shape)} on {t.device}")
    return t


def _bf16s():
    torch = _torch()
    return (torch.bfloat16, torch.int16, torch.uint16)


def _dtype_code(dtype) -> int:
    torch = _torch()
    if dtype in (torch.bfloat16, BF16):
        return BF16
    if dtype in (torch.float32, F32):
        return F32
    raise ValueError(f"partial dtype must be bfloat16 or float32, got {dtype}")


def _workspace(nbytes: int, device):
    torch = _torch()
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------------------

def mlp_swiglu_workspace_bytes(T: int, H: int, I: int) -> int:
    return int(lib().mlp_swiglu_workspace_bytes(T, H, I))


def merged_proj_workspace_bytes(T: int, H: int, q_dim: int, kv_dim: int) -> int:
    return int(lib().merged_proj_workspace_bytes(T, H, q_dim, kv_dim))


def mlp_swiglu_workspace_sync_range(T: int, H: int, I: int, workspace_bytes: int) -> tuple[int, int]:
    """(offset, bytes) of the sync words inside an MLP workspace of workspace_bytes."""
    off, n = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("mlp_swiglu_workspace_sync_range",
           lib().mlp_swiglu_workspace_sync_range(T, H, I, workspace_bytes, ctypes.byref(off), ctypes.byref(n)))
    return int(off.value), int(n.value)


def merged_proj_workspace_sync_range(T: int, H: int, q_dim: int, kv_dim: int, workspace_bytes: int) -> tuple[int, int]:
    """(offset, bytes) of the tile counters inside a merged-projection workspace."""
    off, n = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("merged_proj_workspace_sync_range",
           lib().merged_proj_workspace_sync_range(T, H, q_dim, kv_dim, workspace_bytes, ctypes.byref(off),
                                                  ctypes.byref(n)))
    return int(off.value), int(n.value)


def new_mlp_workspace(T: int, H: int, I: int, device="cuda"):
    """A zero-filled workspace for mlp_swiglu_forward / mlp_swiglu_shard_partial."""
    return _workspace(mlp_swiglu_workspace_bytes(T, H, I), device)


def new_host_workspace(T: int, H: int, I: int, device="cuda"):
    """A zero-filled workspace for mlp_swiglu_forward_host."""
    return _workspace(mlp_swiglu_host_workspace_bytes(T, H, I), device)


def new_merged_workspace(T: int, H: int, q_dim: int, kv_dim: int, device="cuda"):
    return _workspace(merged_proj_workspace_bytes(T, H, q_dim, kv_dim), device)


def mlp_swiglu_forward(x, w_gate_up, w_down, y=None, workspace=None, stream=None):
    """y [T, H] = W_down (silu(W_gate x) * (W_up x)); x [T, H], w_gate_up [2I, H], w_down [H, I]."""
    torch = _torch()
    _need(x, "x", _bf16s(), 2)
    _need(w_gate_up, "w_gate_up", _bf16s(), 2)
    _need(w_down, "w_down", _bf16s(), 2)
    T, H = x.shape
    I = w_down.shape[1]
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", _bf16s(), 2)
    if workspace is None:
        workspace = new_mlp_workspace(T, H, I, x.device)
    st = lib().mlp_swiglu_forward(_ptr(x), T, H, I, _ptr(w_gate_up), _ptr(w_down), _ptr(y), y.numel(),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("mlp_swiglu_forward", st)
    return y


def mlp_swiglu_host_workspace_bytes(T: int, H: int, I: int) -> int:
    return int(lib().mlp_swiglu_host_workspace_bytes(T, H, I))


def mlp_swiglu_forward_host(x_host, w_gate_up, w_down, y_host=None, workspace=None, stream=None):
    """The layer with x and y in page-locked host memory (pinned CPU tensors); y_host holds
    the result once the stream has reached the end of the call."""
    torch = _torch()
    if x_host.is_cuda or x_host.dtype not in _bf16s() or x_host.dim() != 2 or not x_host.is_contiguous() \
            or not x_host.is_pinned():
        raise ValueError("x_host: need a contiguous 2-d pinned CPU bf16 tensor")
    _need(w_gate_up, "w_gate_up", _bf16s(), 2)
    _need(w_down, "w_down", _bf16s(), 2)
    T, H = x_host.shape
    I = w_down.shape[1]
    if y_host is None:
        y_host = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    if workspace is None:
        workspace = new_host_workspace(T, H, I, w_down.device)
    st = lib().mlp_swiglu_forward_host(_ptr(x_host), T, H, I, _ptr(w_gate_up), _ptr(w_down), _ptr(y_host),
                                       y_host.numel(), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream))
    _check("mlp_swiglu_forward_host", st)
    return y_host


def mlp_swiglu_shard_partial(x, w_gate_up, w_down, tp, rank_first=0, rank_count=None, partial_dtype=None,
                             partials=None, workspace=None, stream=None):
    """Partials [rank_count, T, H] of shards rank_first.. of a tp-way intermediate split."""
    torch = _torch()
    _need(x, "x", _bf16s(), 2)
    T, H = x.shape
    I = w_down.shape[1]
    rank_count = tp - rank_first if rank_count is None else rank_count
    code = _dtype_code(torch.bfloat16 if partial_dtype is None else partial_dtype)
    if partials is None:
        partials = torch.empty((max(rank_count, 0), T, H), dtype=torch.float32 if code == F32 else torch.bfloat16,
                               device=x.device)
    if workspace is None:
        workspace = new_mlp_workspace(T, H, I, x.device)
    st = lib().mlp_swiglu_shard_partial(_ptr(x), T, H, I, _ptr(w_gate_up), _ptr(w_down), tp, rank_first,
                                        rank_count, _ptr(partials), code, partials.numel(), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream))
    _check("mlp_swiglu_shard_partial", st)
    return partials


def mlp_swiglu_shard_forward(x, w_gate_up, w_down, tp, rank_first=0, rank_count=None, out_dtype=None,
                             out=None, workspace=None, stream=None):
    """Sum [T, H] of the partials of shards rank_first.. of a tp-way intermediate split,
    reduced inside the down projection (no partial is rounded or stored)."""
    torch = _torch()
    _need(x, "x", _bf16s(), 2)
    _need(w_gate_up, "w_gate_up", _bf16s(), 2)
    _need(w_down, "w_down", _bf16s(), 2)
    T, H = x.shape
    I = w_down.shape[1]
    rank_count = tp - rank_first if rank_count is None else rank_count
    code = _dtype_code(torch.bfloat16 if out_dtype is None else out_dtype)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32 if code == F32 else torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = new_mlp_workspace(T, H, I, x.device)
    st = lib().mlp_swiglu_shard_forward(_ptr(x), T, H, I, _ptr(w_gate_up), _ptr(w_down), tp, rank_first,
                                        rank_count, _ptr(out), code, out.numel(), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream))
    _check("mlp_swiglu_shard_forward", st)
    return out


def shard_sequence_parallel_mlp(enabled, use_sequence_parallel, eligible, tp_size, hidden_size,
                                intermediate_size) -> bool:
    """True when the MLP is to be TP-sharded under sequence parallelism, False when it
    stays replicated (the library's host-side gate; no GPU needed)."""
    return bool(lib().mse_shard_sequence_parallel_mlp(int(bool(enabled)), int(bool(use_sequence_parallel)),
                                                      int(bool(eligible)), int(tp_size), int(hidden_size),
                                                      int(intermediate_size)))


def sequence_parallel_mlp(x, w_gate_up, w_down, tp, enabled, use_sequence_parallel=True, eligible=True,
                          out=None, workspace=None, stream=None):
    """The MLP block of a tp-rank sequence-parallel group on one GPU.

    ``x`` [T, H] holds the group's tokens, rank r's own tokens being the row block
    [r*T/tp, (r+1)*T/tp).  Returns (out [T, H] bf16, sharded); rank r's result is the same
    row block of ``out``.  Sharded: every shard's partial over the gathered tokens, summed
    in the down projection (mlp_swiglu_shard_forward).  Replicated: each rank's full MLP
    on its own tokens, which for independent token rows is one mlp_swiglu_forward call."""
    _need(x, "x", _bf16s(), 2)
    T, H = x.shape
    I = w_down.shape[1]
    if tp < 1 or T % tp != 0:
        raise ValueError(f"{T} tokens cannot be split into {tp} equal rank blocks")
    shard = shard_sequence_parallel_mlp(enabled, use_sequence_parallel, eligible, tp, H, I)
    if shard:
        return mlp_swiglu_shard_forward(x, w_gate_up, w_down, tp, out=out, workspace=workspace,
                                        stream=stream), True
    return mlp_swiglu_forward(x, w_gate_up, w_down, y=out, workspace=workspace, stream=stream), False


def shard_sum(partials, out=None, stream=None):
    """out [T, H] bf16 = sum over the leading axis of partials [n, T, H] (fp32 accumulation)."""
    torch = _torch()
    n, T, H = partials.shape
    code = _dtype_code(partials.dtype)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=partials.device)
    st = lib().shard_sum(_ptr(partials), code, n, T, H, _ptr(out), out.numel(), _stream(stream))
    _check("shard_sum", st)
    return out


def merged_proj_forward(x, w, q_dim, kv_dim, tp, logical=True, rank_major=True, out_logical=None,
                        out_rank_major=None, workspace=None, stream=None):
    """(logical [T, C], rank_major [T, C]) of x w^T; either may be skipped (None returned)."""
    torch = _torch()
    T, H = x.shape
    C = q_dim + kv_dim
    if logical and out_logical is None:
        out_logical = torch.empty((T, C), dtype=torch.bfloat16, device=x.device)
    if rank_major and out_rank_major is None:
        out_rank_major = torch.empty((T, C), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = new_merged_workspace(T, H, q_dim, kv_dim, x.device)
    st = lib().merged_proj_forward(_ptr(x), T, H, _ptr(w), q_dim, kv_dim, tp, _ptr(out_logical),
                                   _ptr(out_rank_major), T * C, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream))
    _check("merged_proj_forward", st)
    return out_logical, out_rank_major


def merged_proj_reorder(rank_major, q_dim, kv_dim, tp, out=None, stream=None):
    torch = _torch()
    T, C = rank_major.shape
    if out is None:
        out = torch.empty_like(rank_major)
    st = lib().merged_proj_reorder(_ptr(rank_major), _ptr(out), T, q_dim, kv_dim, tp, T * C, _stream(stream))
    _check("merged_proj_reorder", st)
    return out


def poll_device_error(stream=None) -> int:
    return int(lib().mse_poll_device_error(_stream(stream)))


def set_wait_limit_ns(ns: int) -> None:
    lib().mse_set_wait_limit_ns(int(ns))


def get_wait_limit_ns() -> int:
    return int(lib().mse_get_wait_limit_ns())


def set_kernel_path(path: int) -> int:
    return int(lib().mse_set_kernel_path(int(path)))


def set_tuning(key: int, value: int) -> int:
    return int(lib().mse_set_tuning(int(key), int(value)))


def mlp_launch_plan(T: int, H: int, I: int, tp: int = 1, rank_count: int = 1, x_early: bool = False,
                    sm_count: int = 152) -> dict:
    """CTA counts of the decode-size kernels of an MLP call (host-side, no GPU): see
    mse_mlp_launch_plan in include/mse.h."""
    out = (ctypes.c_int32 * 8)()
    _check("mse_mlp_launch_plan", lib().mse_mlp_launch_plan(int(T), int(H), int(I), int(tp), int(rank_count),
                                                             int(bool(x_early)), int(sm_count), out))
    keys = ("swapab", "gate_up_ctas", "down_ctas", "gate_up_parts", "down_parts", "bn", "kbs", "stages")
    return {k: int(v) for k, v in zip(keys, out)}


def merged_launch_plan(T: int, H: int, q_dim: int, kv_dim: int, tp: int, sm_count: int = 152) -> dict:
    """CTA count and split of the merged projection's kernel (host-side, no GPU): see
    mse_merged_launch_plan in include/mse.h."""
    out = (ctypes.c_int32 * 8)()
    _check("mse_merged_launch_plan", lib().mse_merged_launch_plan(int(T), int(H), int(q_dim), int(kv_dim), int(tp),
                                                                   int(sm_count), out))
    keys = ("swapab", "ctas", "parts", "joint_finish", "bn", "kbs", "stages")
    return {k: int(v) for k, v in zip(keys, out)}


def set_prefill_kernel(kind: int) -> int:
    return int(lib().mse_set_prefill_kernel(int(kind)))


def selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check("mse_selftest_wait_timeout", lib().mse_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def set_phase_events(ev_begin=None, ev_mid=None, ev_end=None) -> None:
    h = lambda e: None if e is None else e.cuda_event
    lib().mse_set_phase_events(h(ev_begin), h(ev_mid), h(ev_end))
