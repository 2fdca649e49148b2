"""Shared helpers for the GPU tests: numpy bf16 bits <-> torch tensors, the
tolerance of the parity criterion, and path switching."""
import contextlib

import numpy as np

# |gpu - ref| <= ATOL + RTOL * |ref| per element
ATOL = 0.02
RTOL = 0.02


def to_dev(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def to_bits(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_f64(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def err_ratio(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max over elements of |gpu - ref| / (ATOL + RTOL |ref|); <= 1 passes."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu))
    return float(np.max(np.abs(gpu - ref) / (ATOL + RTOL * np.abs(ref)))) if gpu.size else 0.0


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = "") -> float:
    r = err_ratio(gpu, ref)
    assert r <= 1.0, f"{what}: max |gpu-ref|/(0.02+0.02|ref|) = {r:.3f}"
    return r


@contextlib.contextmanager
def kernel_path(path: int):
    import moe_shared_expert_gb300 as mse
    old = mse.set_kernel_path(path)
    try:
        yield
    finally:
        mse.set_kernel_path(old)


@contextlib.contextmanager
def prefill_kernel(kind: int):
    import moe_shared_expert_gb300 as mse
    old = mse.set_prefill_kernel(kind)
    try:
        yield
    finally:
        mse.set_prefill_kernel(old)
