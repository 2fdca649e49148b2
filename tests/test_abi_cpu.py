"""C-ABI checks that need no GPU: the library loads, exports every symbol its
header declares, and rejects invalid arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

import moe_shared_expert_gb300 as mse
from moe_shared_expert_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mse.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return mse.lib()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"^MSE_API\s+[\w\s\*]*?\**\s*(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    for n in ["mlp_swiglu_forward", "mlp_swiglu_shard_partial", "mlp_swiglu_shard_forward",
              "mse_shard_sequence_parallel_mlp", "shard_sum", "merged_proj_forward",
              "merged_proj_reorder", "mlp_swiglu_workspace_bytes", "merged_proj_workspace_bytes",
              "mse_poll_device_error", "mse_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings(L):
    for code, name in mse.STATUS.items():
        assert L.mse_status_string(code).decode() == name
    assert L.mse_version().decode().startswith("mse")


def test_workspace_sizes(L):
    T, H, I = 64, 7168, 6144
    n = L.mlp_swiglu_workspace_bytes(T, H, I)
    assert n >= T * I * 2 and n % 256 == 0
    assert L.mlp_swiglu_workspace_bytes(0, H, I) == 0
    assert L.mlp_swiglu_workspace_bytes(8192, H, I) >= 8192 * I * 2
    assert L.merged_proj_workspace_bytes(128, 7168, 1536, 576) > 0
    assert L.merged_proj_workspace_bytes(128, 7168, -1, 576) == 0


def test_workspace_size_covers_every_smaller_token_count(L):
    # the size query is non-decreasing in T: a buffer sized for T serves every call with
    # fewer tokens (the split-K tiles of T <= 256 outweigh h of a few hundred more tokens)
    for H, I in [(7168, 6144), (384, 320), (2048, 1536)]:
        sizes = [L.mlp_swiglu_workspace_bytes(T, H, I) for T in list(range(1, 400)) + [1024, 8192]]
        assert all(a <= b for a, b in zip(sizes, sizes[1:])), (H, I)
        assert all(n % 256 == 0 for n in sizes)
    m = [L.merged_proj_workspace_bytes(T, 7168, 1536, 576) for T in range(1, 400)]
    assert all(a <= b for a, b in zip(m, m[1:]))


def test_sync_range_sits_at_the_end_of_the_buffer(L):
    # the sync words are the workspace's last, 256-aligned bytes whatever T is, and their
    # size depends on H and I only: a buffer sized for T serves every smaller call
    for H, I in [(7168, 6144), (384, 320), (2048, 1536)]:
        n = L.mlp_swiglu_workspace_bytes(256, H, I)
        ranges = set()
        for T in (1, 16, 64, 65, 200, 256):
            off, b = mse.mlp_swiglu_workspace_sync_range(T, H, I, n)
            assert off % 256 == 0 and b > 0 and off + b <= n and n - (off + b) < 256
            # room for the counters of every gate_up tile, every down tile and every h flag
            assert b >= 4 * ((I // 64) + (I // 64) * (H // 128) + (I // 64) + 3)
            ranges.add((off, b))
        assert len(ranges) == 1, (H, I, ranges)
    # a buffer below the call's minimal need is rejected
    n = L.mlp_swiglu_workspace_bytes(64, 7168, 6144)
    with pytest.raises(mse.MSEError):
        mse.mlp_swiglu_workspace_sync_range(64, 7168, 6144, n - 256)
    n = L.merged_proj_workspace_bytes(128, 7168, 1536, 576)
    off, b = mse.merged_proj_workspace_sync_range(128, 7168, 1536, 576, n)
    assert off + b == n and b >= 4 * 17


# Fake, never-dereferenced addresses: every call below fails validation before any
# CUDA call.  As a second guard they are not run where a CUDA device is visible.
FAKE = 0x10000


def _gpu_visible():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


no_gpu_only = pytest.mark.skipif(_gpu_visible(), reason="fake-pointer validation checks run only without a GPU")
GOOD_WS = 1 << 30


def code(name):
    return mse.STATUS_CODE[name]


@no_gpu_only
def test_forward_validation(L):
    f = L.mlp_swiglu_forward
    assert f(None, 64, 7168, 6144, FAKE, FAKE, FAKE, 64 * 7168, FAKE, GOOD_WS, None) == code("MSE_ERR_INVALID_ARG")
    assert f(FAKE, 0, 7168, 6144, FAKE, FAKE, FAKE, 64 * 7168, FAKE, GOOD_WS, None) == code("MSE_ERR_INVALID_ARG")
    # truncated output geometry
    assert f(FAKE, 64, 7168, 6144, FAKE, FAKE, FAKE, 64 * 7168 - 1, FAKE, GOOD_WS, None) == code("MSE_ERR_GEOMETRY")
    # workspace missing / too small / misaligned
    assert f(FAKE, 64, 7168, 6144, FAKE, FAKE, FAKE, 64 * 7168, None, GOOD_WS, None) == code("MSE_ERR_WORKSPACE")
    assert f(FAKE, 64, 7168, 6144, FAKE, FAKE, FAKE, 64 * 7168, FAKE, 1024, None) == code("MSE_ERR_WORKSPACE")
    assert f(FAKE, 64, 7168, 6144, FAKE, FAKE, FAKE, 64 * 7168, FAKE + 8, GOOD_WS, None) == code("MSE_ERR_WORKSPACE")


@no_gpu_only
def test_forward_host_validation(L):
    f = L.mlp_swiglu_forward_host
    n = L.mlp_swiglu_host_workspace_bytes(64, 7168, 6144)
    # + the copy counts (256 bytes) and the two device copies of x
    assert n == L.mlp_swiglu_workspace_bytes(64, 7168, 6144) + 256 + 2 * 64 * 7168 * 2
    assert f(None, 64, 7168, 6144, FAKE, FAKE, FAKE, 64 * 7168, FAKE, n, None) == code("MSE_ERR_INVALID_ARG")
    assert f(FAKE, 64, 7168, 6144, FAKE, FAKE, FAKE, 64 * 7168 - 1, FAKE, n, None) == code("MSE_ERR_GEOMETRY")
    assert f(FAKE, 64, 7168, 6144, FAKE, FAKE, FAKE * 16, 64 * 7168, FAKE, n - 256, None) == code("MSE_ERR_WORKSPACE")
    # x and y overlap (checked before any CUDA call)
    assert f(FAKE, 64, 7168, 6144, FAKE, FAKE, FAKE + 64, 64 * 7168, FAKE, n, None) == code("MSE_ERR_INVALID_ARG")


@no_gpu_only
def test_shard_partial_validation(L):
    f = L.mlp_swiglu_shard_partial
    args = lambda tp, rf, rc, cap, dt=0: (FAKE, 128, 7168, 6144, FAKE, FAKE, tp, rf, rc, FAKE, dt, cap, FAKE,
                                          GOOD_WS, None)
    full = 8 * 128 * 7168
    # 6144 % 5 != 0: the sharding gate's divisibility rule
    assert f(*args(5, 0, 5, full)) == code("MSE_ERR_NOT_DIVISIBLE")
    # H % tp != 0 (7168 % 3 != 0 although 6144 % 3 == 0)
    assert f(*args(3, 0, 3, full)) == code("MSE_ERR_NOT_DIVISIBLE")
    assert f(*args(8, 6, 3, full)) == code("MSE_ERR_GEOMETRY")       # ranks beyond tp
    assert f(*args(8, -1, 2, full)) == code("MSE_ERR_GEOMETRY")
    assert f(*args(8, 0, 0, full)) == code("MSE_ERR_GEOMETRY")
    assert f(*args(8, 0, 8, full - 1)) == code("MSE_ERR_GEOMETRY")   # truncated partial buffer
    assert f(*args(8, 0, 8, full, 7)) == code("MSE_ERR_INVALID_ARG")  # bad dtype
    assert f(*args(0, 0, 1, full)) == code("MSE_ERR_INVALID_ARG")


@no_gpu_only
def test_shard_forward_validation(L):
    f = L.mlp_swiglu_shard_forward
    args = lambda tp, rf, rc, cap, dt=0: (FAKE, 128, 7168, 6144, FAKE, FAKE, tp, rf, rc, FAKE, dt, cap, FAKE,
                                          GOOD_WS, None)
    one = 128 * 7168
    assert f(*args(5, 0, 5, one)) == code("MSE_ERR_NOT_DIVISIBLE")     # 6144 % 5 != 0
    assert f(*args(3, 0, 3, one)) == code("MSE_ERR_NOT_DIVISIBLE")     # 7168 % 3 != 0
    assert f(*args(8, 6, 3, one)) == code("MSE_ERR_GEOMETRY")
    assert f(*args(8, -1, 2, one)) == code("MSE_ERR_GEOMETRY")
    assert f(*args(8, 0, 0, one)) == code("MSE_ERR_GEOMETRY")
    assert f(*args(8, 0, 8, one - 1)) == code("MSE_ERR_GEOMETRY")      # one [T x H] output, truncated
    assert f(*args(8, 0, 8, one, 7)) == code("MSE_ERR_INVALID_ARG")
    assert f(*args(0, 0, 1, one)) == code("MSE_ERR_INVALID_ARG")
    a = list(args(8, 0, 8, one))
    a[12] = FAKE + 8                                                  # misaligned workspace
    assert f(*a) == code("MSE_ERR_WORKSPACE")


@no_gpu_only
def test_shard_sum_validation(L):
    f = L.shard_sum
    assert f(FAKE, 0, 8, 127, 7168, FAKE, 127 * 7168, None) == code("MSE_ERR_NOT_DIVISIBLE")
    assert f(FAKE, 0, 8, 128, 7168, FAKE, 128 * 7168 - 1, None) == code("MSE_ERR_GEOMETRY")
    assert f(None, 0, 8, 128, 7168, FAKE, 128 * 7168, None) == code("MSE_ERR_INVALID_ARG")
    assert f(FAKE, 3, 8, 128, 7168, FAKE, 128 * 7168, None) == code("MSE_ERR_INVALID_ARG")


@no_gpu_only
def test_merged_validation(L):
    f = L.merged_proj_forward
    C = 1536 + 576
    ok_ws = L.merged_proj_workspace_bytes(128, 7168, 1536, 576)
    # every merged output size must be divisible by tp
    assert f(FAKE, 128, 7168, FAKE, 1536, 576, 5, FAKE, FAKE, 128 * C, FAKE, ok_ws, None) == code("MSE_ERR_NOT_DIVISIBLE")
    assert f(FAKE, 128, 7168, FAKE, 1536, 576, 128, FAKE, FAKE, 128 * C, FAKE, ok_ws, None) == code("MSE_ERR_NOT_DIVISIBLE")
    assert f(FAKE, 128, 7168, FAKE, 1536, 576, 16, FAKE, FAKE, 128 * C - 1, FAKE, ok_ws, None) == code("MSE_ERR_GEOMETRY")
    assert f(FAKE, 128, 7168, FAKE, 1536, 576, 16, None, None, 128 * C, FAKE, ok_ws, None) == code("MSE_ERR_INVALID_ARG")
    r = L.merged_proj_reorder
    assert r(FAKE, FAKE + 1 << 20, 128, 1536, 576, 7, 128 * C, None) == code("MSE_ERR_NOT_DIVISIBLE")
    assert r(FAKE, FAKE + (1 << 24), 128, 1536, 576, 16, 128 * C - 1, None) == code("MSE_ERR_GEOMETRY")
    assert r(FAKE, FAKE + 100, 128, 1536, 576, 16, 128 * C, None) == code("MSE_ERR_INVALID_ARG")  # overlap


def test_settings_roundtrip(L):
    old = L.mse_get_wait_limit_ns()
    L.mse_set_wait_limit_ns(12345)
    assert L.mse_get_wait_limit_ns() == 12345
    L.mse_set_wait_limit_ns(old)
    prev = L.mse_set_kernel_path(mse.PATH_GENERIC)
    assert L.mse_set_kernel_path(prev) == mse.PATH_GENERIC
    assert L.mse_set_kernel_path(99) == prev        # invalid value: unchanged


def test_product_path_does_not_import_oracle():
    import sys
    for mod in ["moe_shared_expert_gb300", "moe_shared_expert_gb300._build"]:
        src = open(sys.modules[mod].__file__).read()
        assert "oracle" not in src.replace("# oracle", "")
    for f in os.listdir(os.path.join(ROOT, "moe_shared_expert_gb300", "csrc")):
        assert "oracle" not in open(os.path.join(ROOT, "moe_shared_expert_gb300", "csrc", f)).read().lower()


# key: (default, accepted values, rejected values)
TUNING = {
    mse.TUNE_ISSUE_GROUP: (0, [0, 1, 4], [-1, 5]),
    mse.TUNE_STAGES: (0, [2, 12], [1, 13]),
    mse.TUNE_CACHE_HINTS: (1, [0, 1], [2, -1]),
    mse.TUNE_GRID: (0, [1, 160], [161, -1]),
    mse.TUNE_SPIN_WAIT: (0, [0, 1], [2]),
    mse.TUNE_ONE_LAUNCH: (0, [1, 2], [3]),
    mse.TUNE_PDL: (1, [0, 1], [2]),
    mse.TUNE_COOP_FINISH: (6, [0, 128], [129, -1]),
    mse.TUNE_PAIR_MIN_T: (0, [1, 256], [-1]),
    mse.TUNE_GRID_DOWN: (0, [1, 160], [161]),
    mse.TUNE_CLUSTER_FINISH: (0, [0, 1], [2]),
    mse.TUNE_L2_PREFETCH: (8, [0, 256], [-1, 257]),
    mse.TUNE_SWAPAB_MAX_T: (160, [0, 256], [-1, 257]),
    mse.TUNE_X_EARLY: (0, [0, 1], [2, -1]),
    mse.TUNE_DOWN_FLAGS: (0, [0, 1], [2, -1]),
    mse.TUNE_HOST_X_COPIERS: (16, [0, 1, 1024], [-1, 1025]),
    mse.TUNE_PAIR_SPLIT: (1, [0, 1], [2, -1]),
}


def test_tuning_keys_defaults_ranges_and_restore(L):
    for key, (default, good, bad) in TUNING.items():
        cur = L.mse_set_tuning(key, default)   # read the current value (and set the default)
        assert L.mse_set_tuning(key, cur) == default, f"key {key}: default"
        for v in good:
            prev = L.mse_set_tuning(key, v)
            assert prev >= 0
            assert L.mse_set_tuning(key, prev) == v, f"key {key} value {v}"
        for v in bad:
            assert L.mse_set_tuning(key, v) == -1, f"key {key} accepted {v}"
        assert L.mse_set_tuning(key, cur) == cur   # unchanged by the rejected values
    assert L.mse_set_tuning(5, 1) == -1         # unused key
    assert L.mse_set_tuning(99, 1) == -1
