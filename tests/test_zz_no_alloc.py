"""mlp_swiglu_forward_static_scratch: the entry point for callers that cannot
allocate device memory (its scratch is a fixed array inside the library).

It is called through the C ABI with only inputs and outputs and must agree with
the workspace-taking mlp_swiglu_forward within the parity tolerance, on two
calls in a row (the second call runs on the array as the first call left it).
"""
import math

import numpy as np
import pytest

import workloads as W
from tests.helpers import assert_close, bits_f64, to_bits, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

mse = pytest.importorskip("moe_shared_expert_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_shared_expert_gb300 import _build
    _build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mse.lib()
    yield


def call_static(x, wgu, wd, y):
    T, H = x.shape
    I = wd.shape[1]
    return mse.lib().mlp_swiglu_forward_static_scratch(
        x.data_ptr(), T, H, I, wgu.data_ptr(), wd.data_ptr(), y.data_ptr(), y.numel(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("case", ["decode_t64", "small_t24", "ragged_t7"])
def test_static_scratch_matches_workspace_entry_point(case):
    if case == "decode_t64":
        w = W.DECODE_T64
        x = W.make_x(w)
        wgu, wd = W.make_mlp_weights(w)
    else:
        T, H, I = (24, 512, 256) if case == "small_t24" else (7, 384, 320)
        x = W.make_custom(61 + T, 0, (T, H))
        wgu = W.make_custom(61 + T, 1, (2 * I, H), 1 / math.sqrt(H))
        wd = W.make_custom(61 + T, 2, (H, I), 1 / math.sqrt(I))
    dx, dgu, dwd = to_dev(x), to_dev(wgu), to_dev(wd)
    ref = mse.mlp_swiglu_forward(dx, dgu, dwd)
    ys = [torch.full_like(ref, float("nan")) for _ in range(2)]
    torch.cuda.synchronize()
    free_before = None
    outs = []
    for i in range(2):                      # two calls in a row on the shared array
        assert call_static(dx, dgu, dwd, ys[i]) == 0
        torch.cuda.synchronize()
        if i == 0:                          # after the first call's one-time set-up
            free_before = torch.cuda.mem_get_info()[0]
        outs.append(to_bits(ys[i]))
    # the second call took no device memory (nothing allocated, nothing cached)
    assert torch.cuda.mem_get_info()[0] == free_before
    assert mse.poll_device_error() == 0
    r = to_bits(ref)
    for o in outs:
        assert_close(bits_f64(o), bits_f64(r), f"{case}: static-scratch vs workspace entry point")


def test_static_scratch_rejects_sizes_beyond_its_maximum():
    T, H, I = 4096, 7168, 6144                # needs far more than the fixed array
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    wgu = torch.zeros((2 * I, H), dtype=torch.bfloat16, device="cuda")
    wd = torch.zeros((H, I), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    assert mse.STATUS[call_static(x, wgu, wd, y)] == "MSE_ERR_WORKSPACE"
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(y).item()) == 0   # nothing was launched
