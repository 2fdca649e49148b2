"""MSE_TUNE_X_EARLY: mlp_swiglu_forward reads x without waiting for the previous kernel on
the stream when x overlaps neither the y nor the workspace of the previous call on that
stream.  Independent calls streamed back to back, and layers chained through device memory
(x of a call is the previous call's y: the library sees the overlap and waits), must give
exactly what the default path gives."""
import math

import pytest

import workloads as W
from tests.helpers import to_dev

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
    assert mse.poll_device_error() == 0


def with_x_early(v, fn):
    old = mse.set_tuning(mse.TUNE_X_EARLY, v)
    try:
        return fn()
    finally:
        mse.set_tuning(mse.TUNE_X_EARLY, old)


@pytest.mark.parametrize("T", [64, 16])
def test_x_early_independent_and_chained_calls(T):
    w = W.DECODE_T64
    wgu, wd = W.make_mlp_weights(w)
    g0, d0 = to_dev(wgu), to_dev(wd)
    gus = [g0, torch.roll(g0, 977, 0).contiguous()]
    wds = [d0, torch.roll(d0, 331, 0).contiguous()]
    xs = [to_dev(W.make_custom(1900 + k, 0, (T, w.H))) for k in range(4)]
    ws = mse.new_mlp_workspace(T, w.H, w.I)

    def independent():
        ys = [torch.empty((T, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(12)]
        for i, y in enumerate(ys):
            mse.mlp_swiglu_forward(xs[i % 4], gus[i % 2], wds[i % 2], y=y, workspace=ws)
        torch.cuda.synchronize()
        return ys

    def chained():
        outs = [xs[0]]
        for i in range(6):
            outs.append(mse.mlp_swiglu_forward(outs[-1], gus[i % 2], wds[i % 2], workspace=ws))
        torch.cuda.synchronize()
        return outs[1:]

    ref_i, ref_c = with_x_early(0, independent), with_x_early(0, chained)
    got_i, got_c = with_x_early(1, independent), with_x_early(1, chained)
    for i, (a, b) in enumerate(zip(got_i, ref_i)):
        assert torch.equal(a, b), f"independent call {i}"
    for i, (a, b) in enumerate(zip(got_c, ref_c)):
        assert torch.equal(a, b), f"chained layer {i}"
    assert mse.poll_device_error() == 0
