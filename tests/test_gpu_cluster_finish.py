"""Two-part split-K tiles finished inside clusters of three CTAs (the option
MSE_TUNE_CLUSTER_FINISH, launched when three CTAs cover two tiles exactly): one
tile's finishing CTA fetches the other part without publishing its own, the other
tile's first part is written straight into the second CTA's shared memory.
Checked against the fp64 oracle and bit for bit against the same launch shape
finishing every tile through L2 (the parts are summed in the same order).

The grid is forced to the size that gives the three-CTAs-per-two-tiles pattern on each
shape: gate_up tiles of 64 intermediate columns, H / 64 k-blocks per tile.
"""
import contextlib
import math

import numpy as np
import pytest

import oracle
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
    assert mse.poll_device_error() == 0


@contextlib.contextmanager
def tuning(**kv):
    keys = {"grid": mse.TUNE_GRID, "cluster": mse.TUNE_CLUSTER_FINISH}
    old = {}
    try:
        for k, v in kv.items():
            old[k] = mse.set_tuning(keys[k], v)
            assert old[k] >= 0
        yield
    finally:
        for k, v in old.items():
            mse.set_tuning(keys[k], v)


def case(T, H, I, seed):
    x = W.make_custom(seed, 0, (T, H))
    wgu = W.make_custom(seed, 1, (2 * I, H), 1 / math.sqrt(H))
    wd = W.make_custom(seed, 2, (H, I), 1 / math.sqrt(I))
    return x, wgu, wd


def forward(x, wgu, wd):
    T, H = x.shape
    I = wd.shape[1]
    ws = mse.new_mlp_workspace(T, H, I)
    y = mse.mlp_swiglu_forward(to_dev(x), to_dev(wgu), to_dev(wd), workspace=ws)
    torch.cuda.synchronize()
    h = ws[: T * I * 2].view(torch.int16).view(T, I).cpu().numpy().view(np.uint16)
    return to_bits(y), h


def trio_grid(H, I):
    """CTAs for which three cover two gate_up tiles: 3 * units = 2 * (H/64) * grid."""
    units = (I // 64) * (H // 64)
    g = 3 * units // (2 * (H // 64))
    assert g % 3 == 0 and 3 * units == 2 * (H // 64) * g
    return g


@pytest.mark.parametrize("T,H,I", [(64, 1024, 768), (7, 768, 384), (128, 1024, 1152), (33, 2048, 768),
                                   (256, 768, 384)])
def test_cluster_finish_matches_oracle_and_l2_finish(T, H, I):
    x, wgu, wd = case(T, H, I, 9500 + T + H + I)
    g = trio_grid(H, I)
    y_ref, _, h_ref = oracle.mlp_forward(x, wgu, wd)
    with tuning(grid=g, cluster=1):
        y1, h1 = forward(x, wgu, wd)
        y1b, h1b = forward(x, wgu, wd)
    with tuning(grid=g, cluster=0):
        y0, h0 = forward(x, wgu, wd)
    assert_close(bits_f64(h1), bits_f64(h_ref), f"h T={T}")
    assert_close(bits_f64(y1), bits_f64(y_ref), f"y T={T}")
    assert np.array_equal(h1, h0), "cluster finish differs from the L2 finish"
    assert np.array_equal(y1, y0)
    assert np.array_equal(h1, h1b) and np.array_equal(y1, y1b), "not deterministic"


def test_cluster_finish_decode_t64_default_shape():
    # the decode workload: 144 CTAs cover the 96 gate_up tiles three per two
    w = W.DECODE_T64
    wgu, wd = W.make_mlp_weights(w)
    x = W.make_x(w)
    rows = [0, 21, 42, 63]
    y_ref, _, _ = oracle.mlp_forward(x[rows], wgu, wd)
    with tuning(cluster=1):
        y1, h1 = forward(x, wgu, wd)
    with tuning(cluster=0):
        y0, h0 = forward(x, wgu, wd)
    assert_close(bits_f64(y1[rows]), bits_f64(y_ref), "decode T=64")
    assert np.array_equal(h1, h0)
    assert np.array_equal(y1, y0)
