"""The joint split-K finish of the merged projection (tiles whose reduction is split
between several CTAs are summed and written slice by slice by the CTAs for which the
tile is the final segment) against the fp64 oracle, with the finish forced on for
every split tile, at its default threshold and off.

The exact permutation check runs through the joint finish too: with integer-valued
inputs and one-hot weight rows every sum is exact whatever its order, so both
layouts must equal the oracle bit for bit.
"""
import contextlib

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
def coop(threshold: int):
    old = mse.set_tuning(mse.TUNE_COOP_FINISH, threshold)
    assert old >= 0
    try:
        yield
    finally:
        mse.set_tuning(mse.TUNE_COOP_FINISH, old)


def run(x, wm, q, kv, tp):
    lo, rm = mse.merged_proj_forward(to_dev(x), to_dev(wm), q, kv, tp)
    torch.cuda.synchronize()
    return to_bits(lo), to_bits(rm)


@pytest.mark.parametrize("threshold", [2, 6, 0])
def test_mla_workload_joint_finish(threshold):
    w = W.MLA_MERGED
    x = W.make_x(w)
    wm = W.make_merged_weight(w)
    with coop(threshold):
        lo, rm = run(x, wm, w.q_dim, w.kv_dim, w.tp)
        lo2, rm2 = run(x, wm, w.q_dim, w.kv_dim, w.tp)
    ref_lo, ref_rm, _ = oracle.merged_proj(x, wm, w.q_dim, w.kv_dim, w.tp)
    assert_close(bits_f64(lo), bits_f64(ref_lo), f"logical (threshold {threshold})")
    assert_close(bits_f64(rm), bits_f64(ref_rm), f"rank-major (threshold {threshold})")
    assert np.array_equal(lo, lo2) and np.array_equal(rm, rm2), "not deterministic"
    perm = oracle.rank_major_to_logical(w.q_dim, w.kv_dim, w.tp)
    assert np.array_equal(rm, lo[:, perm])


@pytest.mark.parametrize("T", [1, 16, 40, 130, 256])
def test_merged_joint_finish_shapes(T):
    # H = 4096 gives 64 k-blocks per tile: split between many CTAs, ragged token counts
    q, kv, tp, H = 512, 192, 8, 4096
    x = W.make_custom(300 + T, 0, (T, H))
    wm = W.make_custom(300 + T, 4, (q + kv, H), 1 / 64)
    ref_lo, ref_rm, _ = oracle.merged_proj(x, wm, q, kv, tp)
    with coop(2):
        lo, rm = run(x, wm, q, kv, tp)
    assert_close(bits_f64(lo), bits_f64(ref_lo), f"logical T={T}")
    assert_close(bits_f64(rm), bits_f64(ref_rm), f"rank-major T={T}")


def test_joint_finish_exact_on_integer_inputs():
    q, kv, tp, H, T = 1536, 576, 16, 7168, 128
    C = q + kv
    xi = ((np.arange(T * H).reshape(T, H) * 7) % 201) - 100
    x = W.f32_to_bf16_bits(xi.astype(np.float32))
    wm = np.zeros((C, H), dtype=np.uint16)
    wm[np.arange(C), (np.arange(C) * 5 + 11) % H] = 0x3F80      # 1.0
    ref_lo, ref_rm, _ = oracle.merged_proj(x, wm, q, kv, tp)
    with coop(2):
        lo, rm = run(x, wm, q, kv, tp)
    assert np.array_equal(lo, ref_lo)
    assert np.array_equal(rm, ref_rm)
