"""Host-side pieces of bench.py that need no GPU: the byte and FLOP models the
roofline divides by (pinned to the sizes the pages print), the collective model
and crossover search of the replicated-vs-sharded sweep, and the --tune parser."""
import math
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

H, I = 7168, 6144


def test_byte_models_match_the_pages_sizes():
    # gate_up 176.2 MB and down 88.1 MB per layer (Kimi-K3 PR, section "Problem")
    assert bench.gate_up_bytes(0, H, I) == 176_160_768
    assert bench.mlp_bytes(0, H, I) == 176_160_768 + 88_080_384
    # decode T = 64: weights + x read + y written
    assert bench.mlp_bytes(64, H, I) == 266_076_160
    # one TP8 rank's slice: 1/8 of the weights
    assert bench.mlp_bytes(0, H, I // 8) * 8 == bench.mlp_bytes(0, H, I)


def test_flop_model():
    # 2 flops per multiply-add over the three weight matrices, per token
    assert bench.mlp_flops(8192, H, I) == 2 * 8192 * 3 * H * I
    assert bench.gate_up_flops(8192, H, I) == 2 * 8192 * 2 * H * I


def test_collectives_model():
    # two collectives, each alpha + (tp-1)/tp of the [T x H] bf16 tensor over beta
    t = bench.collectives_model_s(64, H, 8, 10e-6, 800e9)
    assert t == pytest.approx(2 * (10e-6 + 7 / 8 * 64 * H * 2 / 800e9))
    assert bench.collectives_model_s(64, H, 1, 10e-6, 800e9) == pytest.approx(20e-6)   # nothing moves
    assert bench.collectives_model_s(128, H, 8, 0.0, 800e9) == pytest.approx(
        2 * bench.collectives_model_s(64, H, 8, 0.0, 800e9))


def test_crossovers_pick_the_first_losing_group_size():
    pts = []
    for T, rep, sh, coll in [(16, 50, 20, 40), (64, 50, 25, 55), (256, 50, 60, 80), (1024, 60, 55, 90)]:
        pts.append({"tp": 8, "T": T, "replicated_us": rep, "sharded_kernel_us": sh,
                    "sharded_with_collectives_us": coll})
    pts.append({"tp": 4, "T": 16, "replicated_us": 50, "sharded_kernel_us": 10, "sharded_with_collectives_us": 20})
    c = bench.crossovers(list(reversed(pts)), [8, 4])
    assert c["8"] == {"kernel_only_first_T_replicated_wins": 256,
                      "with_modelled_collectives_first_T_replicated_wins": 64}
    assert c["4"] == {"kernel_only_first_T_replicated_wins": None,
                      "with_modelled_collectives_first_T_replicated_wins": None}


def test_apply_tuning_parses_sets_and_rejects():
    mse = pytest.importorskip("moe_shared_expert_gb300")
    from moe_shared_expert_gb300 import _build
    _build.build()
    mse.lib()
    old = mse.set_tuning(mse.TUNE_GRID, 0)
    try:
        assert bench.apply_tuning("") == {}
        assert bench.apply_tuning("grid=96, one_launch=0") == {"grid": 96, "one_launch": 0}
        assert mse.set_tuning(mse.TUNE_GRID, 0) == 96          # it was set
        with pytest.raises(ValueError):
            bench.apply_tuning("grid=100000")                  # out of range
        with pytest.raises(AttributeError):
            bench.apply_tuning("no_such_key=1")
    finally:
        mse.set_tuning(mse.TUNE_GRID, old)
        mse.set_tuning(mse.TUNE_ONE_LAUNCH, 0)


def test_percentiles_nearest_rank():
    assert bench.percentiles([5, 1, 3, 2, 4]) == [1, 3, 5]
    assert bench.percentiles([7.0]) == [7.0, 7.0, 7.0]
    assert bench.percentiles(list(range(21))) == [2, 10, 18]


def test_crossover_sensitivity_moves_with_the_collective_model():
    # replicated 50 us at every T; sharded kernels 20 us.  A cheaper collective model can
    # only move the crossover to a larger T (or away), a dearer one to a smaller T.
    pts = [{"tp": 8, "T": T, "replicated_us": 50.0, "sharded_kernel_us": 20.0} for T in (16, 64, 256, 1024, 4096)]
    c = bench.crossover_sensitivity(pts, [8], H, alphas_us=(0.0, 10.0, 20.0), betas_gbs=(400.0, 1600.0))["8"]
    # alpha 20 us: 2 x 20 us + 20 us of kernel = 60 us > 50 at any T
    assert c["a20us_b400GBps"] == 16 and c["a20us_b1600GBps"] == 16
    # alpha 0, beta 1600 GB/s: 20 us + 2 * 7/8 * T * H * 2 / 1.6e12 >= 50 us from T = 4096 on
    assert c["a0us_b1600GBps"] == 4096
    order = [c[f"a{a:g}us_b{b:g}GBps"] or 10 ** 9 for a in (0.0, 10.0, 20.0) for b in (1600.0,)]
    assert order == sorted(order, reverse=True)
    # the model is the one the sweep uses
    T = 1024
    assert (20e-6 + bench.collectives_model_s(T, H, 8, 10e-6, 400e9) >= 50e-6) == (c["a10us_b400GBps"] <= T)


def test_decode_config_is_shared_by_both_arms():
    import workloads as W
    a = bench.decode_config(W.DECODE_T64, 4, 1)
    assert a["workload"] == "decode_t64" and a["T"] == 64 and "1057 MB" in a["l2"]
    assert a == bench.decode_config(W.DECODE_T64, 4, 1)


def test_tensor_peak_at_clock():
    # 152 SMs x 8192 dense bf16 FLOP per clock at 2070 MHz
    assert bench.tensor_peak_at_clock(2070) == pytest.approx(152 * 8192 * 2.07e9 / 1e12)
    assert bench.tensor_peak_at_clock(None) is None
