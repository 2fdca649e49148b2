"""The decode-size layer as one launch (gate_up + SiluAndMul passes, then the down
projection, in one kernel) against the fp64 oracle, against the two-launch path,
and across repeated calls, CUDA-graph replays and shard subsets.  Mode 1 runs one
gate_up pass; mode 2 (the default) two half passes with the down pass taking the
first half's k-blocks first.

The down pass reads h tiles that other CTAs of the same launch write; per-tile
flags order the two.  These tests check the results of that hand-off and that
every completed call leaves the workspace's sync words zero for the next one.
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
def one_launch(mode: int):
    old = mse.set_tuning(mse.TUNE_ONE_LAUNCH, int(mode))
    assert old in (0, 1, 2)
    try:
        yield
    finally:
        mse.set_tuning(mse.TUNE_ONE_LAUNCH, old)


def case(T, H, I, seed):
    x = W.make_custom(seed, 0, (T, H))
    wgu = W.make_custom(seed, 1, (2 * I, H), 1 / math.sqrt(H))
    wd = W.make_custom(seed, 2, (H, I), 1 / math.sqrt(I))
    return x, wgu, wd


def sync_region_offset(T, H, I):
    """Start of the counters/flags region of an mlp workspace (after h and the three
    split-K slot regions of 160 CTAs x 2 slots x 128 x bn fp32)."""
    a = lambda v: (v + 255) // 256 * 256
    bn = (T + 15) // 16 * 16
    return a(T * I * 2) + 3 * a(160 * 2 * 128 * bn * 4)


def forward(x, wgu, wd, ws=None):
    T, H = x.shape
    I = wd.shape[1]
    ws = mse.new_mlp_workspace(T, H, I) if ws is None else ws
    y = mse.mlp_swiglu_forward(to_dev(x), to_dev(wgu), to_dev(wd), workspace=ws)
    torch.cuda.synchronize()
    return to_bits(y), ws


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("T,H,I", [(1, 384, 320), (7, 384, 320), (24, 512, 256), (64, 1024, 768),
                                   (100, 640, 448), (256, 384, 320), (40, 768, 640)])
def test_one_launch_matches_oracle_and_two_launches(T, H, I, mode):
    x, wgu, wd = case(T, H, I, 7000 + T + H)
    y_ref, _, _ = oracle.mlp_forward(x, wgu, wd)
    with one_launch(mode):
        y1, ws = forward(x, wgu, wd)
    with one_launch(0):
        y2, _ = forward(x, wgu, wd)
    assert_close(bits_f64(y1), bits_f64(y_ref), f"one launch (mode {mode}) T={T}")
    assert_close(bits_f64(y2), bits_f64(y_ref), f"two launches T={T}")
    tail = ws[sync_region_offset(T, H, I):]
    assert int(torch.count_nonzero(tail).item()) == 0, "sync words not left zero"


@pytest.mark.parametrize("mode", [1, 2])
def test_one_launch_decode_t64_sampled_rows(mode):
    w = W.DECODE_T64
    wgu, wd = W.make_mlp_weights(w)
    x = W.make_x(w)
    rows = [0, 17, 31, 63]
    y_ref, _, _ = oracle.mlp_forward(x[rows], wgu, wd)
    with one_launch(mode):
        y, ws = forward(x, wgu, wd)
        y_again, _ = forward(x, wgu, wd, ws)
    assert_close(bits_f64(y[rows]), bits_f64(y_ref), "decode T=64 one launch")
    assert np.array_equal(y, y_again), "not deterministic across calls"
    tail = ws[sync_region_offset(w.T, w.H, w.I):]
    assert int(torch.count_nonzero(tail).item()) == 0


def test_one_launch_alternating_inputs_on_one_workspace():
    # stale flags would let the down phase read the previous call's h
    T, H, I = 48, 1024, 512
    cases = [case(T, H, I, 7100 + k) for k in range(2)]
    refs = [oracle.mlp_forward(*c)[0] for c in cases]
    ws = mse.new_mlp_workspace(T, H, I)
    dev = [tuple(to_dev(a) for a in c) for c in cases]
    with one_launch(2):
        for it in range(6):
            k = it % 2
            y = mse.mlp_swiglu_forward(*dev[k], workspace=ws)
            torch.cuda.synchronize()
            assert_close(bits_f64(to_bits(y)), bits_f64(refs[k]), f"call {it}")


def test_one_launch_shard_partials():
    T, H, I, tp = 32, 768, 384, 3
    x, wgu, wd = case(T, H, I, 7200)
    with one_launch(2):
        parts = mse.mlp_swiglu_shard_partial(to_dev(x), to_dev(wgu), to_dev(wd), tp, partial_dtype=torch.float32)
        sub = mse.mlp_swiglu_shard_partial(to_dev(x), to_dev(wgu), to_dev(wd), tp, rank_first=1, rank_count=2,
                                           partial_dtype=torch.float32)
    torch.cuda.synchronize()
    for r in range(tp):
        _, pr = oracle.shard_partial(x, wgu, wd, tp, r, oracle.F32)
        assert_close(parts[r].cpu().numpy(), pr, f"partial {r}")
        if r >= 1:
            assert_close(sub[r - 1].cpu().numpy(), pr, f"subset partial {r}")


def test_one_launch_cuda_graph_replay():
    # counters and flags are reset inside the kernel, so a captured launch replays
    T, H, I = 16, 512, 256
    _, wgu, wd = case(T, H, I, 7300)
    xs = [W.make_custom(7310 + k, 0, (T, H)) for k in range(3)]
    refs = [oracle.mlp_forward(x, wgu, wd)[0] for x in xs]
    dx = to_dev(xs[0])
    dgu, dwd = to_dev(wgu), to_dev(wd)
    ws = mse.new_mlp_workspace(T, H, I)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    with one_launch(2):
        mse.mlp_swiglu_forward(dx, dgu, dwd, y, ws)   # set-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                mse.mlp_swiglu_forward(dx, dgu, dwd, y, ws)
        torch.cuda.synchronize()
        for it in range(6):
            k = it % 3
            dx.copy_(to_dev(xs[k]))
            g.replay()
            torch.cuda.synchronize()
            assert_close(bits_f64(to_bits(y)), bits_f64(refs[k]), f"replay {it}")
