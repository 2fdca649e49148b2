"""The shards' partials summed inside the down projection (mlp_swiglu_shard_forward)
and the sequence-parallel MLP block (sequence_parallel_mlp) against the fp64 oracle.

The oracle's reading: the group's fp64 partials summed, ranks ascending, and rounded
once (the reduce-scatter's sum with no partial rounded to a storage dtype).  Also:
the TP4 and TP16 shard shapes of the 7168 x 6144 shared expert (slices of 1536 and
384 intermediate columns), the shapes the pages' tuned GEMM table lists besides TP8.

Criterion: |gpu - oracle| <= 0.02 + 0.02 |oracle| per element; bit-exact where the
inputs make every sum exact.
"""
import contextlib
import math

import numpy as np
import pytest

import oracle
import workloads as W
from tests.helpers import assert_close, bits_f64, kernel_path, to_bits, to_dev

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
    old = mse.set_tuning(mse.TUNE_ONE_LAUNCH, mode)
    assert old >= 0
    try:
        yield
    finally:
        mse.set_tuning(mse.TUNE_ONE_LAUNCH, old)


def case(T, H, I, seed):
    x = W.make_custom(seed, 0, (T, H))
    wgu = W.make_custom(seed, 1, (2 * I, H), 1 / math.sqrt(H))
    wd = W.make_custom(seed, 2, (H, I), 1 / math.sqrt(I))
    return x, wgu, wd


def got_f64(t, dtype):
    return bits_f64(to_bits(t)) if dtype == oracle.BF16 else t.cpu().numpy().astype(np.float64)


def ref_f64(r, dtype):
    return bits_f64(r) if dtype == oracle.BF16 else r.astype(np.float64)


_decode = {}


def decode_weights():
    if not _decode:
        w = W.DECODE_T64
        wgu, wd = W.make_mlp_weights(w)
        _decode.update(x=W.make_x(w), wgu=wgu, wd=wd, dgu=to_dev(wgu), dwd=to_dev(wd))
    return _decode


# ------------------------------------------------------------------ shapes and subsets
@pytest.mark.parametrize("T,H,I,tp,rf,rc", [
    (1, 384, 384, 3, 0, 3), (7, 768, 384, 3, 1, 2), (64, 1024, 768, 4, 0, 4), (65, 640, 512, 4, 1, 2),
    (130, 512, 1024, 8, 3, 4), (256, 384, 768, 4, 2, 1), (257, 512, 512, 4, 0, 4), (300, 384, 768, 3, 1, 2)])
@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.F32])
def test_shard_forward_matches_oracle(T, H, I, tp, rf, rc, dtype):
    x, wgu, wd = case(T, H, I, 9600 + T + H + I + rf)
    td = torch.bfloat16 if dtype == oracle.BF16 else torch.float32
    out = mse.mlp_swiglu_shard_forward(to_dev(x), to_dev(wgu), to_dev(wd), tp, rank_first=rf, rank_count=rc,
                                       out_dtype=td)
    torch.cuda.synchronize()
    _, ref = oracle.shard_group_sum(x, wgu, wd, tp, rf, rc, dtype)
    assert_close(got_f64(out, dtype), ref_f64(ref, dtype), f"T={T} ranks {rf}..{rf + rc - 1}")


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("rf,rc", [(0, 4), (1, 2), (3, 1)])
def test_shard_forward_one_launch(mode, rf, rc):
    # the one-launch layer over a column range that starts inside the intermediate dim
    T, H, I, tp = 48, 768, 1024, 4
    x, wgu, wd = case(T, H, I, 9700 + rf)
    with one_launch(mode):
        out = mse.mlp_swiglu_shard_forward(to_dev(x), to_dev(wgu), to_dev(wd), tp, rank_first=rf, rank_count=rc)
        again = mse.mlp_swiglu_shard_forward(to_dev(x), to_dev(wgu), to_dev(wd), tp, rank_first=rf,
                                             rank_count=rc)
    torch.cuda.synchronize()
    _, ref = oracle.shard_group_sum(x, wgu, wd, tp, rf, rc, oracle.BF16)
    assert_close(bits_f64(to_bits(out)), bits_f64(ref), f"one launch mode {mode}")
    assert torch.equal(out, again)


@pytest.mark.parametrize("path", [mse.PATH_TENSORCORE, mse.PATH_GENERIC])
@pytest.mark.parametrize("T", [18, 300])
def test_shard_forward_bit_exact_on_integer_inputs(path, T):
    # one-hot weights, integer inputs: each output is one h value or an exact zero, so
    # the group's column range is checked bit for bit through the kernels
    H, I, tp = 384, 192, 3
    rng = np.random.default_rng(T + H + I)
    x = W.f32_to_bf16_bits((4.0 * rng.integers(5, 11, size=(T, H))).astype(np.float32))
    wgu = np.zeros((2 * I, H), dtype=np.uint16)
    j = np.arange(I)
    wgu[j, j % H] = 0x3F80
    wgu[I + j, (7 * j + 3) % H] = 0x3F80
    wd = np.zeros((H, I), dtype=np.uint16)
    n = np.arange(H)
    wd[n, (5 * n + 1) % I] = 0x3F80
    with kernel_path(path):
        for rf, rc in [(0, 3), (1, 1), (1, 2)]:
            out = mse.mlp_swiglu_shard_forward(to_dev(x), to_dev(wgu), to_dev(wd), tp, rank_first=rf,
                                               rank_count=rc)
            torch.cuda.synchronize()
            _, ref = oracle.shard_group_sum(x, wgu, wd, tp, rf, rc, oracle.BF16)
            assert np.array_equal(to_bits(out), ref), f"ranks {rf}..{rf + rc - 1}"


def test_shard_forward_unaligned_shape_takes_generic_path():
    T, H, I, tp = 9, 100, 36, 4
    x, wgu, wd = case(T, H, I, 9800)
    out = mse.mlp_swiglu_shard_forward(to_dev(x), to_dev(wgu), to_dev(wd), tp, rank_first=1, rank_count=2)
    torch.cuda.synchronize()
    _, ref = oracle.shard_group_sum(x, wgu, wd, tp, 1, 2, oracle.BF16)
    assert_close(bits_f64(to_bits(out)), bits_f64(ref), "generic")


# ------------------------------------------------------------------ joint finish of narrow slices
@contextlib.contextmanager
def coop(threshold: int):
    old = mse.set_tuning(mse.TUNE_COOP_FINISH, threshold)
    assert old >= 0
    try:
        yield
    finally:
        mse.set_tuning(mse.TUNE_COOP_FINISH, old)


@pytest.mark.parametrize("T", [1, 16, 33, 64, 130, 256])
@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.F32])
def test_one_shard_many_way_split_joint_finish(T, dtype):
    # One shard of a narrow slice: two gate_up tiles of 64 columns over 64 k-blocks each,
    # so every tile is split between dozens of CTAs and the kernels that finish such
    # tiles jointly run (default threshold) or not (threshold 0).  Both sum the parts in
    # the same order: results must agree bit for bit, and with the oracle.
    H, I, tp, rank = 4096, 1024, 8, 5
    x, wgu, wd = case(T, H, I, 9400 + T)
    td = torch.bfloat16 if dtype == oracle.BF16 else torch.float32
    dx, dgu, dwd = to_dev(x), to_dev(wgu), to_dev(wd)
    with coop(6):
        a = mse.mlp_swiglu_shard_partial(dx, dgu, dwd, tp, rank_first=rank, rank_count=1, partial_dtype=td)
        ga = mse.mlp_swiglu_shard_forward(dx, dgu, dwd, tp, rank_first=rank, rank_count=1, out_dtype=td)
    with coop(0):
        b = mse.mlp_swiglu_shard_partial(dx, dgu, dwd, tp, rank_first=rank, rank_count=1, partial_dtype=td)
    torch.cuda.synchronize()
    assert torch.equal(a, b), "joint finish differs from the finish by the last CTA"
    assert torch.equal(a[0], ga)
    _, pr = oracle.shard_partial(x, wgu, wd, tp, rank, dtype)
    assert_close(got_f64(a[0], dtype), ref_f64(pr, dtype), f"T={T}")


@pytest.mark.parametrize("T", [16, 64, 130])
def test_down_projection_joint_finish_bf16_and_f32(T):
    # Two 128-row down tiles over long reductions (64 and 32 k-blocks): each tile is split
    # between dozens of CTAs, so the down kernels with the joint finish write the bf16
    # output and the fp32 partials in token slices.  Bit-identical to the finish by the
    # last CTA (threshold 0), and within tolerance of the oracle.
    H, I = 256, 4096
    x, wgu, wd = case(T, H, I, 9460 + T)
    dx, dgu, dwd = to_dev(x), to_dev(wgu), to_dev(wd)
    with coop(6):
        y = mse.mlp_swiglu_forward(dx, dgu, dwd)
        p32 = mse.mlp_swiglu_shard_partial(dx, dgu, dwd, 2, rank_first=1, rank_count=1,
                                           partial_dtype=torch.float32)
    with coop(0):
        y0 = mse.mlp_swiglu_forward(dx, dgu, dwd)
        p32_0 = mse.mlp_swiglu_shard_partial(dx, dgu, dwd, 2, rank_first=1, rank_count=1,
                                             partial_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(y, y0)
    assert torch.equal(p32, p32_0)
    y_ref, _, _ = oracle.mlp_forward(x, wgu, wd)
    assert_close(bits_f64(to_bits(y)), bits_f64(y_ref), f"y T={T}")
    _, pr = oracle.shard_partial(x, wgu, wd, 2, 1, oracle.F32)
    assert_close(p32[0].cpu().numpy().astype(np.float64), pr.astype(np.float64), f"fp32 partial T={T}")


@pytest.mark.parametrize("tp", [4, 16])
def test_joint_finish_h_matches_oracle(tp):
    # the SiLU*mul epilogue finished in token slices: h of the shard's columns
    T, H, I = 48, 2048, 1024
    x, wgu, wd = case(T, H, I, 9450 + tp)
    ws = mse.new_mlp_workspace(T, H, I)
    s = I // tp
    for rank in (0, tp - 1):
        mse.mlp_swiglu_shard_partial(to_dev(x), to_dev(wgu), to_dev(wd), tp, rank_first=rank, rank_count=1,
                                     workspace=ws)
        torch.cuda.synchronize()
        h = ws[: T * I * 2].view(torch.int16).view(T, I).cpu().numpy().view(np.uint16)
        h_ref = oracle.swiglu_hidden(x, wgu, I, rank * s, (rank + 1) * s)
        assert_close(bits_f64(h[:, rank * s:(rank + 1) * s]), bits_f64(h_ref), f"h tp{tp} rank {rank}")


# ------------------------------------------------------------------ the TP8 workload
def test_tp8_t128_summed_in_the_down_projection():
    # 128 gathered tokens, 8 shards of 768 intermediate columns: the whole group's sum
    w = W.TP8_EMULATED
    wgu, wd = W.make_mlp_weights(w)
    x = W.make_x(w)
    dx, dgu, dwd = to_dev(x), to_dev(wgu), to_dev(wd)
    ws = mse.new_mlp_workspace(w.T, w.H, w.I)
    out = mse.mlp_swiglu_shard_forward(dx, dgu, dwd, w.tp, workspace=ws)
    y = mse.mlp_swiglu_forward(dx, dgu, dwd, workspace=ws)
    parts = mse.mlp_swiglu_shard_partial(dx, dgu, dwd, w.tp, workspace=ws)
    red = mse.shard_sum(parts)
    torch.cuda.synchronize()
    # the same reduction over the same columns as the replicated layer: same launches, same bits
    assert torch.equal(out, y)
    # every one of the 128 token rows (8 ranks x 16) against the oracle's group sum
    _, ref = oracle.shard_group_sum(x, wgu, wd, w.tp, 0, w.tp, oracle.BF16)
    r = assert_close(bits_f64(to_bits(out)), bits_f64(ref), "summed partials, all rows")
    print(f"tp8 summed in the down projection: max err/tol {r:.3f}")
    # against the unfused path (bf16 partials, then their sum): both within tolerance of the oracle
    assert_close(bits_f64(to_bits(red)), bits_f64(ref), "partials then shard_sum")


# ------------------------------------------------------------------ TP4 / TP16 shard shapes
@pytest.mark.parametrize("tp,rank", [(4, 1), (4, 3), (16, 0), (16, 11)])
def test_tp4_tp16_shard_partials_decode_weights(tp, rank):
    # all 64 decode tokens of the rank's partial
    d = decode_weights()
    x = d["x"]
    part = mse.mlp_swiglu_shard_partial(to_dev(x), d["dgu"], d["dwd"], tp, rank_first=rank, rank_count=1)
    torch.cuda.synchronize()
    _, pr = oracle.shard_partial(x, d["wgu"], d["wd"], tp, rank, oracle.BF16)
    assert_close(bits_f64(to_bits(part[0])), bits_f64(pr), f"tp{tp} rank {rank} (s={6144 // tp})")


@pytest.mark.parametrize("tp,rf,rc", [(4, 0, 4), (16, 4, 4), (16, 15, 1)])
def test_tp4_tp16_summed_groups_decode_weights(tp, rf, rc):
    # all 64 decode tokens of the group's summed partials
    d = decode_weights()
    x = d["x"]
    out = mse.mlp_swiglu_shard_forward(to_dev(x), d["dgu"], d["dwd"], tp, rank_first=rf, rank_count=rc,
                                       out_dtype=torch.float32)
    torch.cuda.synchronize()
    _, ref = oracle.shard_group_sum(x, d["wgu"], d["wd"], tp, rf, rc, oracle.F32)
    assert_close(out.cpu().numpy().astype(np.float64), ref.astype(np.float64), f"tp{tp} ranks {rf}+{rc}")


# ------------------------------------------------------------------ the sequence-parallel block
@pytest.mark.parametrize("enabled", [True, False])
def test_sequence_parallel_mlp_block(enabled):
    # disjoint token blocks per rank; sharded or replicated, each rank's rows match
    # the replicated layer on its own tokens
    T, H, I, tp = 96, 1024, 768, 4
    x, wgu, wd = case(T, H, I, 9900)
    out, sharded = mse.sequence_parallel_mlp(to_dev(x), to_dev(wgu), to_dev(wd), tp, enabled)
    torch.cuda.synchronize()
    assert sharded is enabled
    tpr = T // tp
    for r in range(tp):
        own = np.arange(r * tpr, (r + 1) * tpr)
        y_ref, _, _ = oracle.mlp_forward(x[own], wgu, wd)
        assert_close(bits_f64(to_bits(out)[own]), bits_f64(y_ref), f"rank {r} rows")


def test_sequence_parallel_mlp_gate_falls_back_and_checks_blocks():
    T, H, I = 60, 640, 320        # 640 % 3 != 0; 640 and 320 both divide by 5
    x, wgu, wd = case(T, H, I, 9950)
    _, sharded = mse.sequence_parallel_mlp(to_dev(x), to_dev(wgu), to_dev(wd), 3, True)
    assert sharded is False       # 640 % 3 != 0: replicated, no error
    _, sharded = mse.sequence_parallel_mlp(to_dev(x), to_dev(wgu), to_dev(wd), 5, True)
    assert sharded is True
    with pytest.raises(ValueError):
        mse.sequence_parallel_mlp(to_dev(x), to_dev(wgu), to_dev(wd), 8, True)   # 60 % 8 != 0
    torch.cuda.synchronize()
