"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on the
same seeded inputs, for the five workloads and the edge cases of the method.

Criterion: |gpu - oracle| <= 0.02 + 0.02 |oracle| per element for floating
point; permutations (shard slices, rank-major <-> logical) bit-exact.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from tests.helpers import assert_close, bits_f64, kernel_path, prefill_kernel, to_bits, to_dev

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


_cache = {}


def mlp_inputs(w: W.Workload, T=None):
    key = (w.name, T)
    if key not in _cache:
        wgu, wd = W.make_mlp_weights(w)
        _cache[key] = (W.make_x(w, T), wgu, wd)
    return _cache[key]


def run_forward(x, wgu, wd):
    dx, dgu, dwd = to_dev(x), to_dev(wgu), to_dev(wd)
    T, H = x.shape
    I = wd.shape[1]
    ws = mse.new_mlp_workspace(T, H, I)
    y = mse.mlp_swiglu_forward(dx, dgu, dwd, workspace=ws)
    torch.cuda.synchronize()
    h = ws[: T * I * 2].view(torch.int16).view(T, I).cpu().numpy().view(np.uint16)
    return to_bits(y), h


# --------------------------------------------------------------------------- config 1
def test_tiny_sharded_tp4():
    w = W.TINY_SHARDED
    x, wgu, wd = mlp_inputs(w)
    y_ref, _, _ = oracle.mlp_forward(x, wgu, wd)
    y, _ = run_forward(x, wgu, wd)
    assert_close(bits_f64(y), bits_f64(y_ref), "replicated")
    parts = mse.mlp_swiglu_shard_partial(to_dev(x), to_dev(wgu), to_dev(wd), w.tp, partial_dtype=torch.float32)
    red = mse.shard_sum(parts)
    torch.cuda.synchronize()
    ref_parts = [oracle.shard_partial(x, wgu, wd, w.tp, r, oracle.F32)[1] for r in range(w.tp)]
    for r in range(w.tp):
        assert_close(parts[r].cpu().numpy(), ref_parts[r], f"partial {r}")
    ref_red = oracle.shard_sum(np.stack(ref_parts), oracle.F32)
    red_b = to_bits(red)
    assert_close(bits_f64(red_b), bits_f64(ref_red), "shard_sum")
    tpr = w.T // w.tp
    for r in range(w.tp):   # each rank's scatter share equals the replicated rows
        sl = slice(r * tpr, (r + 1) * tpr)
        assert_close(bits_f64(red_b[sl]), bits_f64(y_ref[sl]), f"rank {r} rows")


# --------------------------------------------------------------------------- config 2
@pytest.mark.parametrize("path", [mse.PATH_TENSORCORE, mse.PATH_GENERIC])
def test_decode_t64(path):
    w = W.DECODE_T64
    x, wgu, wd = mlp_inputs(w)
    y_ref, _, h_ref = oracle.mlp_forward(x, wgu, wd)
    with kernel_path(path):
        y, h = run_forward(x, wgu, wd)
        y2, _ = run_forward(x, wgu, wd)
    assert_close(bits_f64(h), bits_f64(h_ref), "h")
    r = assert_close(bits_f64(y), bits_f64(y_ref), "y")
    assert np.array_equal(y, y2), "not deterministic"
    print(f"decode T=64 path {path}: max err/tol {r:.3f}")


# --------------------------------------------------------------------------- config 3
def test_tp8_emulated_t128():
    w = W.TP8_EMULATED
    x, wgu, wd = mlp_inputs(w)
    dx, dgu, dwd = to_dev(x), to_dev(wgu), to_dev(wd)
    ws = mse.new_mlp_workspace(w.T, w.H, w.I)
    parts = mse.mlp_swiglu_shard_partial(dx, dgu, dwd, w.tp, workspace=ws)
    red = mse.shard_sum(parts)
    y = mse.mlp_swiglu_forward(dx, dgu, dwd, workspace=ws)
    torch.cuda.synchronize()
    ref_parts = []
    for r in range(w.tp):
        _, pr = oracle.shard_partial(x, wgu, wd, w.tp, r, oracle.BF16)
        ref_parts.append(pr)
        assert_close(bits_f64(to_bits(parts[r])), bits_f64(pr), f"partial {r}")
    ref_red = oracle.shard_sum(np.stack(ref_parts), oracle.BF16)
    assert_close(bits_f64(to_bits(red)), bits_f64(ref_red), "shard_sum")
    y_ref, _, _ = oracle.mlp_forward(x, wgu, wd)
    assert_close(bits_f64(to_bits(y)), bits_f64(y_ref), "replicated")
    # the pages' equivalence: the reduced partials reproduce the replicated output per token
    assert_close(bits_f64(to_bits(red)), bits_f64(y_ref), "sum of partials vs replicated")


def test_shard_subset_matches_all_shards():
    # rank_first/rank_count select the same partials (the split of the reduction
    # between CTAs differs, so floating point agrees to tolerance, not bit for bit)
    w = W.TP8_EMULATED
    x, wgu, wd = mlp_inputs(w)
    dx, dgu, dwd = to_dev(x), to_dev(wgu), to_dev(wd)
    allp = mse.mlp_swiglu_shard_partial(dx, dgu, dwd, w.tp)
    sub = mse.mlp_swiglu_shard_partial(dx, dgu, dwd, w.tp, rank_first=3, rank_count=2)
    one = mse.mlp_swiglu_shard_partial(dx, dgu, dwd, w.tp, rank_first=7, rank_count=1)
    torch.cuda.synchronize()
    assert_close(bits_f64(to_bits(sub)), bits_f64(to_bits(allp[3:5])), "ranks 3-4")
    assert_close(bits_f64(to_bits(one)), bits_f64(to_bits(allp[7:8])), "rank 7")


def integer_exact_mlp(T, H, I):
    """Inputs on which every step is exact in fp32 and fp64 whatever the summation
    order: x in {20, 24, ..., 40}; one-hot gate/up/down rows.  Then g, u in [20, 40],
    silu(g) rounds to g (e^-20 < 2^-25), h = g*u = 16*m with m <= 100 is a bf16
    value, and each output is one h value (the rest of its sum is exact zeros)."""
    rng = np.random.default_rng(T + H + I)
    xv = 4.0 * rng.integers(5, 11, size=(T, H))
    x = W.f32_to_bf16_bits(xv.astype(np.float32))
    wgu = np.zeros((2 * I, H), dtype=np.uint16)
    j = np.arange(I)
    wgu[j, j % H] = 0x3F80
    wgu[I + j, (7 * j + 3) % H] = 0x3F80
    wd = np.zeros((H, I), dtype=np.uint16)
    n = np.arange(H)
    wd[n, (5 * n + 1) % I] = 0x3F80
    return x, wgu, wd


@pytest.mark.parametrize("path", [mse.PATH_TENSORCORE, mse.PATH_GENERIC])
@pytest.mark.parametrize("T", [18, 300])
def test_shard_slices_bit_exact(path, T):
    # the shard index map (gate rows, up rows I + ..., down columns of slice r) checked
    # bit-exactly through the kernels against the oracle
    H, I, tp = 384, 192, 3
    x, wgu, wd = integer_exact_mlp(T, H, I)
    with kernel_path(path):
        parts = mse.mlp_swiglu_shard_partial(to_dev(x), to_dev(wgu), to_dev(wd), tp)
        sub = mse.mlp_swiglu_shard_partial(to_dev(x), to_dev(wgu), to_dev(wd), tp, rank_first=1, rank_count=2)
        y, _ = run_forward(x, wgu, wd)
    torch.cuda.synchronize()
    for r in range(tp):
        _, pr = oracle.shard_partial(x, wgu, wd, tp, r, oracle.BF16)
        assert np.array_equal(to_bits(parts[r]), pr), f"partial {r}"
    assert torch.equal(sub, parts[1:3])
    y_ref, _, _ = oracle.mlp_forward(x, wgu, wd)
    assert np.array_equal(y, y_ref)
    assert np.array_equal(to_bits(mse.shard_sum(parts)), y_ref)


# --------------------------------------------------------------------------- config 4
def test_mla_merged_tp16():
    w = W.MLA_MERGED
    x = W.make_x(w)
    wm = W.make_merged_weight(w)
    lo, rm = mse.merged_proj_forward(to_dev(x), to_dev(wm), w.q_dim, w.kv_dim, w.tp)
    back = mse.merged_proj_reorder(rm, w.q_dim, w.kv_dim, w.tp)
    torch.cuda.synchronize()
    lo_b, rm_b, back_b = to_bits(lo), to_bits(rm), to_bits(back)
    ref_lo, ref_rm, _ = oracle.merged_proj(x, wm, w.q_dim, w.kv_dim, w.tp)
    assert_close(bits_f64(lo_b), bits_f64(ref_lo), "logical")
    assert_close(bits_f64(rm_b), bits_f64(ref_rm), "rank-major")
    perm = oracle.rank_major_to_logical(w.q_dim, w.kv_dim, w.tp)
    assert np.array_equal(rm_b, lo_b[:, perm]), "rank-major is not the gather permutation of logical"
    assert np.array_equal(back_b, lo_b), "reorder did not restore the logical layout"
    assert np.array_equal(back_b, oracle.reorder(rm_b, w.q_dim, w.kv_dim, w.tp))


def test_mla_permutation_exact_through_projection():
    # integer-valued x and one-hot weight rows: every output is an exact integer
    q, kv, tp, H, T = 1536, 576, 16, 7168, 128
    C = q + kv
    xi = ((np.arange(T * H).reshape(T, H) * 7) % 201) - 100
    x = W.f32_to_bf16_bits(xi.astype(np.float32))
    wm = np.zeros((C, H), dtype=np.uint16)
    wm[np.arange(C), (np.arange(C) * 3) % H] = 0x3F80      # 1.0
    lo, rm = mse.merged_proj_forward(to_dev(x), to_dev(wm), q, kv, tp)
    torch.cuda.synchronize()
    ref_lo, ref_rm, _ = oracle.merged_proj(x, wm, q, kv, tp)
    assert np.array_equal(to_bits(lo), ref_lo)
    assert np.array_equal(to_bits(rm), ref_rm)


# --------------------------------------------------------------------------- config 5
_prefill_ref = {}


def prefill_reference():
    """The oracle's h and y for all 8192 token rows of the prefill workload, computed
    once for the module (about 1.1e12 fp64 multiply-adds: minutes on a few host cores)."""
    if not _prefill_ref:
        w = W.PREFILL_T8192
        x, wgu, wd = mlp_inputs(w)
        y_ref, _, h_ref = oracle.mlp_forward(x, wgu, wd)
        _prefill_ref.update(y=y_ref, h=h_ref)
    return _prefill_ref


@pytest.mark.parametrize("kind", [mse.PREFILL_PAIR, mse.PREFILL_SINGLE])
def test_prefill_t8192_all_rows(kind):
    # every h and y element of the 8192-token layer, for both prefill kernels: every
    # tile that their persistent schedulers hand out is compared
    w = W.PREFILL_T8192
    x, wgu, wd = mlp_inputs(w)
    with prefill_kernel(kind):
        y, h = run_forward(x, wgu, wd)
    ref = prefill_reference()
    assert_close(bits_f64(h), bits_f64(ref["h"]), "h, all rows")
    r = assert_close(bits_f64(y), bits_f64(ref["y"]), "y, all rows")
    print(f"prefill all 8192 rows, kernel {kind}: max err/tol {r:.3f}")


# --------------------------------------------------------------------------- edge cases
def small_case(T, H, I, seed):
    x = W.make_custom(seed, 0, (T, H))
    wgu = W.make_custom(seed, 1, (2 * I, H), 1 / math.sqrt(H))
    wd = W.make_custom(seed, 2, (H, I), 1 / math.sqrt(I))
    return x, wgu, wd


@pytest.mark.parametrize("T", [1, 7, 16, 17, 100, 200, 256, 257, 300, 383])
@pytest.mark.parametrize("path", [mse.PATH_TENSORCORE, mse.PATH_GENERIC])
def test_ragged_tokens(T, path):
    H, I = 384, 320
    x, wgu, wd = small_case(T, H, I, 1000 + T)
    y_ref, _, h_ref = oracle.mlp_forward(x, wgu, wd)
    with kernel_path(path):
        y, h = run_forward(x, wgu, wd)
    assert_close(bits_f64(h), bits_f64(h_ref), f"h T={T}")
    assert_close(bits_f64(y), bits_f64(y_ref), f"y T={T}")


@pytest.mark.parametrize("T", [192, 256])
@pytest.mark.parametrize("swapab_max_t", [160, 256])
def test_near_ridge_tokens_decode_weights(T, swapab_max_t):
    # 129-256 tokens on the Kimi-K3 shapes: the CTA-pair prefill kernels (default above 160
    # tokens for the full layer) and the swap-AB kernels (forced), every row against the oracle
    w = W.DECODE_T64
    wgu, wd = W.make_mlp_weights(w)
    x = W.make_custom(1800 + T, 0, (T, w.H))
    old = mse.set_tuning(mse.TUNE_SWAPAB_MAX_T, swapab_max_t)
    try:
        with kernel_path(mse.PATH_TENSORCORE):
            y, h = run_forward(x, wgu, wd)
    finally:
        mse.set_tuning(mse.TUNE_SWAPAB_MAX_T, old)
    y_ref, _, h_ref = oracle.mlp_forward(x, wgu, wd)
    assert_close(bits_f64(h), bits_f64(h_ref), f"h T={T}")
    r = assert_close(bits_f64(y), bits_f64(y_ref), f"y T={T}")
    print(f"T={T} swap-AB up to {swapab_max_t}: max err/tol {r:.3f}")


@pytest.mark.parametrize("T", [161, 200, 256])
def test_pair_kernel_split_k(T):
    # 161-256 tokens over at least 4096 weight rows take the CTA-pair kernel, whose tiles are
    # then split over more clusters (at most two parts each; the CTA arriving last adds the
    # other part, from its idle ring or from L2).  On a workspace that is 0xFF except the
    # sync range: every row within tolerance of the oracle, bit-identical to a fresh
    # workspace and to a second run (parts summed in part order), the counters left zero;
    # and within tolerance with the split switched off.
    H, I = 1024, 2048
    x, wgu, wd = small_case(T, H, I, 5100 + T)
    dx, dgu, dwd = to_dev(x), to_dev(wgu), to_dev(wd)
    n = mse.mlp_swiglu_workspace_bytes(T, H, I)
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
    off, b = mse.mlp_swiglu_workspace_sync_range(T, H, I, n)
    ws[off:off + b].zero_()
    with kernel_path(mse.PATH_TENSORCORE), prefill_kernel(mse.PREFILL_PAIR):
        old = mse.set_tuning(mse.TUNE_PAIR_SPLIT, 1)
        try:
            y = mse.mlp_swiglu_forward(dx, dgu, dwd, workspace=ws)
            torch.cuda.synchronize()
            h = ws[: T * I * 2].view(torch.int16).view(T, I).cpu().numpy().view(np.uint16).copy()
            y_fresh = mse.mlp_swiglu_forward(dx, dgu, dwd)
            y_again = mse.mlp_swiglu_forward(dx, dgu, dwd, workspace=ws)
            mse.set_tuning(mse.TUNE_PAIR_SPLIT, 0)
            y_whole = mse.mlp_swiglu_forward(dx, dgu, dwd)
        finally:
            mse.set_tuning(mse.TUNE_PAIR_SPLIT, old)
    torch.cuda.synchronize()
    assert torch.equal(y, y_fresh) and torch.equal(y, y_again)
    assert int(torch.count_nonzero(ws[off:off + b]).item()) == 0
    y_ref, _, h_ref = oracle.mlp_forward(x, wgu, wd)
    assert_close(bits_f64(h), bits_f64(h_ref), f"h T={T}")
    assert_close(bits_f64(to_bits(y)), bits_f64(y_ref), f"y T={T} split")
    assert_close(bits_f64(to_bits(y_whole)), bits_f64(y_ref), f"y T={T} whole tiles")
    assert mse.poll_device_error() == 0


@pytest.mark.parametrize("T", [257, 300, 512, 700, 1000])
@pytest.mark.parametrize("kind", [mse.PREFILL_SINGLE, mse.PREFILL_PAIR])
def test_prefill_kernels_ragged(T, kind):
    H, I = 384, 320
    x, wgu, wd = small_case(T, H, I, 3000 + T)
    y_ref, _, h_ref = oracle.mlp_forward(x, wgu, wd)
    with kernel_path(mse.PATH_TENSORCORE), prefill_kernel(kind):
        y, h = run_forward(x, wgu, wd)
    assert_close(bits_f64(h), bits_f64(h_ref), f"h T={T}")
    assert_close(bits_f64(y), bits_f64(y_ref), f"y T={T}")


@pytest.mark.parametrize("kind", [mse.PREFILL_SINGLE, mse.PREFILL_PAIR])
def test_prefill_kernels_shards_and_merged(kind):
    T, H, I, tp = 600, 384, 192, 3
    x, wgu, wd = small_case(T, H, I, 4242)
    with kernel_path(mse.PATH_TENSORCORE), prefill_kernel(kind):
        parts = mse.mlp_swiglu_shard_partial(to_dev(x), to_dev(wgu), to_dev(wd), tp, partial_dtype=torch.float32)
        q, kv, tpm = 96, 36, 4
        wm = W.make_custom(4243, 4, (q + kv, H), 1 / 16)
        lo, rm = mse.merged_proj_forward(to_dev(x), to_dev(wm), q, kv, tpm)
    torch.cuda.synchronize()
    for r in range(tp):
        _, pr = oracle.shard_partial(x, wgu, wd, tp, r, oracle.F32)
        assert_close(parts[r].cpu().numpy(), pr, f"partial {r}")
    ref_lo, ref_rm, _ = oracle.merged_proj(x, wm, q, kv, tpm)
    assert_close(bits_f64(to_bits(lo)), bits_f64(ref_lo), "merged logical")
    assert np.array_equal(to_bits(rm), to_bits(lo)[:, oracle.rank_major_to_logical(q, kv, tpm)])


@pytest.mark.parametrize("T,H,I", [(5, 16, 12), (3, 40, 24), (9, 100, 36), (130, 72, 48)])
def test_unaligned_shapes_take_generic_path(T, H, I):
    x, wgu, wd = small_case(T, H, I, 7 * T + H)
    y_ref, _, _ = oracle.mlp_forward(x, wgu, wd)
    y, _ = run_forward(x, wgu, wd)
    assert_close(bits_f64(y), bits_f64(y_ref), "y")
    with kernel_path(mse.PATH_TENSORCORE):
        with pytest.raises(mse.MSEError) as e:
            run_forward(x, wgu, wd)
        assert e.value.name == "MSE_ERR_UNSUPPORTED_SHAPE"


@pytest.mark.parametrize("T", [4, 64, 300])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_sharded_edge(T, dtype):
    H, I, tp = 384, 192, 3          # s = 64
    x, wgu, wd = small_case(T, H, I, 50 + T)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    parts = mse.mlp_swiglu_shard_partial(to_dev(x), to_dev(wgu), to_dev(wd), tp, partial_dtype=td)
    torch.cuda.synchronize()
    for r in range(tp):
        _, pr = oracle.shard_partial(x, wgu, wd, tp, r, od)
        got = to_bits(parts[r]) if dtype == "bf16" else parts[r].cpu().numpy()
        ref = pr if dtype == "f32" else pr
        assert_close(bits_f64(got) if dtype == "bf16" else got, bits_f64(ref) if dtype == "bf16" else ref,
                     f"partial {r}")


@pytest.mark.parametrize("T", [1, 33, 300])
def test_merged_edge(T):
    q, kv, tp, H = 96, 36, 4, 256
    x = W.make_custom(77 + T, 0, (T, H))
    wm = W.make_custom(77 + T, 4, (q + kv, H), 1 / 16)
    lo, rm = mse.merged_proj_forward(to_dev(x), to_dev(wm), q, kv, tp)
    only_rm = mse.merged_proj_forward(to_dev(x), to_dev(wm), q, kv, tp, logical=False)[1]
    torch.cuda.synchronize()
    ref_lo, ref_rm, _ = oracle.merged_proj(x, wm, q, kv, tp)
    assert_close(bits_f64(to_bits(lo)), bits_f64(ref_lo), "logical")
    perm = oracle.rank_major_to_logical(q, kv, tp)
    assert np.array_equal(to_bits(rm), to_bits(lo)[:, perm])
    assert np.array_equal(to_bits(only_rm), to_bits(rm))


@pytest.mark.parametrize("n,dtype", [(8, "bf16"), (4, "f32"), (3, "bf16")])
def test_shard_sum_ragged(n, dtype):
    T, H = 6 * n, 131          # plane not a multiple of 8 -> scalar kernel
    rng = np.random.default_rng(n)
    vals = rng.standard_normal((n, T, H)).astype(np.float32)
    if dtype == "bf16":
        p = W.f32_to_bf16_bits(vals).reshape(n, T, H)
        dev = to_dev(p)
        ref = oracle.shard_sum(p, oracle.BF16)
    else:
        dev = torch.from_numpy(vals).cuda()
        ref = oracle.shard_sum(vals, oracle.F32)
    out = mse.shard_sum(dev)
    torch.cuda.synchronize()
    assert_close(bits_f64(to_bits(out)), bits_f64(ref), "shard_sum")


def test_workspace_reuse_across_shapes_and_calls():
    # one zeroed workspace serves consecutive calls of different sizes
    H, I = 384, 320
    ws = mse.new_mlp_workspace(256, H, I)
    outs = []
    for T in [256, 40, 256]:
        x, wgu, wd = small_case(T, H, I, 999)
        y = mse.mlp_swiglu_forward(to_dev(x), to_dev(wgu), to_dev(wd), workspace=ws)
        outs.append(to_bits(y))
    assert np.array_equal(outs[0], outs[2])
    assert mse.poll_device_error() == 0


def test_workspace_reuse_across_token_counts_wide_grid():
    # Shapes whose split-K tiles occupy many CTAs' partial-tile slots: a 256-token call
    # writes fp32 tiles far into the buffer, and each later call with fewer (or more than
    # 256) tokens must still find its sync words zero.  Every call equals the same call
    # on a fresh workspace bit for bit (same launches, deterministic sums).
    H, I = 2048, 1536
    _, wgu, wd = small_case(8, H, I, 1200)
    dgu, dwd = to_dev(wgu), to_dev(wd)
    ws = mse.new_mlp_workspace(300, H, I)
    for T in [256, 64, 300, 7, 256, 130, 64, 1]:
        x = to_dev(W.make_custom(1210 + T, 0, (T, H)))
        y = mse.mlp_swiglu_forward(x, dgu, dwd, workspace=ws)
        s = mse.mlp_swiglu_shard_forward(x, dgu, dwd, 4, rank_first=1, rank_count=2, workspace=ws)
        y_fresh = mse.mlp_swiglu_forward(x, dgu, dwd)
        s_fresh = mse.mlp_swiglu_shard_forward(x, dgu, dwd, 4, rank_first=1, rank_count=2)
        torch.cuda.synchronize()
        assert torch.equal(y, y_fresh), f"T={T}"
        assert torch.equal(s, s_fresh), f"T={T} shard group"
    assert mse.poll_device_error() == 0
    # the merged projection's workspace in the same way
    q, kv, tp = 1536, 576, 16
    wm = to_dev(W.make_custom(1230, 4, (q + kv, H), 1 / 45))
    wsm = mse.new_merged_workspace(256, H, q, kv)
    for T in [256, 16, 200, 1]:
        x = to_dev(W.make_custom(1240 + T, 0, (T, H)))
        lo, _ = mse.merged_proj_forward(x, wm, q, kv, tp, workspace=wsm)
        lo_fresh, _ = mse.merged_proj_forward(x, wm, q, kv, tp)
        torch.cuda.synchronize()
        assert torch.equal(lo, lo_fresh), f"merged T={T}"
    assert mse.poll_device_error() == 0


@pytest.mark.parametrize("one_launch", [0, 1])
def test_workspace_poisoned_except_the_sync_range(one_launch):
    # Every byte of the workspace is 0xFF except the range the sync-range query names,
    # which is zeroed: the calls must equal the same calls on a fresh workspace bit for
    # bit, so that range holds every counter, flag and count the kernels rely on (the
    # static-scratch entry point zeroes exactly this range of its array).
    H, I = 2048, 1536
    _, wgu, wd = small_case(8, H, I, 1300)
    dgu, dwd = to_dev(wgu), to_dev(wd)
    n = mse.mlp_swiglu_workspace_bytes(256, H, I)
    old = mse.set_tuning(mse.TUNE_ONE_LAUNCH, one_launch)
    try:
        for T in [64, 256, 7]:
            x = to_dev(W.make_custom(1310 + T, 0, (T, H)))
            ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
            off, b = mse.mlp_swiglu_workspace_sync_range(T, H, I, n)
            ws[off:off + b].zero_()
            y = mse.mlp_swiglu_forward(x, dgu, dwd, workspace=ws)
            torch.cuda.synchronize()
            ws[:off].fill_(0xFF)          # poison h and the partial tiles again between calls
            s = mse.mlp_swiglu_shard_forward(x, dgu, dwd, 8, rank_first=3, rank_count=1, workspace=ws)
            y_fresh = mse.mlp_swiglu_forward(x, dgu, dwd)
            s_fresh = mse.mlp_swiglu_shard_forward(x, dgu, dwd, 8, rank_first=3, rank_count=1)
            torch.cuda.synchronize()
            assert torch.equal(y, y_fresh), f"T={T}"
            assert torch.equal(s, s_fresh), f"T={T} narrow shard"
            assert int(torch.count_nonzero(ws[off:off + b]).item()) == 0   # left zero again
    finally:
        mse.set_tuning(mse.TUNE_ONE_LAUNCH, old)
    assert mse.poll_device_error() == 0
    q, kv, tp = 1536, 576, 16
    wm = to_dev(W.make_custom(1330, 4, (q + kv, H), 1 / 45))
    n = mse.merged_proj_workspace_bytes(128, H, q, kv)
    x = to_dev(W.make_custom(1340, 0, (128, H)))
    wsm = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
    off, b = mse.merged_proj_workspace_sync_range(128, H, q, kv, n)
    wsm[off:off + b].zero_()
    lo, _ = mse.merged_proj_forward(x, wm, q, kv, tp, workspace=wsm)
    lo_fresh, _ = mse.merged_proj_forward(x, wm, q, kv, tp)
    torch.cuda.synchronize()
    assert torch.equal(lo, lo_fresh)
    assert mse.poll_device_error() == 0


def test_timeout_selftest_reports_and_context_survives():
    mse.selftest_wait_timeout(2_000_000)          # 2 ms wait that nothing satisfies
    assert mse.STATUS[mse.poll_device_error()] == "MSE_ERR_TIMEOUT"
    assert mse.poll_device_error() == 0            # the error word was cleared
    a = torch.ones(1024, device="cuda")
    assert float(a.sum().item()) == 1024.0          # the context is still usable
