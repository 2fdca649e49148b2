"""The decode-size kernels run as CTA pairs (one 256-row weight tile per pair, one
M = 256 MMA over both CTAs, each CTA holding half of the token rows) against the fp64
oracle, with the pair path forced on for every token count and forced off.

Shapes include odd numbers of 128-row tiles, where the second CTA of the last pair has
no tile of its own, ragged token counts, shard partials and the merged projection.
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
def pairs(min_t: int):
    old = mse.set_tuning(mse.TUNE_PAIR_MIN_T, min_t)
    assert old >= 0
    try:
        yield
    finally:
        mse.set_tuning(mse.TUNE_PAIR_MIN_T, old)


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


@pytest.mark.parametrize("min_t", [1, 0])
@pytest.mark.parametrize("T,H,I", [(7, 384, 320), (64, 1024, 768), (65, 640, 448), (130, 640, 448),
                                   (256, 384, 320), (200, 896, 192)])
def test_mlp_pairs(T, H, I, min_t):
    x, wgu, wd = case(T, H, I, 9000 + T + H + I)
    y_ref, _, h_ref = oracle.mlp_forward(x, wgu, wd)
    with pairs(min_t):
        y, h = forward(x, wgu, wd)
    assert_close(bits_f64(h), bits_f64(h_ref), f"h T={T} pairs from {min_t}")
    assert_close(bits_f64(y), bits_f64(y_ref), f"y T={T} pairs from {min_t}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_shard_partials_pairs(dtype):
    T, H, I, tp = 96, 768, 384, 3
    x, wgu, wd = case(T, H, I, 9100)
    pdt = torch.float32 if dtype == "f32" else torch.bfloat16
    code = oracle.F32 if dtype == "f32" else oracle.BF16
    with pairs(1):
        parts = mse.mlp_swiglu_shard_partial(to_dev(x), to_dev(wgu), to_dev(wd), tp, partial_dtype=pdt)
        red = mse.shard_sum(parts)
    torch.cuda.synchronize()
    refs = []
    for r in range(tp):
        _, pr = oracle.shard_partial(x, wgu, wd, tp, r, code)
        refs.append(pr)
        got = parts[r].cpu().numpy() if dtype == "f32" else bits_f64(to_bits(parts[r]))
        want = pr if dtype == "f32" else bits_f64(pr)
        assert_close(got, want, f"partial {r}")
    assert_close(bits_f64(to_bits(red)), bits_f64(oracle.shard_sum(np.stack(refs), code)), "shard_sum")


@pytest.mark.parametrize("T,q,kv,tp", [(40, 512, 192, 8), (128, 96, 36, 4), (100, 1536, 576, 16)])
def test_merged_pairs(T, q, kv, tp):
    H = 2048
    x = W.make_custom(9200 + T, 0, (T, H))
    wm = W.make_custom(9200 + T, 4, (q + kv, H), 1 / math.sqrt(H))
    ref_lo, ref_rm, _ = oracle.merged_proj(x, wm, q, kv, tp)
    with pairs(1):
        lo, rm = mse.merged_proj_forward(to_dev(x), to_dev(wm), q, kv, tp)
    torch.cuda.synchronize()
    assert_close(bits_f64(to_bits(lo)), bits_f64(ref_lo), "logical")
    assert_close(bits_f64(to_bits(rm)), bits_f64(ref_rm), "rank-major")


def test_pairs_integer_exact():
    # one-hot weights and integer inputs: exact whatever the split; checks the row and
    # token index maps of both CTAs of a pair bit for bit
    T, H, I = 130, 384, 192
    rng = np.random.default_rng(5)
    x = W.f32_to_bf16_bits((4.0 * rng.integers(5, 11, size=(T, H))).astype(np.float32))
    wgu = np.zeros((2 * I, H), dtype=np.uint16)
    j = np.arange(I)
    wgu[j, j % H] = 0x3F80
    wgu[I + j, (7 * j + 3) % H] = 0x3F80
    wd = np.zeros((H, I), dtype=np.uint16)
    n = np.arange(H)
    wd[n, (5 * n + 1) % I] = 0x3F80
    y_ref, _, _ = oracle.mlp_forward(x, wgu, wd)
    with pairs(1):
        y, _ = forward(x, wgu, wd)
    assert np.array_equal(y, y_ref)
