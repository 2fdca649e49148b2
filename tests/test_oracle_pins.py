"""Pins for the fp64 CPU oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: exact rational
brute force, closed forms, a library routine for a special case, values printed
on the pages, or the pages' sharded == replicated invariant.  A plausible slip
anywhere in the oracle (a dropped term, gate/up swapped, a transposed operand,
a wrong rounding point or rounding mode, a wrong permutation) fails one of them.
"""
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [p.strip() for p in line.split("|")]
            out[parts[0]] = parts[1:]
    return out


# ----------------------------------------------------------------------------------
# exact helpers (brute force)
# ----------------------------------------------------------------------------------

def bf16_exact(bits: int) -> Fraction:
    """Decode bf16 bits from the format definition (sign, 8-bit exponent, 7-bit fraction)."""
    s = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    assert e != 0xFF
    if e == 0:
        return s * Fraction(f, 1 << 7) * Fraction(1, 1 << 126)
    v = Fraction(128 + f, 128)
    return s * (v * (Fraction(2) ** (e - 127)))


def round_bf16_exact(v: Fraction):
    """Exact round-to-nearest-even onto the bf16 grid; returns (value, distance-to-tie ratio)."""
    if v == 0:
        return Fraction(0), 1.0
    a = abs(v)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = Fraction(2) ** (e - 7)
    n = a / q
    fl = n.numerator // n.denominator
    frac = n - fl
    if frac > Fraction(1, 2):
        r = fl + 1
    elif frac < Fraction(1, 2):
        r = fl
    else:
        r = fl if fl % 2 == 0 else fl + 1
    tie_dist = float(abs(frac - Fraction(1, 2)))
    return (1 if v > 0 else -1) * r * q, tie_dist


def silu_decimal(g: Fraction) -> Fraction:
    getcontext().prec = 60
    gd = Decimal(g.numerator) / Decimal(g.denominator)
    return Fraction(gd / (1 + (-gd).exp()))


def f64(bits):
    return oracle.bf16_array_to_f64(bits)


# ----------------------------------------------------------------------------------
# bf16 conversion and SiLU
# ----------------------------------------------------------------------------------

def test_bf16_decode_matches_format_definition():
    for bits in [0x0000, 0x8000, 0x3F80, 0xBF80, 0x4000, 0xC000, 0x0001, 0x007F, 0x0080,
                 0x7F7F, 0xFF7F, 0x3E4D, 0x4049]:
        assert oracle.bf16_to_f64(bits) == float(bf16_exact(bits)), hex(bits)
    assert math.isinf(oracle.bf16_to_f64(0x7F80))


def test_bf16_roundtrip_every_finite_pattern():
    L = oracle.lib()
    for bits in range(0x10000):
        e = (bits >> 7) & 0xFF
        if e == 0xFF:
            continue
        v = L.oracle_bf16_to_f64(bits)
        assert L.oracle_f64_to_bf16_rne(v) == bits, hex(bits)


def test_bf16_rne_midpoints_go_to_even():
    # For adjacent bf16 values a < b (positive), the exact midpoint rounds to the one
    # whose last fraction bit is 0, and points just off the midpoint go to the nearer one.
    L = oracle.lib()
    rng = np.random.default_rng(7)
    for bits in list(range(0x0000, 0x0100)) + list(rng.integers(0x0100, 0x7F7F, 3000)):
        bits = int(bits)
        a = L.oracle_bf16_to_f64(bits)
        b = L.oracle_bf16_to_f64(bits + 1)
        mid = (a + b) / 2.0                      # exact in binary64
        even = bits if bits % 2 == 0 else bits + 1
        assert L.oracle_f64_to_bf16_rne(mid) == even
        assert L.oracle_f64_to_bf16_rne(-mid) == (even | 0x8000)
        assert L.oracle_f64_to_bf16_rne(math.nextafter(mid, 0.0)) == bits
        assert L.oracle_f64_to_bf16_rne(math.nextafter(mid, math.inf)) == bits + 1


def test_bf16_rne_matches_torch_on_fp32_values():
    # For doubles that are fp32 values, direct fp64->bf16 rounding equals the library's
    # fp32->bf16 round-to-nearest-even conversion.
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 37.0,
                        (rng.standard_normal(2000) * 1e-39).astype(np.float32),
                        np.float32([3.3895314e38, -3.3895314e38, 1e-45, 65504.0, 0.0])])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    L = oracle.lib()
    got = np.array([L.oracle_f64_to_bf16_rne(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_overflow_and_specials():
    assert oracle.f64_to_bf16(1e300) == 0x7F80
    assert oracle.f64_to_bf16(-1e300) == 0xFF80
    assert oracle.f64_to_bf16(float("nan")) == 0x7FC0
    assert oracle.f64_to_bf16(-0.0) == 0x8000
    assert oracle.f64_to_bf16(1e-300) == 0x0000
    # largest finite bf16 and the halfway point to 2^128 (ties-to-even rounds up to inf)
    assert oracle.f64_to_bf16(float(bf16_exact(0x7F7F))) == 0x7F7F
    assert oracle.f64_to_bf16(float.fromhex("0x1.ffp127")) == 0x7F80
    assert oracle.f64_to_bf16(math.nextafter(float.fromhex("0x1.ffp127"), 0)) == 0x7F7F


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    # silu(1) = e / (1 + e)
    assert oracle.silu(1.0) == pytest.approx(math.e / (1 + math.e), rel=1e-15)
    # odd-part identity: silu(z) - silu(-z) = z, since sigma(z) + sigma(-z) = 1
    for z in [0.3, 1.7, -2.5, 5.0, 11.0]:
        assert oracle.silu(z) - oracle.silu(-z) == pytest.approx(z, rel=1e-14, abs=1e-15)
    # saturation: silu(z) -> z for z >> 0, -> 0 for z << 0
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle.silu(-40.0)) < 1e-15
    assert oracle.silu(-1000.0) == 0.0
    for z in [-3.25, -0.5, 0.125, 2.0, 7.5]:
        exact = silu_decimal(Fraction(z))
        assert oracle.silu(z) == pytest.approx(float(exact), rel=1e-15)


# ----------------------------------------------------------------------------------
# brute force on tiny inputs with exact rationals
# ----------------------------------------------------------------------------------

def brute_force_mlp(x, wgu, wd):
    """Exact evaluation: g, u exact; h = RNE(silu(g) u) with a 60-digit exp; y = RNE(sum h W_down)."""
    T, H = x.shape
    I = wgu.shape[0] // 2
    X = [[bf16_exact(int(b)) for b in row] for row in x]
    G = [[bf16_exact(int(b)) for b in row] for row in wgu]
    D = [[bf16_exact(int(b)) for b in row] for row in wd]
    h = np.zeros((T, I), dtype=np.float64)
    h_tie = np.ones((T, I))
    for t in range(T):
        for j in range(I):
            g = sum(X[t][k] * G[j][k] for k in range(H))
            u = sum(X[t][k] * G[I + j][k] for k in range(H))
            v, tie = round_bf16_exact(silu_decimal(g) * u)
            h[t, j] = float(v)
            h_tie[t, j] = tie
    return h, h_tie, D


@pytest.mark.parametrize("T,H,I,seed", [(1, 1, 1, 0), (2, 3, 2, 1), (3, 8, 4, 2), (4, 5, 6, 3),
                                        (3, 16, 12, 4), (5, 7, 3, 5)])
def test_mlp_matches_exact_brute_force(T, H, I, seed):
    x = W.make_custom(seed, 0, (T, H), 1.5)
    wgu = W.make_custom(seed, 1, (2 * I, H), 1.0)
    wd = W.make_custom(seed, 2, (H, I), 1.0)
    y, yf, h = oracle.mlp_forward(x, wgu, wd)
    hb, h_tie, D = brute_force_mlp(x, wgu, wd)
    hf = f64(h)
    uncertain = h_tie < 1e-9         # exact value sits on a rounding tie: either side is fine
    assert np.array_equal(hf[~uncertain], hb[~uncertain])
    assert uncertain.sum() <= 1
    # y from the oracle's own (already checked) h, summed exactly, rounded exactly
    Hq = [[Fraction(float(v)) for v in row] for row in hf]
    for t in range(T):
        for n in range(H):
            s = sum(Hq[t][j] * D[n][j] for j in range(I))
            v, tie = round_bf16_exact(s)
            assert abs(float(s) - yf[t, n]) <= 1e-13 * max(1.0, abs(float(s)))
            if tie > 1e-9:
                assert oracle.bf16_to_f64(int(y[t, n])) == float(v)


def test_gate_and_up_order_and_operand_orientation():
    # Gate rows come first: swapping gate and up halves must change the result
    # (silu is not symmetric), and the down weight is [H x I] (out x in).
    w = W.TINY_SHARDED
    x = W.make_x(w)
    wgu, wd = W.make_mlp_weights(w)
    y, yf, h = oracle.mlp_forward(x, wgu, wd)
    swapped = np.concatenate([wgu[w.I:], wgu[:w.I]])
    _, yf2, _ = oracle.mlp_forward(x, swapped, wd)
    assert np.abs(yf2 - yf).max() > 1.0
    # library routine for the bilinear part (fp64 BLAS), activation from the definition
    X, G, D = f64(x), f64(wgu), f64(wd)
    gu = X @ G.T
    g, u = gu[:, :w.I], gu[:, w.I:]
    h_ref = g / (1.0 + np.exp(-g)) * u
    assert np.abs(f64(h) - h_ref).max() <= 2.0 ** -8 * np.abs(h_ref).max() + 1e-12
    y_ref = f64(h) @ D.T
    np.testing.assert_allclose(yf, y_ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------------

def test_zero_weights_give_zero():
    T, H, I = 4, 24, 10
    x = W.make_custom(3, 0, (T, H))
    wgu = W.make_custom(3, 1, (2 * I, H))
    wd = W.make_custom(3, 2, (H, I))
    z_gu = np.zeros_like(wgu)
    for args in [(np.zeros_like(x), wgu, wd), (x, z_gu, wd), (x, wgu, np.zeros_like(wd))]:
        y, yf, h = oracle.mlp_forward(*args)
        assert np.all(yf == 0.0)
        assert np.all((y & 0x7FFF) == 0)
    # only gate zero -> silu(0) * u = 0
    g0 = wgu.copy(); g0[:I] = 0
    _, yf, h = oracle.mlp_forward(x, g0, wd)
    assert np.all(yf == 0.0)


def test_one_hot_closed_form():
    # Wg[j,:] = a e_k, Wu[j,:] = b e_m, Wd[:,j] = c e_n  =>  y[t,n] = bf16(bf16(silu(a x_k) b x_m) c)
    T, H, I = 5, 9, 4
    x = W.make_custom(9, 0, (T, H), 2.0)
    wgu = np.zeros((2 * I, H), dtype=np.uint16)
    wd = np.zeros((H, I), dtype=np.uint16)
    j, k, m, n = 2, 3, 7, 5
    a, b, c = 0x3FC0, 0xC040, 0x3F00       # 1.5, -3.0, 0.5
    wgu[j, k] = a
    wgu[I + j, m] = b
    wd[n, j] = c
    y, yf, h = oracle.mlp_forward(x, wgu, wd)
    A, B, C = (oracle.bf16_to_f64(v) for v in (a, b, c))
    for t in range(T):
        xk, xm = oracle.bf16_to_f64(int(x[t, k])), oracle.bf16_to_f64(int(x[t, m]))
        gz = A * xk
        hv = oracle.f64_to_bf16(gz / (1 + math.exp(-gz)) * (B * xm))
        expect = oracle.f64_to_bf16(oracle.bf16_to_f64(hv) * C)
        assert int(y[t, n]) == expect
        others = np.delete(yf[t], n)
        assert np.all(others == 0.0)


# ----------------------------------------------------------------------------------
# the pages' invariant: sum of per-shard partials == replicated output, per token
# ----------------------------------------------------------------------------------

def test_golden_tiny_case_shape():
    g = read_golden("tiny_sharded_case.txt")
    w = W.TINY_SHARDED
    assert int(g["tp_size"][0]) == w.tp
    assert int(g["hidden"][0]) == w.H
    assert int(g["intermediate"][0]) == w.I
    assert int(g["tokens_per_rank"][0]) * w.tp == w.T


@pytest.mark.parametrize("dtype", [oracle.F32, oracle.BF16])
def test_shard_partials_sum_to_replicated_tiny(dtype):
    w = W.TINY_SHARDED
    x = W.make_x(w)
    wgu, wd = W.make_mlp_weights(w)
    y, yf, _ = oracle.mlp_forward(x, wgu, wd)
    parts = [oracle.shard_partial(x, wgu, wd, w.tp, r, dtype) for r in range(w.tp)]
    s64 = sum(p[0] for p in parts)
    # fp64 partials reassociate the intermediate sum only
    np.testing.assert_allclose(s64, yf, rtol=1e-13, atol=1e-12)
    reduced = oracle.shard_sum(np.stack([p[1] for p in parts]), dtype)
    # error bound of "round each partial, sum, round once": with unit roundoff u_p of the
    # partial dtype, |reduced - exact| <= u_p * sum_r |P_r| + 2^-8 * |reduced| (+ fp64 noise)
    u_p = 2.0 ** -8 if dtype == oracle.BF16 else 2.0 ** -24
    abs_sum = sum(np.abs(p[0]) for p in parts)
    g = read_golden("tiny_sharded_case.txt")
    tpr = int(g["tokens_per_rank"][0])
    for r in range(w.tp):
        sl = slice(r * tpr, (r + 1) * tpr)
        mine = f64(reduced[sl])
        bound = u_p * abs_sum[sl] + 2.0 ** -8 * np.abs(mine) + 1e-12
        assert np.all(np.abs(mine - yf[sl]) <= bound)
        if dtype == oracle.F32:
            # fp32 partials keep the page's 1e-5 closeness before the final bf16 rounding
            s32 = sum(p[1].astype(np.float64) for p in parts)
            np.testing.assert_allclose(s32[sl], yf[sl], rtol=float(g["rtol"][0]), atol=float(g["atol"][0]))


def test_shard_partials_sum_to_replicated_mid_shape():
    T, H, I, tp = 6, 64, 48, 8
    x = W.make_custom(21, 0, (T, H))
    wgu = W.make_custom(21, 1, (2 * I, H), 1 / 8)
    wd = W.make_custom(21, 2, (H, I), 1 / 7)
    _, yf, _ = oracle.mlp_forward(x, wgu, wd)
    s = sum(oracle.shard_partial(x, wgu, wd, tp, r)[0] for r in range(tp))
    np.testing.assert_allclose(s, yf, rtol=1e-12, atol=1e-13)


def test_shard_sum_exact_small():
    rng = np.random.default_rng(5)
    p = W.f32_to_bf16_bits(rng.standard_normal((3, 4, 5)).astype(np.float32))
    out = oracle.shard_sum(p, oracle.BF16)
    for t in range(4):
        for n in range(5):
            s = sum(bf16_exact(int(p[r, t, n])) for r in range(3))
            v, tie = round_bf16_exact(s)
            if tie > 1e-12:
                assert oracle.bf16_to_f64(int(out[t, n])) == float(v)


def test_shard_geometry_rejected():
    w = W.TINY_SHARDED
    x = W.make_x(w)
    wgu, wd = W.make_mlp_weights(w)
    with pytest.raises(ValueError):
        oracle.shard_partial(x, wgu, wd, 5, 0)      # 12 % 5 != 0 (cf. 6144 % 5 != 0)
    with pytest.raises(ValueError):
        oracle.shard_partial(x, wgu, wd, 4, 4)      # rank out of range
    with pytest.raises(ValueError):
        oracle.rank_major_to_logical(1536, 576, 5)  # merged sizes not divisible


# ----------------------------------------------------------------------------------
# partials of a group of shards summed before any rounding (the fused reduce)
# ----------------------------------------------------------------------------------

@pytest.mark.parametrize("T,H,I,tp,rf,rc,seed", [(2, 5, 4, 2, 0, 2, 11), (3, 6, 6, 3, 1, 2, 12),
                                                 (2, 8, 8, 4, 1, 2, 13), (3, 4, 6, 3, 2, 1, 14)])
def test_shard_group_sum_matches_exact_brute_force(T, H, I, tp, rf, rc, seed):
    # exact rationals: h rounded exactly, then the sum over the group's intermediate
    # columns [rf*s, (rf+rc)*s) only, rounded once (bf16) or to fp32
    x = W.make_custom(seed, 0, (T, H), 1.5)
    wgu = W.make_custom(seed, 1, (2 * I, H), 1.0)
    wd = W.make_custom(seed, 2, (H, I), 1.0)
    hb, h_tie, D = brute_force_mlp(x, wgu, wd)
    assert (h_tie < 1e-9).sum() == 0
    s = I // tp
    j0, j1 = rf * s, (rf + rc) * s
    sf, sb = oracle.shard_group_sum(x, wgu, wd, tp, rf, rc, oracle.BF16)
    _, s32 = oracle.shard_group_sum(x, wgu, wd, tp, rf, rc, oracle.F32)
    for t in range(T):
        for n in range(H):
            exact = sum(Fraction(float(hb[t, j])) * D[n][j] for j in range(j0, j1))
            assert abs(float(exact) - sf[t, n]) <= 1e-13 * max(1.0, abs(float(exact)))
            v, tie = round_bf16_exact(exact)
            if tie > 1e-9:
                assert oracle.bf16_to_f64(int(sb[t, n])) == float(v)
            assert s32[t, n] == np.float32(float(exact))


def test_shard_group_sum_of_all_shards_is_the_replicated_layer():
    # the pages' invariant: summing every shard's partial gives the replicated output
    T, H, I, tp = 6, 64, 48, 8
    x = W.make_custom(22, 0, (T, H))
    wgu = W.make_custom(22, 1, (2 * I, H), 1 / 8)
    wd = W.make_custom(22, 2, (H, I), 1 / 7)
    y, yf, _ = oracle.mlp_forward(x, wgu, wd)
    sf, sb = oracle.shard_group_sum(x, wgu, wd, tp, 0, tp, oracle.BF16)
    np.testing.assert_allclose(sf, yf, rtol=1e-12, atol=1e-13)
    differ = sb != y
    # only where the two fp64 sums straddle a bf16 rounding boundary
    for t, n in zip(*np.nonzero(differ)):
        _, tie = round_bf16_exact(Fraction(float(yf[t, n])))
        assert tie < 1e-9


def test_shard_group_sum_tiny_case_within_page_tolerance():
    # the page's equivalence case at fp32: each rank's token rows of the summed
    # partials are within the printed 1e-5 of the replicated layer
    w = W.TINY_SHARDED
    x = W.make_x(w)
    wgu, wd = W.make_mlp_weights(w)
    _, yf, _ = oracle.mlp_forward(x, wgu, wd)
    _, s32 = oracle.shard_group_sum(x, wgu, wd, w.tp, 0, w.tp, oracle.F32)
    g = read_golden("tiny_sharded_case.txt")
    tpr = int(g["tokens_per_rank"][0])
    for r in range(w.tp):
        sl = slice(r * tpr, (r + 1) * tpr)
        np.testing.assert_allclose(s32[sl].astype(np.float64), yf[sl], rtol=float(g["rtol"][0]),
                                   atol=float(g["atol"][0]))


def test_shard_group_geometry_rejected():
    w = W.TINY_SHARDED
    x = W.make_x(w)
    wgu, wd = W.make_mlp_weights(w)
    for tp, rf, rc in [(5, 0, 5), (4, 3, 2), (4, -1, 2), (4, 0, 0)]:
        with pytest.raises(ValueError):
            oracle.shard_group_sum(x, wgu, wd, tp, rf, rc)


def test_feature_slice_concatenation_design_fails():
    """The rejected earlier design (output-dim sharding + all-gather of feature slices)
    under disjoint token shards must NOT match; with every rank holding the same tokens
    it would have passed.  The mistake is planted in a CPU composition of oracle steps."""
    w = W.TINY_SHARDED
    x = W.make_x(w)
    wgu, wd = W.make_mlp_weights(w)
    y, yf, _ = oracle.mlp_forward(x, wgu, wd)
    tp, tpr, s = w.tp, w.T // w.tp, w.I // w.tp

    def broken(x_tokens_of_rank):
        # rank r computes h for ITS tokens over ITS intermediate slice only, then the
        # feature slices are concatenated as if they belonged to the same tokens.
        h_mixed = np.zeros((tpr, w.I), dtype=np.float64)
        for r in range(tp):
            h_r = oracle.swiglu_hidden(x_tokens_of_rank(r), wgu, w.I, r * s, (r + 1) * s)
            h_mixed[:, r * s:(r + 1) * s] = f64(h_r)
        return h_mixed @ f64(wd).T

    disjoint = broken(lambda r: x[r * tpr:(r + 1) * tpr])
    tol_ok = np.abs(disjoint - f64(y[0:tpr])) <= 0.02 + 0.02 * np.abs(f64(y[0:tpr]))
    assert not tol_ok.all()
    # same tokens on every rank: the broken design is indistinguishable
    same = broken(lambda r: x[0:tpr])
    np.testing.assert_allclose(same, yf[0:tpr], rtol=2e-2, atol=2e-2)


# ----------------------------------------------------------------------------------
# merged q_a / kv_a projection and the rank-major -> logical permutation
# ----------------------------------------------------------------------------------

def simulate_gather(logical, q_dim, kv_dim, tp):
    """Each rank's local output is [its q_a columns | its kv_a columns]; the gather
    concatenates the ranks in rank order."""
    qs, ks = q_dim // tp, kv_dim // tp
    cols = []
    for r in range(tp):
        cols.append(logical[:, r * qs:(r + 1) * qs])
        cols.append(logical[:, q_dim + r * ks:q_dim + (r + 1) * ks])
    return np.concatenate(cols, axis=1)


@pytest.mark.parametrize("q,kv,tp", [(1536, 576, 16), (1536, 576, 8), (1536, 576, 1), (12, 8, 4), (6, 3, 3)])
def test_rank_major_map_matches_simulated_gather(q, kv, tp):
    m = oracle.rank_major_to_logical(q, kv, tp)
    ident = np.arange(q + kv, dtype=np.int64)[None, :]
    assert np.array_equal(simulate_gather(ident, q, kv, tp)[0], m)
    assert np.array_equal(np.sort(m), np.arange(q + kv))
    if tp == 16 and q == 1536:
        # rank 0 holds q_a rows 0..95 then kv_a rows 1536..1571 (132 columns per rank)
        assert list(m[:3]) == [0, 1, 2] and m[95] == 95 and m[96] == 1536 and m[131] == 1571
        assert m[132] == 96 and m[-1] == 2111


def test_merged_proj_exact_integer_permutation():
    # Integer-valued x (|x| <= 256, exact in bf16) and one-hot rows W[c] = e_{c mod H} * v_c:
    # every output column is an exact integer known in advance, so the rank-major buffer
    # is checked bit-exactly through the projection.
    q, kv, tp, H, T = 48, 16, 4, 32, 5
    C = q + kv
    xi = (np.arange(T * H).reshape(T, H) % 97) - 48
    x = W.f32_to_bf16_bits(xi.astype(np.float32))
    w = np.zeros((C, H), dtype=np.uint16)
    scale = np.array([1.0, 2.0, -1.0, 0.5], dtype=np.float32)
    for c in range(C):
        w[c, c % H] = W.f32_to_bf16_bits(np.float32([scale[c % 4]]))[0]
    lo, rm, f = oracle.merged_proj(x, w, q, kv, tp)
    expect = np.array([[xi[t, c % H] * scale[c % 4] for c in range(C)] for t in range(T)])
    assert np.array_equal(f, expect)
    assert np.array_equal(f64(lo), expect)
    assert np.array_equal(rm, simulate_gather(lo, q, kv, tp))
    assert np.array_equal(oracle.reorder(rm, q, kv, tp), lo)


def test_merged_proj_matches_blas_and_reorder_roundtrip():
    q, kv, tp, H, T = 96, 36, 4, 40, 7
    x = W.make_custom(31, 0, (T, H))
    w = W.make_custom(31, 4, (q + kv, H), 1 / math.sqrt(H))
    lo, rm, f = oracle.merged_proj(x, w, q, kv, tp)
    np.testing.assert_allclose(f, f64(x) @ f64(w).T, rtol=1e-12, atol=1e-13)
    assert np.array_equal(rm, simulate_gather(lo, q, kv, tp))
    assert np.array_equal(oracle.reorder(rm, q, kv, tp), lo)
    rows = np.array([6, 0, 3])
    lo2, rm2, _ = oracle.merged_proj(x, w, q, kv, tp, rows=rows)
    assert np.array_equal(lo2, lo[rows]) and np.array_equal(rm2, rm[rows])


# ----------------------------------------------------------------------------------
# byte model printed on the pages
# ----------------------------------------------------------------------------------

def test_byte_model_matches_pages():
    g = read_golden("byte_model.txt")
    H, I = int(g["hidden_size"][0]), int(g["shared_intermediate"][0])
    assert (H, I) == (W.DECODE_T64.H, W.DECODE_T64.I) == (W.PREFILL_T8192.H, W.PREFILL_T8192.I)
    gate_up = 2 * I * H * 2
    down = H * I * 2
    assert round(gate_up / 1e6, 1) == float(g["gate_up_bytes"][0])          # 176.2 MB
    assert round(down / 1e6, 1) == float(g["down_bytes"][0])                # 88.1 MB
    assert round((gate_up + down) / 1e6, 1) == float(g["layer_bytes"][0])   # 264.2 MB
    layers = int(g["moe_layers"][0])
    assert round(layers * (gate_up + down) / 2**30, 1) == float(g["all_layers_bytes"][0])
    # the profiled gate_up kernel time corresponds to the ~5.9 TB/s quoted for the pair
    tbps = gate_up / (float(g["gate_up_kernel_us"][0]) * 1e-6) / 1e12
    assert abs(tbps - float(g["gemm_pair_tbps"][0])) < 0.1
    rows, cols = int(g["mla_rows"][0]), int(g["mla_cols"][0])
    assert rows == W.MLA_MERGED.q_dim + W.MLA_MERGED.kv_dim and cols == W.MLA_MERGED.H
    tp, nl = int(g["mla_tp"][0]), int(g["mla_layers"][0])
    assert tp == W.MLA_MERGED.tp
    saving = nl * rows * cols * 2 * (tp - 1) / tp / 2**30
    assert round(saving, 3) == float(g["mla_saving_gib"][0])


# ----------------------------------------------------------------------------------
# row sampling, threading determinism, generator
# ----------------------------------------------------------------------------------

def test_row_subset_and_thread_count_do_not_change_bits():
    T, H, I = 9, 72, 40
    x = W.make_custom(41, 0, (T, H))
    wgu = W.make_custom(41, 1, (2 * I, H), 1 / math.sqrt(H))
    wd = W.make_custom(41, 2, (H, I), 1 / math.sqrt(I))
    y1, yf1, h1 = oracle.mlp_forward(x, wgu, wd, nthreads=1)
    y8, yf8, h8 = oracle.mlp_forward(x, wgu, wd, nthreads=8)
    assert np.array_equal(yf1, yf8) and np.array_equal(h1, h8)
    rows = np.array([8, 2, 2, 5])
    ys, yfs, hs = oracle.mlp_forward(x, wgu, wd, rows=rows, nthreads=3)
    assert np.array_equal(yfs, yf1[rows]) and np.array_equal(hs, h1[rows])


def test_generator_is_counter_based_and_gaussian():
    a = W.normal_f64(5, 2, 1000)
    b = W.normal_f64(5, 2, 1001)
    assert np.array_equal(a, b[:1000])
    c = W.normal_f64(5, 2, 1 << 21, chunk=1 << 16)
    d = W.normal_f64(5, 2, 1 << 21, chunk=1 << 20)
    assert np.array_equal(c, d)
    assert abs(c.mean()) < 0.005 and abs(c.std() - 1) < 0.005
    assert not np.array_equal(W.normal_f64(5, 3, 100), a[:100])
    w = W.gaussian_bf16(1, 1, (64, 7168), 1 / math.sqrt(7168))
    s = W.bf16_bits_to_f32(w).std()
    assert abs(s - 1 / math.sqrt(7168)) < 2e-4
