"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test names what fixes the expected value: a library conversion, an
exhaustive sweep, exact rational arithmetic, a closed form, a hand-worked
example, or a planted mistake that must be caught.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))
ALL16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


# ---------------------------------------------------------------- formats
def test_fp16_decode_matches_numpy_all_patterns():
    ours = oracle.fp16_to_f64(ALL16)
    ref = ALL16.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros are distinct patterns with the right sign
    assert np.signbit(oracle.fp16_to_f64(np.uint16(0x8000)))
    assert not np.signbit(oracle.fp16_to_f64(np.uint16(0x0000)))


def test_bf16_decode_matches_torch_all_patterns():
    ours = oracle.bf16_to_f64(ALL16)
    ref = torch.from_numpy(ALL16.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_fp16_rounding_is_nearest_even_at_every_midpoint():
    # every pair of adjacent positive finite FP16 values, including subnormals
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)
    a = oracle.fp16_to_f64(lo)
    b = oracle.fp16_to_f64(lo + 1)
    mid = (a + b) / 2                       # exact in fp64
    r = oracle.f64_to_fp16_bits(mid)
    even = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(r, even)
    # just below / above the midpoint goes to the nearer value
    below = np.nextafter(mid, -np.inf)
    above = np.nextafter(mid, np.inf)
    assert np.array_equal(oracle.f64_to_fp16_bits(below), lo)
    assert np.array_equal(oracle.f64_to_fp16_bits(above), lo + 1)
    # overflow threshold: 65504 + half an ulp (16) rounds to inf (ties to even)
    assert oracle.f64_to_fp16_bits(65519.99) == 0x7BFF
    assert oracle.f64_to_fp16_bits(65520.0) == 0x7C00
    # negative values mirror positive ones
    assert np.array_equal(oracle.f64_to_fp16_bits(-mid), even | 0x8000)


# ---------------------------------------------------------------- encoder
def _nearest_fp16_exact(q: Fraction) -> int:
    """Nearest FP16 pattern to a positive rational, ties to even, by search."""
    approx = int(np.float64(float(q)).astype(np.float16).view(np.uint16))
    best = None
    for p in range(max(0, approx - 2), min(0x7C00, approx + 3)):
        v = Fraction(float(oracle.fp16_to_f64(np.uint16(p))))
        d = abs(v - q)
        key = (d, p % 2)
        if best is None or key < best[0]:
            best = (key, p)
    return best[1]


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_rtn_scale_is_exact_nearest_fp16(bits):
    rng = synth.generator(0, 100, bits)
    w = synth.gauss_weights(rng, 64, 64 * 8)
    # add groups with tiny and subnormal-scale magnitudes
    w[0, :64] *= np.float32(1e-5)
    w[1, :64] *= np.float32(1e-7)
    s = oracle.rtn_scales(w, oracle.QMAX[bits])
    a = np.abs(w.reshape(64, 8, 64)).max(axis=2)
    for i in range(64):
        for g in range(8):
            q = Fraction(float(a[i, g])) / oracle.QMAX[bits]
            assert s[i, g] == _nearest_fp16_exact(q), (i, g)


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_rtn_code_is_brute_force_nearest(bits):
    rng = synth.generator(0, 101, bits)
    n, k = 8, 256
    w = synth.gauss_weights(rng, n, k)
    codes, sb = oracle.rtn_encode(w, bits)
    lo, hi = oracle.code_range(bits)
    s = oracle.fp16_to_f64(sb)
    for i in range(n):
        for j in range(k):
            sv = Fraction(float(s[i, j // 64]))
            wv = Fraction(float(w[i, j]))
            best = min(range(lo, hi + 1), key=lambda c: (abs(wv - sv * c), c % 2))
            assert codes[i, j] == best, (i, j)


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_rtn_invariants(bits):
    rng = synth.generator(0, 102, bits)
    w = synth.gauss_weights(rng, 64, 1024)
    codes, sb = oracle.rtn_encode(w, bits)
    qmax = oracle.QMAX[bits]
    assert codes.min() >= -qmax and codes.max() <= qmax   # positive scale: no -qmax-1
    s = np.repeat(oracle.fp16_to_f64(sb), 64, axis=1)
    err = np.abs(w.astype(np.float64) - s * codes)
    clamped = np.abs(codes) == qmax
    assert np.all(err[~clamped] <= s[~clamped] / 2)
    # the group maximum lands on +-qmax
    amax_idx = np.abs(w.reshape(64, 16, 64)).argmax(axis=2)
    c_at = np.take_along_axis(codes.reshape(64, 16, 64), amax_idx[..., None], axis=2)
    assert np.all(np.abs(c_at) == qmax)


def test_rtn_zero_group_and_overflow():
    w = np.zeros((1, 128), dtype=np.float32)
    w[0, 64:] = 1.0
    codes, sb = oracle.rtn_encode(w, 4)
    assert sb[0, 0] == 0 and np.all(codes[0, :64] == 0)
    assert np.all(codes[0, 64:] == 7)
    big = np.full((1, 64), 7.0 * 65520.0, dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.rtn_encode(big, 4)


def test_worked_example_golden():
    with open(os.path.join(HERE, "golden", "rtn_worked_example.json")) as f:
        g = json.load(f)
    w = np.zeros((1, 64), dtype=np.float32)
    for k, v in g["weights_fp32_nonzero"].items():
        w[0, int(k)] = v
    for case in g["cases"]:
        codes, sb = oracle.rtn_encode(w, case["bits"])
        assert int(sb[0, 0]) == int(case["scale_bits"], 16)
        assert oracle.fp16_to_f64(sb[0, 0]) == case["scale"]
        assert list(codes[0, :3]) == case["codes_first3"]
        assert np.all(codes[0, 3:] == 0)
    p = g["product"]
    codes, sb = oracle.rtn_encode(w, p["bits"])
    x = np.zeros((1, 64), dtype=np.float32)
    for k, v in p["x_nonzero"].items():
        x[0, int(k)] = v
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)   # exact: these are bf16 values
    y, e = oracle.gemv(codes, sb, xb)
    assert y[0, 0] == p["y"] and e[0, 0] == p["E"]


# ---------------------------------------------------------------- dequant
def test_dequant_exact_all_fp16_times_all_codes():
    finite = ALL16[(ALL16 & 0x7C00) != 0x7C00]
    s = oracle.fp16_to_f64(finite)[:, None]
    c = np.arange(-128, 128, dtype=np.float64)[None, :]       # every code of every width (4..8 bits)
    p = s * c
    # exact in fp32: casting to fp32 and back loses nothing (11 x 8 significant bits)
    assert np.array_equal(p.astype(np.float32).astype(np.float64), p)
    # and the oracle's dequant gives exactly these products
    codes = np.tile(np.arange(-128, 128, dtype=np.int16).astype(np.int8), (finite.size, 1))
    w = oracle.dequant(codes, np.repeat(finite[:, None], 4, axis=1))   # 4 groups, one scale per row
    assert np.array_equal(w, p)
    # signed zero: -0 scale times positive code is -0
    assert np.signbit(oracle.dequant(np.full((1, 64), 3, np.int8), np.array([[0x8000]], np.uint16)))[0, 0]


def test_dequant_matches_rationals_sample():
    rng = synth.generator(0, 103)
    sb = rng.integers(0, 0x7C00, size=(4, 4), dtype=np.uint16) | (rng.integers(0, 2, (4, 4), dtype=np.uint16) << 15)
    codes = synth.uniform_codes(rng, 4, 256, 6)
    w = oracle.dequant(codes, sb)
    for i in range(4):
        for j in range(0, 256, 7):
            sv = Fraction(float(oracle.fp16_to_f64(sb[i, j // 64])))
            assert Fraction(float(w[i, j])) == sv * int(codes[i, j])


# ---------------------------------------------------------------- product
@pytest.mark.parametrize("bits,k,n,t", [(4, 64, 3, 1), (5, 128, 4, 2), (6, 256, 8, 4), (6, 192, 5, 3),
                                         (8, 128, 4, 2)])
def test_gemv_against_exact_rationals(bits, k, n, t):
    rng = synth.generator(0, 104, bits, k)
    codes = synth.uniform_codes(rng, n, k, bits)
    sb = oracle.rtn_scales(synth.gauss_weights(rng, n, k), oracle.QMAX[bits])
    sb = sb ^ (synth.sign_flips(rng, n, k // 64).astype(np.uint16) << 15)
    xb = synth.gauss_x_bf16(rng, t, k, outliers=synth.outlier_channels(rng, k, 0.05))
    y, e = oracle.gemv(codes, sb, xb)
    s = oracle.fp16_to_f64(sb)
    xv = oracle.bf16_to_f64(xb)
    for ti in range(t):
        for ni in range(n):
            exact = sum(Fraction(float(s[ni, kk // 64])) * int(codes[ni, kk]) * Fraction(float(xv[ti, kk]))
                        for kk in range(k))
            eabs = sum(abs(Fraction(float(s[ni, kk // 64])) * int(codes[ni, kk]) * Fraction(float(xv[ti, kk])))
                       for kk in range(k))
            # fp64 summation error bound: K * 2^-53 * sum|terms|
            assert abs(Fraction(float(y[ti, ni])) - exact) <= Fraction(k, 2 ** 53) * eabs
            assert abs(Fraction(float(e[ti, ni])) - eabs) <= Fraction(k, 2 ** 53) * eabs


def test_special_cases():
    rng = synth.generator(0, 105)
    n, k = 6, 256
    codes = synth.uniform_codes(rng, n, k, 5)
    sb = oracle.rtn_scales(synth.gauss_weights(rng, n, k), 15)
    w = oracle.dequant(codes, sb)
    # one-hot x reproduces a column of w exactly
    for kk in (0, 63, 64, 200):
        x = np.zeros((1, k), np.uint16)
        x[0, kk] = 0x3F80           # bf16 1.0
        y, _ = oracle.gemv(codes, sb, x)
        assert np.array_equal(y[0], w[:, kk])
    # zero codes give zero
    y, e = oracle.gemv(np.zeros_like(codes), sb, synth.gauss_x_bf16(rng, 2, k))
    assert np.all(y == 0) and np.all(e == 0)
    # x = 1 on one group gives s * sum(c) exactly
    x = np.zeros((1, k), np.uint16)
    x[0, 64:128] = 0x3F80
    y, _ = oracle.gemv(codes, sb, x)
    ref = oracle.fp16_to_f64(sb[:, 1]) * codes[:, 64:128].astype(np.int64).sum(axis=1)
    assert np.array_equal(y[0], ref)
    # negating every scale negates the output exactly
    xb = synth.gauss_x_bf16(rng, 3, k)
    y1, e1 = oracle.gemv(codes, sb, xb)
    y2, e2 = oracle.gemv(codes, sb ^ np.uint16(0x8000), xb)
    assert np.array_equal(y1, -y2) and np.array_equal(e1, e2)


# ---------------------------------------------------------------- tolerance sensitivity
def _planted(codes, sb, xb, kind):
    """The oracle's product with one deliberate mistake."""
    c = codes.astype(np.float64)
    n, k = codes.shape
    s = oracle.fp16_to_f64(sb)
    if kind == "group_off_by_one":
        idx = np.minimum((np.arange(k) + 1) // 64, k // 64 - 1)
        w = s[:, idx] * c
    elif kind == "scale_sign_dropped":
        w = np.repeat(np.abs(s), 64, axis=1) * c
    elif kind == "code_bias":
        w = np.repeat(s, 64, axis=1) * (c + 1)
    elif kind == "k_pairs_swapped":
        perm = np.arange(k).reshape(-1, 2)[:, ::-1].reshape(-1)
        w = np.repeat(s, 64, axis=1) * c[:, perm]
    elif kind == "tokens_swapped":
        w = np.repeat(s, 64, axis=1) * c
        return oracle.bf16_to_f64(xb[::-1]) @ w.T
    elif kind == "high_plane_factor":
        # an 8-bit code taken as hi * 16 + lo with the high nibble weighed 15
        u = codes.astype(np.int64) + 128
        w = np.repeat(s, 64, axis=1) * (15 * ((u >> 4) - 8) + (u & 15))
    elif kind == "k_order_of_other_layout":
        # x read in the K order k = 16j + 2r + 8h + c instead of 16r + 4j + 2h + c
        perm = np.empty(64, dtype=np.int64)
        for j in range(4):
            for r in range(4):
                for h in range(2):
                    for cc in range(2):
                        perm[16 * r + 4 * j + 2 * h + cc] = 16 * j + 2 * r + 8 * h + cc
        full = (np.arange(k) // 64) * 64 + perm[np.arange(k) % 64]
        w = np.repeat(s, 64, axis=1) * c[:, full]
    else:
        raise ValueError(kind)
    return oracle.bf16_to_f64(xb) @ w.T


@pytest.mark.parametrize("bits,kind", [(5, "group_off_by_one"), (5, "scale_sign_dropped"),
                                       (5, "code_bias"), (5, "k_pairs_swapped"),
                                       (5, "tokens_swapped"), (8, "high_plane_factor"),
                                       (5, "k_order_of_other_layout"),
                                       (8, "k_order_of_other_layout")])
def test_tolerance_catches_planted_mistakes(bits, kind):
    rng = synth.generator(0, 106, bits)
    n, k, t = 32, 1024, 2
    codes = synth.uniform_codes(rng, n, k, bits)
    sb = oracle.rtn_scales(synth.gauss_weights(rng, n, k), oracle.QMAX[bits])
    sb = sb ^ (synth.sign_flips(rng, n, k // 64).astype(np.uint16) << 15)
    xb = synth.gauss_x_bf16(rng, t, k, outliers=synth.outlier_channels(rng, k))
    y, e = oracle.gemv(codes, sb, xb)
    bad = _planted(codes, sb, xb, kind)
    assert oracle.tolerance_ok(y.astype(np.float32), y, e)
    assert not oracle.tolerance_ok(bad, y, e)


# ---------------------------------------------------------------- verify-head reductions
def test_head_logsumexp_closed_forms():
    # sum_{k=1..N} exp(log k) = N (N + 1) / 2
    for n in (1, 2, 7, 1000, 248320):
        y = np.log(np.arange(1, n + 1, dtype=np.float64))[None, :]
        _, _, lse = oracle.head_reduce(y)
        assert abs(lse[0] - np.log(n * (n + 1) / 2)) <= 1e-12 * max(1.0, np.log(n * n))
    # N equal values v: v + log N; one value far above the rest: that value
    y = np.full((1, 4096), -3.25)
    assert abs(oracle.head_reduce(y)[2][0] - (-3.25 + np.log(4096))) <= 1e-13
    y = np.array([[0.0, -1000.0, -2000.0, -745.0]])
    assert oracle.head_reduce(y)[2][0] == 0.0


def test_head_logsumexp_large_logits_do_not_overflow():
    # a naive sum of exp would overflow fp64 here
    y = np.array([[1000.0, 1000.0, 999.0]])
    _, m, lse = oracle.head_reduce(y)
    assert m[0] == 1000.0
    assert abs(lse[0] - (1000.0 + np.log(2.0 + np.exp(-1.0)))) <= 1e-12


def test_head_infinite_logits():
    """log(sum exp y) is +inf as soon as one logit is +inf (also with several),
    and -inf logits contribute exp(-inf) = 0."""
    inf = np.inf
    y = np.array([[1.0, inf, 3.0, inf], [-inf, 2.0, -inf, 2.0], [inf, inf, inf, inf]])
    am, m, lse = oracle.head_reduce(y)
    assert am.tolist() == [1, 1, 0]
    assert m.tolist() == [inf, 2.0, inf]
    assert lse[0] == inf and lse[2] == inf
    assert abs(lse[1] - (2.0 + np.log(2.0))) <= 1e-15


def test_head_argmax_ties_take_the_first_index():
    y = np.array([[1.0, 5.0, 2.0, 5.0, 5.0], [7.0, 7.0, 7.0, 7.0, 7.0], [-1.0, -2.0, -1.0, -3.0, -1.5]])
    am, m, _ = oracle.head_reduce(y)
    assert am.tolist() == [1, 0, 0]
    assert m.tolist() == [5.0, 7.0, -1.0]


def test_head_rows_are_independent_tokens():
    rng = np.random.default_rng(5)
    y = rng.standard_normal((6, 333))
    am, m, lse = oracle.head_reduce(y)
    for t in range(6):
        a1, m1, l1 = oracle.head_reduce(y[t:t + 1])
        assert am[t] == a1[0] and m[t] == m1[0] and lse[t] == l1[0]
    # shift invariance: lse(y + c) = lse(y) + c, argmax unchanged
    am2, _, lse2 = oracle.head_reduce(y + 123.5)
    assert np.array_equal(am, am2)
    assert np.all(np.abs(lse2 - (lse + 123.5)) <= 1e-12 * np.abs(lse2))


def test_head_topk_worked_example():
    # by hand: values 3 (rows 1, 2), 2 (row 5), 1 (row 0), +0 (row 4), -0 (row 3)
    y = np.array([[1.0, 3.0, 3.0, -0.0, 0.0, 2.0]])
    idx, val = oracle.head_topk(y, 8)
    assert idx.tolist() == [[1, 2, 5, 0, 4, 3, -1, -1]]
    assert val[0, :6].tolist() == [3.0, 3.0, 2.0, 1.0, 0.0, -0.0]
    assert not np.signbit(val[0, 4]) and np.signbit(val[0, 5])
    assert np.all(np.isneginf(val[0, 6:]))


def test_head_topk_against_sorting_and_argmax():
    rng = np.random.default_rng(9)
    y = rng.standard_normal((5, 1000)).astype(np.float32)
    y[2, 100:110] = y[2].max() + 1                         # a ten-way tie at the top
    for k in (1, 7, 32):
        idx, val = oracle.head_topk(y, k)
        # the values are the k largest (a library sort, no index logic)
        assert np.array_equal(val, -np.sort(-y, axis=1)[:, :k])
        assert np.array_equal(np.take_along_axis(y, idx, axis=1), val)
        assert len({tuple(r) for r in idx}) == 5 and all(len(set(r)) == k for r in idx)
    am, _, _ = oracle.head_reduce(y)
    assert np.array_equal(oracle.head_topk(y, 1)[0][:, 0], am)
    assert oracle.head_topk(y, 12)[0][2, :10].tolist() == list(range(100, 110))


def test_head_topk_selection_property_brute_force():
    # every chosen row ranks above every row left out, under (value, then +0
    # over -0, then smaller index), checked pair by pair on small rows
    rng = np.random.default_rng(10)
    for _ in range(50):
        n = int(rng.integers(1, 12))
        y = rng.integers(-3, 4, size=(1, n)).astype(np.float64)
        y[0, rng.random(n) < 0.2] = -0.0
        k = int(rng.integers(1, 14))
        idx, val = oracle.head_topk(y, k)
        chosen = [int(i) for i in idx[0] if i >= 0]
        assert len(chosen) == min(k, n)

        def above(a, b):
            if y[0, a] != y[0, b]:
                return y[0, a] > y[0, b]
            if np.signbit(y[0, a]) != np.signbit(y[0, b]):
                return not np.signbit(y[0, a])
            return a < b
        for p in range(len(chosen) - 1):
            assert above(chosen[p], chosen[p + 1])
        for a in chosen:
            for b in set(range(n)) - set(chosen):
                assert above(a, b)


# ---------------------------------------------------------------- searched encoder
def _exact_group(values, step_bits):
    """One 64-weight row group w = step * values (values integers), step an FP16
    bit pattern; returns fp32 [1, 64]."""
    step = float(oracle.fp16_to_f64(np.array([step_bits], np.uint16))[0])
    return (np.asarray(values, np.float64) * step).astype(np.float32)[None, :]


def test_search_never_worse_than_rtn():
    rng = synth.generator(0, 900)
    for bits in (4, 5, 6):
        w = synth.gauss_weights(rng, 24, 512)
        w[3, 64:128] *= np.float32(50.0)          # a group with one large channel
        q = synth.imatrix(rng, 512)
        for imp in (None, q):
            c, s = oracle.search_encode(w, bits, imp)
            cr, sr = oracle.rtn_encode(w, bits)
            e = oracle.weighted_error(w, c, s, imp)
            er = oracle.weighted_error(w, cr, sr, imp)
            assert np.all(e <= er * (1 + 1e-12)), bits
            lo, hi = oracle.code_range(bits)
            assert c.min() >= lo and c.max() <= hi


def test_search_picks_a_negative_scale_when_only_it_is_exact():
    # values -7..8: representable as step * c with c in [-8, 7] only if the
    # scale is -step (the +8 needs code -8); the largest value is 8 steps, so
    # the first candidate magnitude h_0 = fp16(a / 8) is the step itself.
    vals = (np.arange(64) % 16) - 7                        # -7 .. 8
    w = _exact_group(vals, 0x2000)                           # step 2^-7
    c, s = oracle.search_encode(w, 4)
    assert s[0, 0] == 0xA000                                 # -2^-7: candidate 1
    assert np.array_equal(c[0], -vals)
    assert oracle.weighted_error(w, c, s)[0, 0] == 0.0
    # -8 .. 7: the positive candidate 0 is exact
    vals = (np.arange(64) % 16) - 8
    w = _exact_group(vals, 0x2000)
    c, s = oracle.search_encode(w, 4)
    assert s[0, 0] == 0x2000 and np.array_equal(c[0], vals)


def _exact_candidates(a: float, qmax: int) -> list[int]:
    """The 50 candidate scale patterns of the searched encoder's reading,
    computed here in exact rational arithmetic (nearest FP16 by search, ties
    to even): +h_i, -h_i for h_i = fp16(12 a / (12 (qmax + 1) - i))."""
    out = []
    for i in range(oracle.SEARCH_STEPS):
        q = Fraction(12) * Fraction(float(a)) / (12 * (qmax + 1) - i)
        h = 0 if q == 0 else _nearest_fp16_exact(q)
        out += [h, h | 0x8000]
    return out


def test_search_candidates_worked_example():
    """The hand-worked candidate lists of tests/golden (two group maxima)."""
    with open(os.path.join(HERE, "golden", "search_candidates_worked_example.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        a, qmax = float(case["absmax"]), case["qmax"]
        assert qmax == oracle.QMAX[case["bits"]]
        want = []
        for i, den, m, plus, minus in case["candidates"]:
            assert den == 12 * (qmax + 1) - i
            want += [int(plus, 16), int(minus, 16)]
        got = oracle.search_candidates(np.array([a]), qmax)[0]
        assert [int(v) for v in got] == want
        assert _exact_candidates(a, qmax) == want


def test_search_candidates_exact_over_binades():
    """oracle.search_candidates against exact rational rounding for group
    maxima spread over the FP16 range (subnormal scales included)."""
    rng = np.random.default_rng(905)
    a = (rng.uniform(1.0, 2.0, 60) * 2.0 ** rng.integers(-22, 15, 60)).astype(np.float32)
    for bits in (4, 5, 6, 8):
        qmax = oracle.QMAX[bits]
        cand = oracle.search_candidates(a.astype(np.float64), qmax)
        for ai, row in zip(a, cand):
            assert [int(v) for v in row] == _exact_candidates(float(ai), qmax), (bits, ai)


def test_search_ties_go_to_the_first_candidate():
    rng = synth.generator(0, 901)
    w = synth.gauss_weights(rng, 2, 64)
    c, s = oracle.search_encode(w, 5, imatrix=np.zeros(64, np.float32))   # every error 0
    for r in range(2):
        assert s[r, 0] == _exact_candidates(float(np.abs(w[r]).max()), 15)[0]
    z = np.zeros((1, 128), np.float32)
    c, s = oracle.search_encode(z, 6)
    assert np.all(s == 0) and np.all(c == 0)


def test_search_single_important_channel_matches_exact_brute_force():
    """Importance on one channel only: the chosen candidate must minimise that
    one weight's error, checked in exact rational arithmetic over the 50
    candidates (first one on ties)."""
    rng = synth.generator(0, 902)
    for bits in (4, 5, 6):
        lo, hi = oracle.code_range(bits)
        for trial in range(6):
            w = synth.gauss_weights(rng, 1, 64)
            j = int(rng.integers(64))
            q = np.zeros(64, np.float32)
            q[j] = 1.0
            c, s = oracle.search_encode(w, bits, q)
            cand = _exact_candidates(float(np.abs(w).max()), oracle.QMAX[bits])
            wj = Fraction(float(w[0, j]))
            errs = []
            for b in cand:
                sv = Fraction(float(oracle.fp16_to_f64(np.array([b], np.uint16))[0]))
                code = 0 if sv == 0 else min(max(round(wj / sv), lo), hi)   # round: half to even
                errs.append((wj - sv * code) ** 2)
            best = min(range(len(errs)), key=lambda i: (errs[i], i))
            assert s[0, 0] == cand[best], (bits, trial)


def test_search_importance_scale_invariance_and_overflow():
    rng = synth.generator(0, 903)
    w = synth.gauss_weights(rng, 8, 256)
    q = synth.imatrix(rng, 256)
    c1, s1 = oracle.search_encode(w, 4, q)
    c2, s2 = oracle.search_encode(w, 4, q * np.float32(4.0))     # errors scale exactly by 4
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)
    big = np.full((1, 64), 7.0e5, np.float32)                     # every candidate > 65504
    with pytest.raises(ValueError):
        oracle.search_encode(big, 4)


# ---------------------------------------------------------------- bf16 rounding, SwiGLU
def test_bf16_rounding_identity_and_ties():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = bits[(bits & 0x7F80) != 0x7F80]
    v = oracle.bf16_to_f64(finite)
    back = oracle.f64_to_bf16_bits(v)
    # every finite bf16 value maps to itself (both zeros keep their sign)
    assert np.array_equal(back, finite)
    # midpoints between neighbours round to the even pattern (positive, normal)
    lo = np.arange(0x0080, 0x7F7F, 7, dtype=np.uint16)
    a, b = oracle.bf16_to_f64(lo), oracle.bf16_to_f64(lo + 1)
    mid = (a + b) / 2.0                                        # exact in fp64
    got = oracle.f64_to_bf16_bits(mid)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(got, want)
    assert oracle.f64_to_bf16_bits(np.array([3.5e38]))[0] == 0x7F80      # overflow
    assert oracle.f64_to_bf16_bits(np.array([2.0 ** -134]))[0] == 0x0000  # half the subnormal step: to even (0)


def test_bf16_rounding_nearest_in_exact_arithmetic():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(2000) * np.exp(rng.uniform(-30, 30, 2000))
    r = oracle.bf16_to_f64(oracle.f64_to_bf16_bits(x))
    for xi, ri in zip(x[:300], r[:300]):
        m, e = np.frexp(xi)
        q = Fraction(2) ** int(e - 8)
        assert abs(Fraction(float(xi)) - Fraction(float(ri))) <= q / 2


def test_silu_identities():
    g = np.linspace(-30.0, 30.0, 601)
    s = oracle.silu(g)
    # silu(g) - silu(-g) = g and silu(0) = 0, silu(g) -> g for large g, -> 0 for very negative g
    assert np.allclose(s - oracle.silu(-g), g, rtol=0, atol=1e-12)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.silu(np.array([40.0]))[0] - 40.0) < 1e-15 * 40
    assert abs(oracle.silu(np.array([-800.0]))[0]) == 0.0
    # swiglu of (g, 1) is silu(g) rounded to bf16; (0, u) gives 0
    act = oracle.swiglu_bf16(g, np.ones_like(g))
    assert np.array_equal(act, oracle.f64_to_bf16_bits(s))
    assert np.all(oracle.bf16_to_f64(oracle.swiglu_bf16(np.zeros(5), np.arange(5.0))) == 0.0)


# ---------------------------------------------------------------- the layer MLP
def _one_hot_mlp_case():
    """A layer with H = 64 (one group), I = 64, H_out = 16 whose every value is
    known in closed form: x is one-hot at k = 5 with value 1, so gate[i] and
    up[i] are scale * code of column 5; gates are +-64 or 0, ups small
    dyadic values, and the down weights 0.25 times small codes."""
    H, I, Ho = 64, 64, 16
    gate_codes = [4, 4, -4, 0, 4, -4, 4, 4] + [0] * (I - 8)   # gate = 16 c: 64, 64, -64, 0, ...
    up_codes = [3, -5, 7, 6, 1, 2, -8, 0] + [1] * (I - 8)     # up = 0.5 c
    cg = np.zeros((I, H), np.int8)
    cu = np.zeros((I, H), np.int8)
    cg[:, 5] = gate_codes
    cu[:, 5] = up_codes
    sg = np.full((I, 1), 0x4C00, np.uint16)             # 16.0
    su = np.full((I, 1), 0x3800, np.uint16)             # 0.5
    x = np.zeros((1, H), np.uint16)
    x[0, 5] = 0x3F80                                      # bf16 1.0
    rng = np.random.default_rng(31)
    cd = rng.integers(-8, 8, (Ho, I)).astype(np.int8)
    sd = np.full((Ho, 1), 0x3400, np.uint16)            # 0.25
    return cg, sg, cu, su, cd, sd, x, gate_codes, up_codes


def test_mlp_closed_form():
    """oracle.mlp on a one-hot layer: silu(64) = 64 and silu(0) = 0 exactly in
    fp64, silu(-64) = -64 / (1 + e^64) (below 1e-25), so act = bf16(64 u) is
    exact, act for a zero gate is 0, and y = sum_i w_down[:, i] act[i] is
    checked in exact rational arithmetic."""
    cg, sg, cu, su, cd, sd, x, gcodes, ucodes = _one_hot_mlp_case()
    I = len(gcodes)
    act, y, e, gate, up, e_g, e_u = oracle.mlp(np.concatenate([cg, cu]), np.concatenate([sg, su]),
                                               cd, sd, x)            # (gate; up) row order
    assert act.shape == (1, I) and y.shape == (1, cd.shape[0])
    assert list(gate[0]) == [16.0 * c for c in gcodes]
    assert list(up[0]) == [0.5 * c for c in ucodes]
    a = oracle.bf16_to_f64(act[0])
    for i in range(I):
        u = 0.5 * ucodes[i]
        if gcodes[i] > 0:
            assert a[i] == 64.0 * u                      # exact in bf16 (small dyadic)
        elif gcodes[i] == 0:
            assert a[i] == 0.0
        else:
            assert abs(a[i]) < 1e-25 * max(1.0, abs(u))
            assert a[i] == 0.0 or np.sign(a[i]) == -np.sign(u)
    # y in exact rationals from those activations: every term is a dyadic
    # rational with few bits, so the fp64 sums are exact up to the tiny
    # negative-gate terms
    for n in range(cd.shape[0]):
        ref = sum(Fraction(int(cd[n, i]), 4) * Fraction(float(a[i])) for i in range(I))
        assert abs(Fraction(float(y[0, n])) - ref) <= Fraction(1, 10 ** 20)
        big = sum(Fraction(int(cd[n, i]), 4) * Fraction(float(a[i])) for i in range(I) if gcodes[i] > 0)
        assert abs(Fraction(float(y[0, n])) - big) <= Fraction(1, 10 ** 20)


def test_mlp_planted_mistakes_are_caught():
    """Swapping the gate and up halves, or skipping the bf16 rounding of act,
    changes the closed-form result of test_mlp_closed_form."""
    cg, sg, cu, su, cd, sd, x, gcodes, ucodes = _one_hot_mlp_case()
    act, y, *_ = oracle.mlp(np.concatenate([cg, cu]), np.concatenate([sg, su]), cd, sd, x)
    act_sw, y_sw, *_ = oracle.mlp(np.concatenate([cu, cg]), np.concatenate([su, sg]), cd, sd, x)
    assert not np.array_equal(act, act_sw) and not np.array_equal(y, y_sw)
    # a layer that rounds act only after the down product would differ where
    # silu(g) u is not a bf16 value: g = 1 gives silu(1) = 0.7310585786...
    cg1 = cg.copy()
    cg1[:, 5] = 0
    cg1[0, 5] = 1
    sg1 = np.full_like(sg, 0x3C00)                       # 1.0: gate[0] = 1
    act1, y1, *_ = oracle.mlp(np.concatenate([cg1, cu]), np.concatenate([sg1, su]), cd, sd, x)
    exact_act0 = 1.0 / (1.0 + np.exp(-1.0)) * (0.5 * ucodes[0])
    assert oracle.bf16_to_f64(act1[0, 0]) != exact_act0
    assert abs(oracle.bf16_to_f64(act1[0, 0]) - exact_act0) <= abs(exact_act0) * 2.0 ** -8   # half a bf16 step
