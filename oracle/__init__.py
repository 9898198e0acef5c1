"""CPU oracle for groupwise-quantized small-T GEMV -- test infrastructure only.

This package is the slow, plain reference that the CUDA path is checked
against.  It is not part of the product: only the test-suite, the smoke check
and the CPU-baseline leg of the benchmark may import it.  It shares no code
with the CUDA library (no layout, no packer, no kernels) and imports nothing
from it.

What it computes, and where that is defined
-------------------------------------------
Page "Qwen3.8-27B for NInfer on the RTX 3090" (model card of the 3090 fork's
groupwise-int artifact), section "What is different from the upstream
artifact":

* the upstream encoder rounds every group of 64 consecutive weights to the
  nearest integer code, with one FP16 scale per group equal to the group's
  absolute maximum divided by the largest positive code (qmax);
* the fork's searched encoder may store negative scales, which lets a group
  reach the most negative code (-8 for 4-bit, -16 for 5-bit);
* a weight is the product scale * code.

The code widths are 4, 5 and 6 bits, signed two's-complement ranges
[-8, 7], [-16, 15] and [-32, 31] (same section: "Q4 ... Q5", "a 6-bit output
head").  Activations are bf16 and outputs fp32; the oracle works in fp64.

Readings where the page is silent (each is listed in the design notes):

* scale = FP16 round-to-nearest-even of the exact quotient absmax / qmax;
  the quotient is formed in fp64, whose rounding never crosses an FP16
  rounding boundary for an fp32 numerator and qmax in {7, 15, 31};
* code = round-half-to-even(w / scale), computed in fp64 (exact decision),
  then clamped to [-qmax-1, qmax];
* an all-zero group, or a scale that rounds to zero, gives scale +0 and
  code 0 everywhere in the group;
* a quotient that overflows FP16 is an error.

Pins: every function here is checked in ``tests/test_oracle_pins.py``
against facts that do not come from the oracle itself (library conversions,
exhaustive sweeps, exact rational arithmetic, closed forms, planted
mistakes).  See the header of each function for its pin.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "QMAX", "GROUP", "fp16_to_f64", "bf16_to_f64", "f64_to_fp16_bits",
    "rtn_scales", "rtn_encode", "dequant", "dequant_f32", "gemv",
    "tolerance_ok", "max_violation",
]

GROUP = 64                       # weights per group along K
QMAX = {4: 7, 5: 15, 6: 31, 8: 127}   # largest positive code per width


def code_range(bits: int) -> tuple[int, int]:
    """Signed two's-complement range of a `bits`-wide code."""
    return -(1 << (bits - 1)), (1 << (bits - 1)) - 1


# --------------------------------------------------------------------------
# Number formats (IEEE-754 binary16 and bfloat16), decoded from their
# definitions.  Pin: exhaustive comparison with numpy's float16 and torch's
# bfloat16 conversions over all 65,536 bit patterns.
# --------------------------------------------------------------------------
def fp16_to_f64(bits) -> np.ndarray:
    """Value of IEEE binary16 bit patterns, as float64 (exact).

    sign (1) | exponent (5, bias 15) | fraction (10).  Exponent 0 encodes
    zero and subnormals (fraction * 2^-24); exponent 31 encodes inf/NaN.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    sub = f * 2.0 ** -24
    nrm = (1024.0 + f) * np.exp2((e - 25).astype(np.float64))
    val = np.where(e == 0, sub, nrm)
    special = np.where(f == 0, np.inf, np.nan)
    val = np.where(e == 31, special, val)
    return sign * val


def bf16_to_f64(bits) -> np.ndarray:
    """Value of bfloat16 bit patterns: the upper 16 bits of an IEEE binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f64_to_fp16_bits(v) -> np.ndarray:
    """IEEE round-to-nearest-even of float64 values to binary16 bit patterns
    (numpy's float64 -> float16 conversion, which rounds once from the
    double; overflow gives inf)."""
    with np.errstate(over="ignore"):
        return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def f64_to_bf16_bits(v) -> np.ndarray:
    """IEEE round-to-nearest-even of float64 values to bfloat16 bit patterns in
    one rounding: 8 significant bits, step 2^-133 below the normal range,
    overflow to infinity."""
    x = np.asarray(v, dtype=np.float64)
    fin = np.isfinite(x)
    xf = np.where(fin, x, 0.0)
    _, e = np.frexp(xf)
    q = np.ldexp(1.0, np.maximum(e - 8, -133))
    r = np.rint(xf / q) * q
    with np.errstate(over="ignore"):
        r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, xf), r)
    r = np.where(fin, r, x)
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


# --------------------------------------------------------------------------
# Round-to-nearest encoder ("upstream" encoder on the 3090 model card).
# Pin: exact rational nearest-FP16 search for the scale, brute-force nearest
# code over the whole code range, and the |w - s*c| <= |s|/2 invariant.
# --------------------------------------------------------------------------
def rtn_scales(w: np.ndarray, qmax: int) -> np.ndarray:
    """FP16 scale bits [N, K/64]: fp16_rne(max|w| / qmax) per 64-group.

    Raises ValueError if a scale overflows FP16.
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % GROUP:
        raise ValueError("K must be a multiple of 64")
    a = np.abs(w.reshape(n, k // GROUP, GROUP)).max(axis=2).astype(np.float64)
    s = f64_to_fp16_bits(a / float(qmax))
    if np.any((s & 0x7C00) == 0x7C00):
        raise ValueError("group scale overflows FP16")
    return s


def rtn_codes(w: np.ndarray, scale_bits: np.ndarray, bits: int) -> np.ndarray:
    """int8 codes [N, K]: clamp(rint(w / s), -qmax-1, qmax), s the FP16 scale.

    A zero scale gives code 0.  The quotient and the rounding are done in
    fp64; rint rounds half to even.
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    lo, hi = code_range(bits)
    s = fp16_to_f64(scale_bits).reshape(n, k // GROUP, 1)
    wg = w.reshape(n, k // GROUP, GROUP).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(wg / s)
    q = np.where(s == 0.0, 0.0, q)
    q = np.clip(q, lo, hi)
    return q.reshape(n, k).astype(np.int8)


def rtn_encode(w: np.ndarray, bits: int, chunk_rows: int = 2048):
    """Round-to-nearest encode: returns (codes int8 [N,K], scale bits uint16 [N,K/64])."""
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    qmax = QMAX[bits]
    codes = np.empty((n, k), dtype=np.int8)
    scales = np.empty((n, k // GROUP), dtype=np.uint16)
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        s = rtn_scales(w[r0:r1], qmax)
        scales[r0:r1] = s
        codes[r0:r1] = rtn_codes(w[r0:r1], s, bits)
    return codes, scales


# --------------------------------------------------------------------------
# Searched encoder ("grouped_search" on the 3090 model card, section "What is
# different from the upstream artifact"): each group's FP16 scale is the best
# of 50 candidates by importance-weighted squared error, importance being a
# per-channel imatrix (mean squared input activation); scales may be negative.
# The page does not list the candidates; the reading taken here (also in the
# design notes): with a = max|w| over the group and qmax the largest positive
# code, the 25 magnitudes h_i = fp16_rne(12 a / (12 (qmax + 1) - i)), i = 0..24,
# i.e. a / L for L from qmax + 1 down to qmax - 1 in steps of 1/12, each tried
# as +h_i and -h_i (candidate 2i and 2i + 1).  A candidate's codes are
# clamp(rint(w / s)) as in the round-to-nearest encoder (a zero scale gives
# code 0); its error is sum_k q_k (w_k - s c_k)^2, accumulated over k in
# order in fp64 with every product and sum rounded separately.  The smallest
# error wins, ties to the lower candidate number; candidates whose scale
# overflows FP16 take no part.  i = 12 is the round-to-nearest scale, so the
# search never does worse than that encoder under the same importance.
# --------------------------------------------------------------------------
SEARCH_STEPS = 25


def search_candidates(a: np.ndarray, qmax: int) -> np.ndarray:
    """FP16 bit patterns of the 50 candidate scales for group maxima a (fp64),
    shape a.shape + (50,), in candidate order (+h_0, -h_0, +h_1, ...)."""
    a = np.asarray(a, dtype=np.float64)
    den = 12.0 * (qmax + 1) - np.arange(SEARCH_STEPS, dtype=np.float64)
    h = f64_to_fp16_bits((12.0 * a)[..., None] / den)          # [..., 25]
    out = np.empty(a.shape + (2 * SEARCH_STEPS,), dtype=np.uint16)
    out[..., 0::2] = h
    out[..., 1::2] = h | np.uint16(0x8000)
    return out


def search_encode(w: np.ndarray, bits: int, imatrix=None, chunk_groups: int = 2048):
    """Searched encode: returns (codes int8 [N, K], scale bits uint16 [N, K/64]).
    imatrix: per-channel importance [K] (>= 0), None for all ones.  Raises
    ValueError if every candidate of some group overflows FP16."""
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % GROUP:
        raise ValueError("K must be a multiple of 64")
    g = k // GROUP
    lo, hi = code_range(bits)
    q = np.ones(k, np.float64) if imatrix is None else np.asarray(imatrix, np.float32).astype(np.float64)
    qg = q.reshape(g, GROUP)
    wg = w.reshape(n * g, GROUP).astype(np.float64)
    qrow = np.tile(qg, (n, 1))                                   # [n*g, 64]
    codes = np.empty((n * g, GROUP), np.int8)
    scales = np.empty(n * g, np.uint16)
    for r0 in range(0, n * g, chunk_groups):
        r1 = min(n * g, r0 + chunk_groups)
        ww, qq = wg[r0:r1], qrow[r0:r1]
        cand = search_candidates(np.abs(ww).max(axis=1), QMAX[bits])      # [m, 50]
        sv = fp16_to_f64(cand)[:, :, None]                                 # [m, 50, 1]
        with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
            c = np.rint(ww[:, None, :] / sv)
            c = np.where(sv == 0.0, 0.0, c)
            c = np.clip(c, lo, hi)
            d = ww[:, None, :] - sv * c          # (overflowed candidates give NaN here)
            err = np.add.accumulate(qq[:, None, :] * (d * d), axis=2)[:, :, -1]   # in order over k
        err = np.where(np.isinf(sv[:, :, 0]), np.inf, err)
        if np.any(np.all(np.isinf(sv[:, :, 0]), axis=1)):
            raise ValueError("every candidate scale overflows FP16")
        best = np.argmin(err, axis=1)                                      # first minimum
        idx = np.arange(r1 - r0)
        scales[r0:r1] = cand[idx, best]
        codes[r0:r1] = c[idx, best].astype(np.int8)
    return codes.reshape(n, k), scales.reshape(n, g)


def weighted_error(w: np.ndarray, codes: np.ndarray, scale_bits: np.ndarray, imatrix=None):
    """sum_k q_k (w_k - s c_k)^2 per group [N, K/64] in fp64 (for tests)."""
    w = np.asarray(w, dtype=np.float32).astype(np.float64)
    n, k = w.shape
    q = np.ones(k) if imatrix is None else np.asarray(imatrix, np.float32).astype(np.float64)
    s = np.repeat(fp16_to_f64(scale_bits), GROUP, axis=1)
    d = w - s * codes.astype(np.float64)
    return (q[None, :] * d * d).reshape(n, k // GROUP, GROUP).sum(axis=2)


# --------------------------------------------------------------------------
# Dequantisation and the product.
# Pin: exhaustive FP16 x code sweep (product exact in fp32), one-hot and
# constant inputs, and exact rational arithmetic on small shapes.
# --------------------------------------------------------------------------
def dequant(codes: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """w[n, k] = s[n, k // 64] * c[n, k] in fp64 (exact: an 11-bit significand
    times a code of at most 6 bits)."""
    c = np.asarray(codes, dtype=np.int8)
    n, k = c.shape
    s = fp16_to_f64(scale_bits).reshape(n, k // GROUP, 1)
    return (s * c.reshape(n, k // GROUP, GROUP).astype(np.float64)).reshape(n, k)


def dequant_f32(codes: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """The dequantised weights as fp32 (the cast is exact)."""
    return dequant(codes, scale_bits).astype(np.float32)


def gemv(codes: np.ndarray, scale_bits: np.ndarray, x_bits: np.ndarray):
    """y*[t, n] = sum_k w[n, k] * x[t, k] and E[t, n] = sum_k |w[n, k] * x[t, k]|,
    both in fp64.  x is given as bf16 bit patterns [T, K]."""
    w = dequant(codes, scale_bits)
    x = bf16_to_f64(x_bits)
    y = x @ w.T
    e = np.abs(x) @ np.abs(w).T
    return y, e


# --------------------------------------------------------------------------
# Verify-head reductions over the outputs of one token (page "giveen/ninfer-ext",
# section "Engineering": single-pass logsumexp; page "Qwen3.8-27B for NInfer on
# the RTX 3090", section "Run it": candidate top-k over the full head).
# --------------------------------------------------------------------------
def head_reduce(y):
    """Per token t of y[T, N] (fp64): the argmax (first index of the largest
    value), the largest value, and logsumexp = log(sum_n exp(y[t, n])),
    evaluated as m + log(sum exp(y - m)) with m the maximum so no term
    overflows."""
    y = np.asarray(y, dtype=np.float64)
    am = np.argmax(y, axis=1)                       # first occurrence of the maximum
    m = y[np.arange(y.shape[0]), am]
    # a +inf logit makes the sum +inf; the shifted form would compute inf - inf
    fin = np.where(np.isposinf(m), 0.0, m)
    with np.errstate(invalid="ignore"):
        lse = fin + np.log(np.sum(np.exp(y - fin[:, None]), axis=1))
    lse = np.where(np.isposinf(m), np.inf, lse)
    return am, m, lse


def head_topk(y, k):
    """Per token t of y[T, N]: the k largest outputs as (index [T, k] int64,
    value [T, k]) in the order larger value first, -0 below +0, equal values
    by smaller index (the pages leave k and the order of ties open; this
    reading makes the answer unique).  With k > N the tail is index -1, value
    -inf.  A stable sort on (value descending, then the sign of zero), the
    index order being kept by stability."""
    y = np.asarray(y)
    T, N = y.shape
    idx = np.full((T, k), -1, dtype=np.int64)
    val = np.full((T, k), -np.inf, dtype=y.dtype if y.dtype.kind == "f" else np.float64)
    for t in range(T):
        row = y[t]
        # lexsort: last key primary.  Primary: value descending; secondary:
        # +0 before -0 (signbit ascending); stability keeps index order.
        order = np.lexsort((np.signbit(row), -row))
        n = min(k, N)
        idx[t, :n] = order[:n]
        val[t, :n] = row[order[:n]]
    return idx, val


# --------------------------------------------------------------------------
# MLP of the decoder layer (page "giveen/ninfer-ext", fused gate+up; page
# "Qwen3.8-27B for NInfer on the RTX 3090", Q4 gate/up and down projections):
# act = silu(gate) * up with silu(g) = g / (1 + exp(-g)), rounded to bf16
# because it is the bf16 input of the down projection; y = act W_down^T.
# --------------------------------------------------------------------------
def silu(g):
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_bf16(gate, up):
    """bf16 bit patterns of silu(gate) * up, computed in fp64, rounded once."""
    return f64_to_bf16_bits(silu(gate) * np.asarray(up, dtype=np.float64))


def mlp(codes_gu, scales_gu, codes_down, scales_down, x_bits):
    """The layer's MLP on x [T, H] (bf16 bits): gate+up [2I, H] in (gate; up)
    row order, act [T, I] (bf16 bits), y [T, H'] and the down product's error
    scale E = sum |w act|.  Returns (act_bits, y, E, gate, up, E_gate, E_up)."""
    y_gu, e_gu = gemv(codes_gu, scales_gu, x_bits)
    i = y_gu.shape[1] // 2
    act = swiglu_bf16(y_gu[:, :i], y_gu[:, i:])
    y, e = gemv(codes_down, scales_down, act)
    return act, y, e, y_gu[:, :i], y_gu[:, i:], e_gu[:, :i], e_gu[:, i:]


# --------------------------------------------------------------------------
# Acceptance test on outputs: |y - y*| <= 1e-4 * E + 1e-6 per element.
# --------------------------------------------------------------------------
REL_TOL = 1e-4
ABS_TOL = 1e-6


def max_violation(y, y_star, e) -> float:
    """max over elements of |y - y*| / (1e-4 E + 1e-6); <= 1 means pass.
    A NaN or inf in y counts as a failure."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_star)
    bound = REL_TOL * e + ABS_TOL
    r = err / bound
    r = np.where(np.isfinite(r), r, np.inf)
    return float(r.max()) if r.size else 0.0


def tolerance_ok(y, y_star, e) -> bool:
    return max_violation(y, y_star, e) <= 1.0
