"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Bar: bit-exact for the encoder (codes, scale bits), the packers and the
dequantised weights; |y - y*| <= 1e-4 * sum|w x| + 1e-6 per output for the
GEMV (the tolerance of oracle.tolerance_ok); exact equality where the
arithmetic is provably identical (one-hot inputs, zero codes, negated scales,
T-invariance at a fixed launch plan, repeat runs)."""
import numpy as np
import pytest
import torch

import oracle
import quantized_weight_decode_gb300 as nqp
import synth
from cases import device_weight, device_x, oracle_inputs, rtn_case, uniform_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def built():
    nqp.build()
    nqp.lib()
    torch.cuda.set_device(0)
    assert nqp.last_device_error() == 0


def _y(case, packed, sp, route=0, ksplit=0, T=None):
    T = case["T"] if T is None else T
    x = device_x(torch, case, DEV)[:T].contiguous()
    y = torch.full((T, case["N"]), float("nan"), dtype=torch.float32, device=DEV)
    nqp.gemv(packed, sp, x, y, case["K"], case["N"], T, case["bits"], route=route, ksplit=ksplit)
    assert nqp.last_device_error() == 0
    return y.cpu().numpy()


def _check(case, y, rows=None):
    codes, sb = oracle_inputs(case, rows)
    y_ref, e_ref = oracle.gemv(codes, sb, case["xb"][: y.shape[0]])
    got = y if rows is None else y[:, rows]
    v = oracle.max_violation(got, y_ref, e_ref)
    assert v <= 1.0, f"tolerance ratio {v}"
    return v


# ---------------------------------------------------------------- encoder, packers, dequant
@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_quantize_rtn_bit_exact(bits):
    case = rtn_case((300, bits), bits, 96, 512, 1)
    w = case["w"]
    w[0, :64] = 0                                    # all-zero group
    w[1, :64] *= np.float32(1e-6)                    # subnormal-scale group
    w[2, 64:128] = np.float32(0.5)                   # constant group
    w[3, 128:192] *= np.float32(300.0)               # large magnitudes
    codes, scales = nqp.quantize_rtn(torch.from_numpy(w).to(DEV), bits)
    assert nqp.last_device_error() == 0
    c_ref, s_ref = oracle.rtn_encode(w, bits)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), s_ref)


def test_quantize_rtn_overflow_sets_status():
    w = torch.full((16, 64), 7.0 * 70000.0, dtype=torch.float32, device=DEV)
    nqp.quantize_rtn(w, 4)
    assert nqp.last_device_error() == nqp.ERANGE
    assert nqp.last_device_error() == 0              # read clears


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_pack_device_matches_host_pack(bits):
    case = uniform_case((301, bits), bits, 53, 320, 1)
    codes, sb = oracle_inputs(case)
    hp, hs = nqp.pack(codes, sb, bits)
    dp, ds = nqp.pack_device(torch.from_numpy(codes).to(DEV),
                             torch.from_numpy(sb.view(np.int16)).to(DEV), bits)
    assert nqp.last_device_error() == 0
    assert np.array_equal(dp.cpu().numpy(), hp)
    assert np.array_equal(ds.cpu().numpy().view(np.uint16), hs)


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("kind", ["rtn", "uniform"])
def test_dequant_bit_exact(bits, kind):
    mk = rtn_case if kind == "rtn" else uniform_case
    case = mk((302, bits), bits, 77, 384, 1)
    packed, sp = device_weight(nqp, torch, case, DEV)
    w = nqp.dequant(packed, sp, case["K"], case["N"], bits).cpu().numpy()
    codes, sb = oracle_inputs(case)
    ref = oracle.dequant_f32(codes, sb)
    assert np.array_equal(w.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_dequant_every_scale_pattern(bits):
    # all 63,488 finite FP16 scale patterns x codes cycling through the range
    finite = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = finite[(finite & 0x7C00) != 0x7C00]
    G = 8
    N = -(-finite.size // G)
    sb = np.zeros(N * G, np.uint16)
    sb[: finite.size] = finite
    sb = sb.reshape(N, G)
    lo, hi = oracle.code_range(bits)
    codes = (lo + (np.arange(N * G * 64) % (hi - lo + 1))).astype(np.int8).reshape(N, G * 64)
    hp, hs = nqp.pack(codes, sb, bits)
    w = nqp.dequant(torch.from_numpy(hp).to(DEV), torch.from_numpy(hs.view(np.int16)).to(DEV),
                    G * 64, N, bits).cpu().numpy()
    ref = oracle.dequant_f32(codes, sb)
    assert np.array_equal(w.view(np.uint32), ref.view(np.uint32))


# ---------------------------------------------------------------- GEMV parity
SHAPES = [(512, 256), (1024, 200), (2048, 37), (64, 16), (192, 1)]


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("T", [1, 2, 3, 8, 9, 16])
def test_gemv_mma_parity(bits, T):
    for i, (K, N) in enumerate(SHAPES):
        case = uniform_case((303, bits, T, i), bits, N, K, T) if i % 2 else \
            rtn_case((303, bits, T, i), bits, N, K, T)
        packed, sp = device_weight(nqp, torch, case, DEV)
        _check(case, _y(case, packed, sp, route=nqp.ROUTE_MMA))


@pytest.mark.parametrize("bits", [4, 5, 6])
@pytest.mark.parametrize("T", [1, 2, 4])
def test_gemv_ffma_parity(bits, T):
    for i, (K, N) in enumerate(SHAPES[:3]):
        case = uniform_case((304, bits, T, i), bits, N, K, T)
        packed, sp = device_weight(nqp, torch, case, DEV)
        _check(case, _y(case, packed, sp, route=nqp.ROUTE_FFMA))


@pytest.mark.parametrize("ksplit", [1, 2, 4, 8])
@pytest.mark.parametrize("T", [1, 5, 8, 12, 16])
def test_gemv_ksplit_parity(ksplit, T):
    case = uniform_case((305, ksplit, T), 5, 300, 17408 // 8, T)
    packed, sp = device_weight(nqp, torch, case, DEV)
    _check(case, _y(case, packed, sp, route=nqp.ROUTE_MMA, ksplit=ksplit))


def test_tiny_config():
    case = rtn_case((1,), 4, 256, 512, 1)
    packed, sp = device_weight(nqp, torch, case, DEV)
    _check(case, _y(case, packed, sp))


def test_many_jobs_per_cluster():
    # more row tiles than resident clusters: every CTA runs several jobs and
    # the reduction slots wrap around many times
    case = rtn_case((306,), 6, 16 * 700 + 5, 256, 3)
    packed, sp = device_weight(nqp, torch, case, DEV)
    for ks in (1, 2):
        _check(case, _y(case, packed, sp, route=nqp.ROUTE_MMA, ksplit=ks))


# ---------------------------------------------------------------- two token blocks, hybrid x
# (K, N, K split): whole warp slices of 5 groups, uneven slices, K splits 2 and 4
HYBRID_SHAPES = [(2560, 300, 1), (1088, 37, 1), (4096, 170, 2), (8192, 50, 4)]


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("T", [9, 11, 13, 15, 16])
def test_hybrid_x_parity(bits, T, monkeypatch):
    """T > 8 through the kernel that keeps tokens 0-7 in registers and tokens
    8.. in shared memory: ragged row tiles, uneven warp slices, K splits 1 to
    4, element by element against the oracle."""
    monkeypatch.setenv("NQ_XREGH", "1")
    # five groups per warp at K = 5120: the x tile (T - 8) x 10 KB and two
    # stages fit next to each other up to 5-bit codes at every T
    shapes = HYBRID_SHAPES + ([(5120, 200, 1)] if bits <= 5 else [])
    for i, (K, N, ks) in enumerate(shapes):
        assert nqp.plan(K, N, T, bits, route=nqp.ROUTE_MMA, ksplit=ks)["x"] == "hybrid"
        case = uniform_case((330, bits, T, i), bits, N, K, T) if i % 2 else \
            rtn_case((330, bits, T, i), bits, N, K, T)
        packed, sp = device_weight(nqp, torch, case, DEV)
        _check(case, _y(case, packed, sp, route=nqp.ROUTE_MMA, ksplit=ks))


@pytest.mark.parametrize("bits", [4, 8])
def test_hybrid_x_one_hot_tokens_exact(bits, monkeypatch):
    """One-hot x at T = 12 (tokens 8-11 come from the shared-memory tile):
    every token's output is its weight column exactly, for both two-block
    kernels."""
    case = uniform_case((331, bits), bits, 90, 2560, 12)
    codes, sb = oracle_inputs(case)
    packed, sp = _upload_packed(codes, sb, bits)
    ks_cols = [0, 63, 64, 511, 512, 1000, 1279, 1280, 2047, 2100, 2558, 2559]
    xb = np.zeros((12, 2560), np.uint16)
    for t, k in enumerate(ks_cols):
        xb[t, k] = 0x3F80
    c2 = dict(case, xb=xb)
    wref = oracle.dequant_f32(codes, sb)
    for env, place in (("1", "hybrid"), ("0", "regs2")):
        monkeypatch.setenv("NQ_XREGH", env)
        for ks in (1, 2):
            pl = nqp.plan(2560, 90, 12, bits, route=nqp.ROUTE_MMA, ksplit=ks)
            assert pl["x"] == place, (env, ks, pl)
            y = _y(c2, packed, sp, route=nqp.ROUTE_MMA, ksplit=ks)
            for t in range(12):
                assert np.array_equal(y[t], wref[:, ks_cols[t]]), (env, ks, t)


def test_two_block_kernel_choice():
    """The planner's measured rule for T > 8: the hybrid where it allows a
    smaller K split than both blocks in registers, both in registers at an
    equal split."""
    p = nqp.plan(5120, 34816, 16, 4)      # gate+up: hybrid at KS 1 (regs2 needs KS 2)
    assert (p["x"], p["ksplit"]) == ("hybrid", 1), p
    p = nqp.plan(17408, 5120, 12, 5)      # down: hybrid at KS 4 (regs2 needs KS 8)
    assert (p["x"], p["ksplit"]) == ("hybrid", 4), p
    p = nqp.plan(5120, 248320, 16, 6)     # head: the hybrid does not fit at KS 1
    assert (p["x"], p["ksplit"]) == ("regs2", 2), p
    assert nqp.plan(5120, 34816, 8, 4)["x"] == "regs"


# ---------------------------------------------------------------- exact invariants
def _upload_packed(codes, sb, bits):
    hp, hs = nqp.pack(codes, sb, bits)
    return torch.from_numpy(hp).to(DEV), torch.from_numpy(hs.view(np.int16)).to(DEV)


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_one_hot_x_gives_weight_column_exactly(bits):
    case = uniform_case((307, bits), bits, 100, 1024, 4)
    codes, sb = oracle_inputs(case)
    packed, sp = _upload_packed(codes, sb, bits)
    ks_cols = [0, 63, 64, 517, 1023]
    xb = np.zeros((len(ks_cols), 1024), np.uint16)
    for t, k in enumerate(ks_cols):
        xb[t, k] = 0x3F80
    c2 = dict(case, xb=xb, T=len(ks_cols))
    routes = ((nqp.ROUTE_MMA, 1), (nqp.ROUTE_MMA, 4)) + (((nqp.ROUTE_FFMA, 2),) if bits < 8 else ())
    for route, ks in routes:
        y = _y(c2, packed, sp, route=route, ksplit=ks, T=4)
        wref = oracle.dequant_f32(codes, sb)
        for t in range(4):
            assert np.array_equal(y[t], wref[:, ks_cols[t]]), (route, ks, t)


def test_zero_codes_and_negated_scales():
    case = uniform_case((308,), 5, 80, 512, 8)
    codes, sb = oracle_inputs(case)
    packed, sp = _upload_packed(np.zeros_like(codes), sb, 5)
    assert np.all(_y(case, packed, sp) == 0)
    p1, s1 = _upload_packed(codes, sb, 5)
    p2, s2 = _upload_packed(codes, sb ^ np.uint16(0x8000), 5)
    for route in (nqp.ROUTE_MMA, nqp.ROUTE_FFMA):
        y1 = _y(case, p1, s1, route=route, ksplit=2, T=4)
        y2 = _y(case, p2, s2, route=route, ksplit=2, T=4)
        assert np.array_equal(y1, -y2)


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_t_invariance_exact(bits):
    case = rtn_case((309, bits), bits, 150, 1024, 16)
    packed, sp = device_weight(nqp, torch, case, DEV)
    y16 = _y(case, packed, sp, route=nqp.ROUTE_MMA, ksplit=2, T=16)
    for T in (1, 5, 8, 12):
        yt = _y(case, packed, sp, route=nqp.ROUTE_MMA, ksplit=2, T=T)
        assert np.array_equal(yt, y16[:T]), T
    # a single-token call on token 11 alone equals row 11
    c1 = dict(case, xb=case["xb"][11:12].copy(), T=1)
    y1 = _y(c1, packed, sp, route=nqp.ROUTE_MMA, ksplit=2)
    assert np.array_equal(y1[0], y16[11])


def test_repeat_runs_identical():
    case = uniform_case((310,), 5, 1000, 4096, 8)
    packed, sp = device_weight(nqp, torch, case, DEV)
    a = _y(case, packed, sp)
    b = _y(case, packed, sp)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- fp16 route of 4-bit codes
def _scaled_x(xb, factors):
    """bf16 bit patterns of x[t] * factors[t] (fp32 product rounded to bf16)."""
    xf = (xb.astype(np.uint32) << 16).view(np.float32)
    return synth._f32_to_bf16_bits(xf * np.asarray(factors, np.float32)[:, None])


def _x_edge_cases(xb):
    T = xb.shape[0]
    tiny = xb.copy()
    tiny[T - 1, 70] = np.uint16(np.float32(2.0 ** -40).view(np.uint32) >> 16)  # ~53 binades down
    zero = xb.copy()
    zero[0] = 0                                                              # an all-zero token
    return {
        "tiny_element": tiny,                                # the CTA falls back to bf16
        "huge": _scaled_x(xb, [2.0 ** 110] * T),             # max above 2^101: bf16 route
        "subnormal_scale": _scaled_x(xb, [2.0 ** -118] * T),  # max below 2^-100: bf16 route
        "token_scales": _scaled_x(xb, [2.0 ** (40 * t - 30) for t in range(T)]),
        "zero_token": zero,
    }


def _check_x(case, packed, sp, xb, name):
    c = dict(case, xb=xb)
    y = _y(c, packed, sp, route=nqp.ROUTE_MMA)
    assert np.isfinite(y).all(), name
    codes, sb = oracle_inputs(c)
    y_ref, e_ref = oracle.gemv(codes, sb, xb)
    v = oracle.max_violation(y, y_ref, e_ref)
    assert v <= 1.0, (name, v)
    return y


@pytest.mark.parametrize("T", [1, 2])
def test_q4_f16_route_x_edge_cases(T):
    """4-bit codes with x in registers at T <= 2 go through fp16 when every x
    converts exactly after a per-token power-of-two scaling, else through
    bf16; both must meet the oracle's tolerance whatever x looks like."""
    case = rtn_case((314, T), 4, 100, 1024, T)
    packed, sp = device_weight(nqp, torch, case, DEV)
    assert nqp.plan(1024, 100, T, 4)["ksplit"] == 1
    for name, xb in _x_edge_cases(case["xb"]).items():
        _check_x(case, packed, sp, xb, name)


@pytest.mark.parametrize("ksplit", [2, 4])
@pytest.mark.parametrize("T", [1, 2])
def test_q4_f16_route_with_k_split(T, ksplit):
    """The fp16 route of 4-bit codes inside K-split clusters (the route the
    4-bit down projections of the stack take at T <= 2): every x edge case
    against the oracle, with the cluster's partial sums exchanged."""
    case = rtn_case((316, T, ksplit), 4, 300, 4096, T)
    packed, sp = device_weight(nqp, torch, case, DEV)
    assert nqp.plan(4096, 300, T, 4, route=nqp.ROUTE_MMA, ksplit=ksplit)["ksplit"] == ksplit
    for name, xb in _x_edge_cases(case["xb"]).items():
        c = dict(case, xb=xb)
        y = _y(c, packed, sp, route=nqp.ROUTE_MMA, ksplit=ksplit)
        assert np.isfinite(y).all(), name
        codes, sb = oracle_inputs(c)
        y_ref, e_ref = oracle.gemv(codes, sb, xb)
        v = oracle.max_violation(y, y_ref, e_ref)
        assert v <= 1.0, (name, v)


@pytest.mark.parametrize("T", [1, 2])
def test_q4_f16_and_bf16_routes_agree(T, monkeypatch):
    """The same product through the fp16 route (default at T <= 2) and through
    the bf16 route (NQ_X_F16=0): both within the oracle's tolerance, and
    one-hot x gives the weight column exactly on both."""
    case = rtn_case((315, T), 4, 2000, 5120, T)
    packed, sp = device_weight(nqp, torch, case, DEV)
    y16 = _check_x(case, packed, sp, case["xb"], "fp16 route")
    monkeypatch.setenv("NQ_X_F16", "0")
    ybf = _check_x(case, packed, sp, case["xb"], "bf16 route")
    monkeypatch.delenv("NQ_X_F16")
    codes, sb = oracle_inputs(case)
    _, e_ref = oracle.gemv(codes, sb, case["xb"])
    assert np.all(np.abs(y16 - ybf) <= 2e-4 * e_ref + 2e-6)
    wref = oracle.dequant_f32(codes, sb)
    xb = np.zeros((T, 5120), np.uint16)
    for t in range(T):
        xb[t, 777 + 1000 * t] = 0x3F80
    for env in ("1", "0"):
        monkeypatch.setenv("NQ_X_F16", env)
        y = _y(dict(case, xb=xb), packed, sp)
        for t in range(T):
            assert np.array_equal(y[t], wref[:, 777 + 1000 * t]), (env, t)
    monkeypatch.delenv("NQ_X_F16")


def test_gemv_right_after_device_pack():
    """A GEMV launched directly after nq_pack_device on the same stream (no
    other launch between them) reads the freshly packed weights: the library
    launches that GEMV without programmatic dependent launch.  x and y are
    prepared before the packing so that nothing else runs in between."""
    for bits in (4, 5):
        case = uniform_case((317, bits), bits, 600, 2048, 3)
        codes, sb = oracle_inputs(case)
        dcodes = torch.from_numpy(codes).to(DEV)
        dsb = torch.from_numpy(sb.view(np.int16)).to(DEV)
        cb, sbytes = nqp.packed_bytes(case["K"], case["N"], bits)
        packed = torch.zeros(cb, dtype=torch.uint8, device=DEV)     # stale contents: zeros
        sp = torch.zeros(sbytes // 2, dtype=torch.int16, device=DEV)
        x = device_x(torch, case, DEV)
        y = torch.full((3, case["N"]), float("nan"), dtype=torch.float32, device=DEV)
        torch.cuda.synchronize()
        nqp.pack_device(dcodes, dsb, bits, packed=packed, scales_packed=sp)
        nqp.gemv(packed, sp, x, y, case["K"], case["N"], 3, bits)
        assert nqp.last_device_error() == 0
        y_ref, e_ref = oracle.gemv(codes, sb, case["xb"])
        assert oracle.max_violation(y.cpu().numpy(), y_ref, e_ref) <= 1.0


# ---------------------------------------------------------------- errors and edge cases
def test_invalid_arguments():
    case = rtn_case((311,), 4, 32, 128, 2)
    packed, sp = device_weight(nqp, torch, case, DEV)
    x = device_x(torch, case, DEV)
    y = torch.empty((2, 32), dtype=torch.float32, device=DEV)
    bad = [dict(T=0), dict(T=17), dict(route=nqp.ROUTE_FFMA, T=5), dict(ksplit=3), dict(route=9),
           dict(K=100), dict(bits=7), dict(bits=8, route=nqp.ROUTE_FFMA)]
    for kw in bad:
        args = dict(K=128, N=32, T=2, bits=4, route=0, ksplit=0)
        args.update(kw)
        with pytest.raises(nqp.NQError) as e:
            nqp.gemv(packed, sp, x, y, args["K"], args["N"], args["T"], args["bits"],
                     route=args["route"], ksplit=args["ksplit"])
        assert e.value.code == nqp.EINVAL, kw
    xbuf = torch.zeros(2 * 128 + 8, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nqp.NQError) as e:
        nqp.gemv(packed, sp, xbuf[1:], y, 128, 32, 2, 4)
    assert e.value.code == nqp.EALIGN
    with pytest.raises(nqp.NQError) as e:
        nqp.plan(262144, 64, 16, 4)
    assert e.value.code == nqp.EUNSUPPORTED
    assert nqp.last_device_error() == 0


def test_bounded_wait_times_out_and_context_survives():
    nqp.selftest_wait_timeout(50_000)
    assert nqp.last_device_error() == nqp.ETIMEOUT
    case = rtn_case((312,), 4, 64, 256, 1)
    packed, sp = device_weight(nqp, torch, case, DEV)
    _check(case, _y(case, packed, sp))


def test_max_t_long_k():
    case = uniform_case((313,), 5, 96, 17408, 16)
    packed, sp = device_weight(nqp, torch, case, DEV)
    p = nqp.plan(17408, 96, 16, 5)
    assert p["ksplit"] >= 4
    _check(case, _y(case, packed, sp))


# ---------------------------------------------------------------- full-size shapes, sampled rows
FULL = {
    "gate_up_q4": ("rtn", 4, 34816, 5120, [1], 0.0),
    "down_q5": ("uniform", 5, 5120, 17408, [1, 8], 0.01),
    # the 4-bit down projections of layers 36-63 of the 64-layer stack
    "down_q4": ("rtn", 4, 5120, 17408, [1, 2, 4, 8, 16], 0.0),
    "head_q6": ("rtn", 6, 248320, 5120, [1, 2, 4, 8], 0.0),
    "down_q8": ("rtn", 8, 5120, 17408, [1, 8, 16], 0.0),
}
SAMPLE_ROWS = 384


@pytest.fixture(scope="module")
def full_cases():
    """Full-size weights built once per module: device tensors, plus the
    oracle's inputs for a sample of rows."""
    out = {}
    for name, (kind, bits, N, K, Ts, outl) in FULL.items():
        mk = rtn_case if kind == "rtn" else uniform_case
        case = mk((400, bits), bits, N, K, 16, outlier_frac=outl)
        packed, sp = device_weight(nqp, torch, case, DEV)
        rng = np.random.default_rng(7)
        rows = np.unique(np.concatenate([[0, 1, 15, 16, N // 2, N - 17, N - 1],
                                         rng.choice(N, SAMPLE_ROWS, replace=False)]))
        sub = dict(case, w=case["w"][rows])
        if kind == "uniform":
            sub["flips"] = case["flips"][rows]
            sub["codes"] = case["codes"][rows]
        codes, sb = oracle_inputs(sub)
        del case["w"]
        out[name] = {"case": case, "packed": packed, "sp": sp, "rows": rows, "codes": codes,
                     "sb": sb, "Ts": Ts}
    return out


def _check_rows(fc, y, T):
    y_ref, e_ref = oracle.gemv(fc["codes"], fc["sb"], fc["case"]["xb"][:T])
    v = oracle.max_violation(y[:, fc["rows"]], y_ref, e_ref)
    assert v <= 1.0, (T, v)
    assert np.isfinite(y).all()


@pytest.mark.slow
@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled(full_cases, name):
    fc = full_cases[name]
    case = fc["case"]
    K, N, bits = case["K"], case["N"], case["bits"]
    # dequant of the sampled rows is bit-exact
    wd = nqp.dequant(fc["packed"], fc["sp"], K, N, bits)
    assert np.array_equal(wd[torch.from_numpy(fc["rows"]).to(DEV)].cpu().numpy().view(np.uint32),
                          oracle.dequant_f32(fc["codes"], fc["sb"]).view(np.uint32))
    del wd
    for t in fc["Ts"]:
        _check_rows(fc, _y(case, fc["packed"], fc["sp"], T=t), t)


@pytest.mark.slow
def test_full_size_graph_launch_path(full_cases):
    """The launch configuration the benchmark times: back-to-back GEMVs of the
    full-size shapes at T = 1, 8, 16 on a side stream, captured into one
    CUDA graph (programmatic dependent launch between the kernels), replayed
    twice; sampled rows of every output against the oracle, and the two
    replays bitwise equal."""
    stream = torch.cuda.Stream(device=DEV)
    jobs = []
    for name in FULL:
        fc = full_cases[name]
        case = fc["case"]
        x16 = device_x(torch, case, DEV)
        for T in (1, 8, 16):
            y = torch.full((T, case["N"]), float("nan"), dtype=torch.float32, device=DEV)
            jobs.append((fc, x16[:T].contiguous(), y, T))

    def run():
        for fc, x, y, T in jobs:
            c = fc["case"]
            nqp.gemv(fc["packed"], fc["sp"], x, y, c["K"], c["N"], T, c["bits"], stream=stream)

    with torch.cuda.stream(stream):
        run()                      # plans and kernel attributes set before capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    outs = []
    for _ in range(2):
        for _, _, y, _ in jobs:
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        assert nqp.last_device_error() == 0
        outs.append([y.cpu().numpy() for _, _, y, _ in jobs])
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
    for (fc, _, _, T), y in zip(jobs, outs[0]):
        _check_rows(fc, y, T)
