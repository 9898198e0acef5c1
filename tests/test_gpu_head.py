"""GPU checks of the fused verify head (nq_gemv_head): argmax, maximum and
logsumexp of every token's outputs, through the C ABI.

Bars: the logits equal nq_gemv's bit for bit; argmax / maximum are exact with
respect to the kernel's own logits (first index of the maximum); logsumexp
is within 4e-5 + 1e-6 |lse| of the fp64 logsumexp of those logits (fp32
running sums over up to a few hundred values per lane, merged in a fixed
order); against the oracle, the argmax is a valid one (its true logit is
within the two outputs' tolerances of the true maximum) and logsumexp is
within the largest output tolerance (logsumexp is 1-Lipschitz in the largest
output error) plus the same 4e-5."""
import numpy as np
import pytest
import torch

import oracle
import quantized_weight_decode_gb300 as nqp
from cases import (LSE_ABS, LSE_REL, device_weight, device_x, head_check_self, oracle_inputs,
                   rtn_case, uniform_case)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def built():
    nqp.build()
    nqp.lib()
    torch.cuda.set_device(0)
    assert nqp.last_device_error() == 0


def _head(case, packed, sp, store_y=True, ws=None):
    T, K, N, bits = case["T"], case["K"], case["N"], case["bits"]
    x = device_x(torch, case, DEV)[:T].contiguous()
    y = torch.full((T, N), float("nan"), dtype=torch.float32, device=DEV) if store_y else None
    am, mx, lse = nqp.gemv_head(packed, sp, x, K, N, T, bits, y=y, workspace=ws)
    assert nqp.last_device_error() == 0
    return (None if y is None else y.cpu().numpy()), am.cpu().numpy(), mx.cpu().numpy(), lse.cpu().numpy()


def _check_oracle(case, am, mx, lse, rows=None):
    codes, sb = oracle_inputs(case)
    y_ref, e_ref = oracle.gemv(codes, sb, case["xb"][: case["T"]])
    tol = oracle.REL_TOL * e_ref + oracle.ABS_TOL
    a_ref, m_ref, l_ref = oracle.head_reduce(y_ref)
    T = y_ref.shape[0]
    t = np.arange(T)
    # the chosen row is a maximum within the two tolerances
    assert np.all(y_ref[t, am] >= m_ref - tol[t, am] - tol[t, a_ref]), (am, a_ref)
    assert np.all(np.abs(mx - y_ref[t, am]) <= tol[t, am])
    assert np.all(np.abs(lse - l_ref) <= tol.max(axis=1) + LSE_ABS + LSE_REL * np.abs(l_ref))


SHAPES = [(6, 1024, 1000), (6, 512, 17), (4, 2048, 300), (5, 1024, 1), (6, 17408 // 4, 160),
          (5, 17408, 100)]   # the last one runs as clusters of 4 CTAs (K split)


# T = 5 and 12: the second value slot of a hand-off is partly filled (the K
# split's reduce-scatter sends it to rank 1 for some lanes only)
@pytest.mark.parametrize("T", [1, 2, 3, 5, 8, 9, 12, 15, 16])
def test_head_matches_gemv_and_oracle(T):
    for i, (bits, K, N) in enumerate(SHAPES):
        case = rtn_case((500, T, i), bits, N, K, T)
        packed, sp = device_weight(nqp, torch, case, DEV)
        if K == 17408:
            assert nqp.plan(K, N, T, bits)["ksplit"] > 1
        y, am, mx, lse = _head(case, packed, sp)
        # logits identical to the plain GEMV
        x = device_x(torch, case, DEV)[:T].contiguous()
        y2 = torch.full((T, N), float("nan"), dtype=torch.float32, device=DEV)
        nqp.gemv(packed, sp, x, y2, K, N, T, bits)
        assert np.array_equal(y.view(np.uint32), y2.cpu().numpy().view(np.uint32))
        head_check_self(y, am, mx, lse)
        _check_oracle(case, am, mx, lse)


def test_head_without_logits_and_repeat_calls():
    case = uniform_case((501,), 5, 777, 2048, 8)
    packed, sp = device_weight(nqp, torch, case, DEV)
    ws = torch.empty(nqp.head_workspace_bytes(), dtype=torch.uint8, device=DEV)
    y, am, mx, lse = _head(case, packed, sp, ws=ws)
    for _ in range(2):      # no logits stored; the workspace carries over between calls
        _, am2, mx2, lse2 = _head(case, packed, sp, store_y=False, ws=ws)
        assert np.array_equal(am, am2)
        assert np.array_equal(mx.view(np.uint32), mx2.view(np.uint32))
        assert np.array_equal(lse.view(np.uint32), lse2.view(np.uint32))
    head_check_self(y, am, mx, lse)


def test_head_ties_go_to_the_smallest_row():
    T, K, N, bits = 2, 1024, 300, 6
    case = rtn_case((502,), bits, N, K, T)
    codes, sb = oracle_inputs(case)
    codes, sb = codes.copy(), sb.copy()
    big = oracle.f64_to_fp16_bits(np.array([1.0]))[0]
    for r in (37, 150, 299, 38):          # four identical rows with large positive weights
        codes[r] = 31
        sb[r] = big
    hp, hs = nqp.pack(codes, sb, bits)
    packed = torch.from_numpy(hp).to(DEV)
    sp = torch.from_numpy(hs.view(np.int16)).to(DEV)
    xb = np.full((T, K), 0x3F80, np.uint16)   # x = 1: those rows give 31 K, every other less
    c2 = dict(case, xb=xb)
    y, am, mx, _ = _head(c2, packed, sp)
    assert am.tolist() == [37, 37]
    assert np.all(y[:, [37, 38, 150, 299]] == y[:, [37]])
    assert np.all(mx == 31.0 * K)


@pytest.mark.parametrize("ksplit_rows", [(6, 256, 16 * 400), (5, 17408, 16 * 40)])
def test_head_infinite_logits(ksplit_rows):
    """Token 0 has x = +inf on one channel where every row's code is +1 or -1,
    so its logits are +inf on a few rows spread over several CTAs (and
    clusters) and -inf elsewhere: argmax is the first +inf row, the maximum
    and logsumexp are +inf (merging two +inf states must not form inf - inf).
    Token 1 is ordinary and must be unaffected."""
    bits, K, N = ksplit_rows
    rng = np.random.default_rng(77)
    lo, hi = oracle.code_range(bits)
    codes = rng.integers(lo, hi + 1, (N, K)).astype(np.int8)
    plus = [37, N // 2 + 3, N - 1]
    codes[:, 5] = -1
    codes[plus, 5] = 1
    sb = oracle.rtn_scales(rng.standard_normal((N, K)).astype(np.float32) * 0.02, oracle.QMAX[bits])
    hp, hs = nqp.pack(codes, sb, bits)
    packed, sp = torch.from_numpy(hp).to(DEV), torch.from_numpy(hs.view(np.int16)).to(DEV)
    xb = ((rng.standard_normal((2, K)).astype(np.float32).view(np.uint32) >> 16)).astype(np.uint16)
    xb[0, 5] = 0x7F80                                    # +inf
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    am, mx, lse = nqp.gemv_head(packed, sp, x, K, N, 2, bits)
    assert nqp.last_device_error() == 0
    am, mx, lse = am.cpu().numpy(), mx.cpu().numpy(), lse.cpu().numpy()
    y_ref, e_ref = oracle.gemv(codes, sb, xb)
    a_ref, m_ref, l_ref = oracle.head_reduce(y_ref)
    assert a_ref[0] == plus[0] and m_ref[0] == np.inf and l_ref[0] == np.inf
    assert am[0] == plus[0] and mx[0] == np.inf and lse[0] == np.inf
    tol = oracle.REL_TOL * e_ref[1] + oracle.ABS_TOL
    assert y_ref[1, am[1]] >= m_ref[1] - tol[am[1]] - tol[a_ref[1]]
    assert abs(mx[1] - y_ref[1, am[1]]) <= tol[am[1]]
    assert abs(lse[1] - l_ref[1]) <= tol.max() + LSE_ABS + LSE_REL * abs(l_ref[1])


def test_head_workspace_errors():
    case = rtn_case((503,), 4, 64, 256, 1)
    packed, sp = device_weight(nqp, torch, case, DEV)
    x = device_x(torch, case, DEV)[:1].contiguous()
    out = [torch.empty(1, dtype=torch.int32, device=DEV)] + \
          [torch.empty(1, dtype=torch.float32, device=DEV) for _ in range(2)]
    small = torch.empty(nqp.head_workspace_bytes() - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(nqp.NQError) as e:
        nqp.gemv_head(packed, sp, x, 256, 64, 1, 4, workspace=small, argmax=out[0], maxval=out[1],
                      lse=out[2])
    assert e.value.code == nqp.EINVAL
    big = torch.empty(nqp.head_workspace_bytes() + 64, dtype=torch.uint8, device=DEV)
    with pytest.raises(nqp.NQError) as e:
        nqp.gemv_head(packed, sp, x, 256, 64, 1, 4, workspace=big[8:], argmax=out[0],
                      maxval=out[1], lse=out[2])
    assert e.value.code == nqp.EALIGN
    assert nqp.last_device_error() == 0


def test_head_reduce_scatter_k_split():
    """6-bit codes, K = 5120, T = 16: both token blocks in registers at K
    split 2, the kernel whose epilogue finalises by reduce-scatter (each rank
    of a cluster takes a slot of every hand-off and publishes its own
    states).  Fused results against the kernel's own logits, logits against
    the oracle, and argmax / maximum against the plain GEMV's logits."""
    K, N, bits, T = 5120, 16 * 187 + 7, 6, 16   # (at T = 15 the hybrid still fits)
    p = nqp.plan(K, N, T, bits)
    assert (p["x"], p["ksplit"]) == ("regs2", 2), p
    case = rtn_case((506, T), bits, N, K, T)
    packed, sp = device_weight(nqp, torch, case, DEV)
    y, am, mx, lse = _head(case, packed, sp)
    head_check_self(y, am, mx, lse)
    _check_oracle(case, am, mx, lse)
    x = device_x(torch, case, DEV)[:T].contiguous()
    y2 = torch.full((T, N), float("nan"), dtype=torch.float32, device=DEV)
    nqp.gemv(packed, sp, x, y2, K, N, T, bits)
    assert np.array_equal(y2.cpu().numpy().view(np.uint32), y.view(np.uint32))
    _, am2, mx2, lse2 = _head(case, packed, sp, store_y=False)
    assert np.array_equal(am, am2) and np.array_equal(mx.view(np.uint32), mx2.view(np.uint32))
    assert np.array_equal(lse.view(np.uint32), lse2.view(np.uint32))


def test_head_reduce_scatter_in_graph():
    """The reduce-scatter head and its top-k captured into one CUDA graph and
    replayed twice (the exchange barriers' phases and the arrival counters
    carry over between replays): bitwise the eager calls' results."""
    K, N, bits, T = 5120, 16 * 131 + 3, 6, 16
    case = rtn_case((507,), bits, N, K, T)
    packed, sp = device_weight(nqp, torch, case, DEV)
    x = device_x(torch, case, DEV)[:T].contiguous()
    ws = torch.empty(nqp.head_topk_workspace_bytes(), dtype=torch.uint8, device=DEV)
    outs = [torch.empty(T, dtype=dt, device=DEV) for dt in (torch.int32, torch.float32, torch.float32)]
    tki = torch.empty((T, 8), dtype=torch.int32, device=DEV)
    tkv = torch.empty((T, 8), dtype=torch.float32, device=DEV)
    stream = torch.cuda.Stream(device=DEV)

    def run():
        nqp.gemv_head_topk(packed, sp, x, K, N, T, bits, 8, workspace=ws, topk_idx=tki,
                           topk_val=tkv, argmax=outs[0], maxval=outs[1], lse=outs[2],
                           stream=stream)
    with torch.cuda.stream(stream):
        run()
    stream.synchronize()
    ref = [o.clone() for o in outs] + [tki.clone(), tkv.clone()]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    for _ in range(2):
        for o in outs + [tki, tkv]:
            o.fill_(0)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        assert nqp.last_device_error() == 0
        for a, b in zip(ref, outs + [tki, tkv]):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    _, am, mx, lse = _head(case, packed, sp)
    assert np.array_equal(am, ref[0].cpu().numpy())
    assert np.array_equal(tki.cpu().numpy()[:, 0], am)


@pytest.mark.slow
@pytest.mark.parametrize("T", [1, 8, 16])
def test_head_full_size(T):
    """The 248,320-row 6-bit output head: fused results against the kernel's own
    logits (all rows), and the logits of sampled rows against the oracle."""
    K, N, bits = 5120, 248320, 6
    case = rtn_case((504, T), bits, N, K, T)
    packed, sp = device_weight(nqp, torch, case, DEV)
    y, am, mx, lse = _head(case, packed, sp)
    head_check_self(y, am, mx, lse)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([am, rng.choice(N, 256, replace=False)]))
    codes, sb = oracle_inputs(case, rows)
    y_ref, e_ref = oracle.gemv(codes, sb, case["xb"][:T])
    assert oracle.max_violation(y[:, rows], y_ref, e_ref) <= 1.0


@pytest.mark.slow
@pytest.mark.parametrize("bits,T", [(4, 8), (6, 1), (8, 2)])
def test_head_proposal_head_shape(bits, T):
    """The 131,072-row proposal head (K = 5120): fused results against the
    kernel's own logits, logits of sampled rows against the oracle."""
    K, N = 5120, 131072
    case = rtn_case((505, bits, T), bits, N, K, T)
    packed, sp = device_weight(nqp, torch, case, DEV)
    y, am, mx, lse = _head(case, packed, sp)
    head_check_self(y, am, mx, lse)
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([am, rng.choice(N, 256, replace=False)]))
    codes, sb = oracle_inputs(case, rows)
    y_ref, e_ref = oracle.gemv(codes, sb, case["xb"][:T])
    assert oracle.max_violation(y[:, rows], y_ref, e_ref) <= 1.0
