"""GPU checks of the fused head's top-k (nq_gemv_head_topk) through the C ABI.

Bars: the top k (indices and values) equal the oracle's head_topk of the
kernel's own logits exactly (selection only: no arithmetic beyond the
logits); argmax, maximum and logsumexp meet nq_gemv_head's bars;
against the oracle's fp64 logits, the j-th returned value is within the
largest output tolerance of the true j-th largest logit (order statistics are
1-Lipschitz in the largest output error), and every returned row's true logit
is within twice that tolerance of the true k-th largest."""
import numpy as np
import pytest
import torch

import oracle
import quantized_weight_decode_gb300 as nqp
from cases import device_weight, device_x, head_check_self, oracle_inputs, rtn_case, uniform_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def built():
    nqp.build()
    nqp.lib()
    torch.cuda.set_device(0)
    assert nqp.last_device_error() == 0


def _topk(case, packed, sp, k, store_y=True, ws=None):
    T, K, N, bits = case["T"], case["K"], case["N"], case["bits"]
    x = device_x(torch, case, DEV)[:T].contiguous()
    y = torch.full((T, N), float("nan"), dtype=torch.float32, device=DEV) if store_y else None
    out = nqp.gemv_head_topk(packed, sp, x, K, N, T, bits, k, y=y, workspace=ws)
    assert nqp.last_device_error() == 0
    out = [o.cpu().numpy() for o in out]
    return (None if y is None else y.cpu().numpy()), out


def _check_self(y, k, idx, val):
    ref_idx, ref_val = oracle.head_topk(y, k)
    assert np.array_equal(idx, ref_idx), (idx, ref_idx)
    assert np.array_equal(val.view(np.uint32), ref_val.astype(np.float32).view(np.uint32))


def _check_oracle(case, k, idx, val, rows=None):
    codes, sb = oracle_inputs(case, rows)
    y_ref, e_ref = oracle.gemv(codes, sb, case["xb"][: case["T"]])
    tol = (oracle.REL_TOL * e_ref + oracle.ABS_TOL).max(axis=1)
    n = min(k, y_ref.shape[1])
    srt = -np.sort(-y_ref, axis=1)[:, :n]
    assert np.all(np.abs(val[:, :n] - srt) <= tol[:, None]), (val, srt)
    if rows is None:
        true = np.take_along_axis(y_ref, idx[:, :n].astype(np.int64), axis=1)
        assert np.all(true >= srt[:, -1:] - 2 * tol[:, None])
    assert np.all(idx[:, n:] == -1) and np.all(np.isneginf(val[:, n:]))


SHAPES = [(6, 1024, 1000), (6, 512, 17), (4, 2048, 300), (5, 1024, 1), (8, 1024, 700),
          (5, 17408, 100)]   # the last one runs as clusters of 4 CTAs (K split)


@pytest.mark.parametrize("T", [1, 2, 5, 8, 9, 12, 16])
def test_topk_matches_own_logits_and_oracle(T):
    for i, (bits, K, N) in enumerate(SHAPES):
        case = rtn_case((520, T, i), bits, N, K, T)
        packed, sp = device_weight(nqp, torch, case, DEV)
        for k in (1, 5, 32):
            y, (idx, val, am, mx, lse) = _topk(case, packed, sp, k)
            _check_self(y, k, idx, val)
            # argmax / maximum / logsumexp as nq_gemv_head's bars (the launch
            # plan, and so the fp32 reduction order, may differ from that call's)
            head_check_self(y, am, mx, lse)
            assert np.array_equal(idx[:, 0], am)
            _check_oracle(case, k, idx, val)


def test_topk_reduce_scatter_k_split():
    """The top-k of the kernel that finalises by reduce-scatter (6-bit, K =
    5120, T = 16, both token blocks in registers at K split 2): one list per CTA and
    epilogue warp, merged; against the kernel's own logits and the oracle."""
    K, N, bits, T = 5120, 16 * 187 + 7, 6, 16
    assert (nqp.plan(K, N, T, bits)["x"], nqp.plan(K, N, T, bits)["ksplit"]) == ("regs2", 2)
    case = rtn_case((521, T), bits, N, K, T)
    packed, sp = device_weight(nqp, torch, case, DEV)
    for k in (1, 8, 32):
        y, (idx, val, am, mx, lse) = _topk(case, packed, sp, k)
        _check_self(y, k, idx, val)
        head_check_self(y, am, mx, lse)
        assert np.array_equal(idx[:, 0], am)
        _check_oracle(case, k, idx, val)


def test_topk_without_logits_and_repeat_calls():
    case = uniform_case((521,), 5, 3000, 2048, 8)
    packed, sp = device_weight(nqp, torch, case, DEV)
    ws = torch.empty(nqp.head_topk_workspace_bytes(), dtype=torch.uint8, device=DEV)
    y, (idx, val, *_) = _topk(case, packed, sp, 16, ws=ws)
    _check_self(y, 16, idx, val)
    for _ in range(2):      # no logits stored; the workspace carries over between calls
        _, (idx2, val2, *_) = _topk(case, packed, sp, 16, store_y=False, ws=ws)
        assert np.array_equal(idx, idx2)
        assert np.array_equal(val.view(np.uint32), val2.view(np.uint32))


def test_topk_ties_go_to_the_smallest_rows():
    T, K, N, bits = 3, 1024, 2000, 6
    case = rtn_case((522,), bits, N, K, T)
    codes, sb = oracle_inputs(case)
    codes, sb = codes.copy(), sb.copy()
    big = oracle.f64_to_fp16_bits(np.array([1.0]))[0]
    tied = [1999, 37, 1500, 38, 150, 0, 801]     # seven identical rows, the largest logits
    for r in tied:
        codes[r] = 31
        sb[r] = big
    hp, hs = nqp.pack(codes, sb, bits)
    packed = torch.from_numpy(hp).to(DEV)
    sp = torch.from_numpy(hs.view(np.int16)).to(DEV)
    c2 = dict(case, xb=np.full((T, K), 0x3F80, np.uint16))   # x = 1
    y, (idx, val, *_) = _topk(c2, packed, sp, 10)
    assert idx[:, :7].tolist() == [sorted(tied)] * T
    assert np.all(val[:, :7] == 31.0 * K)
    _check_self(y, 10, idx, val)


def test_topk_argument_errors():
    case = rtn_case((523,), 4, 64, 256, 1)
    packed, sp = device_weight(nqp, torch, case, DEV)
    x = device_x(torch, case, DEV)[:1].contiguous()
    for k in (0, 33, -1):
        with pytest.raises(nqp.NQError) as e:
            nqp.gemv_head_topk(packed, sp, x, 256, 64, 1, 4, k)
        assert e.value.code == nqp.EINVAL
    small = torch.empty(nqp.head_topk_workspace_bytes() - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(nqp.NQError) as e:
        nqp.gemv_head_topk(packed, sp, x, 256, 64, 1, 4, 8, workspace=small)
    assert e.value.code == nqp.EINVAL
    assert nqp.head_topk_workspace_bytes() > nqp.head_workspace_bytes()
    assert nqp.last_device_error() == 0


@pytest.mark.slow
@pytest.mark.parametrize("T,k", [(1, 32), (8, 8)])
def test_topk_full_size_head(T, k):
    """The 248,320-row 6-bit output head: top-k against the kernel's own logits
    (all rows), the returned rows' logits against the oracle."""
    K, N, bits = 5120, 248320, 6
    case = rtn_case((524, T), bits, N, K, T)
    packed, sp = device_weight(nqp, torch, case, DEV)
    y, (idx, val, am, *_) = _topk(case, packed, sp, k)
    _check_self(y, k, idx, val)
    rows = np.unique(idx.ravel())
    codes, sb = oracle_inputs(case, rows)
    y_ref, e_ref = oracle.gemv(codes, sb, case["xb"][:T])
    assert oracle.max_violation(y[:, rows], y_ref, e_ref) <= 1.0
