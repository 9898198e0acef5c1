"""The fused verify head through the entry point that allocates nothing
(nq_gemv_head_noalloc), for callers that cannot allocate device memory
themselves -- a library embedded in a runtime that owns every device
allocation, or a loop where a cudaMalloc / cudaFree would synchronise the
device.  It must give what nq_gemv_head gives with a caller workspace, on two
calls in a row (the second finds the first call's contents in the shared
scratch).  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import quantized_weight_decode_gb300 as nqp
from cases import LSE_ABS, LSE_REL, device_weight, device_x, rtn_case, uniform_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def built():
    nqp.build()
    nqp.lib()
    torch.cuda.set_device(0)
    assert nqp.last_device_error() == 0


def _both(case, packed, sp, T):
    K, N, bits = case["K"], case["N"], case["bits"]
    x = device_x(torch, case, DEV)[:T].contiguous()
    ya = torch.empty((T, N), dtype=torch.float32, device=DEV)
    yb = torch.empty((T, N), dtype=torch.float32, device=DEV)
    ref = nqp.gemv_head(packed, sp, x, K, N, T, bits, y=ya)
    got = nqp.gemv_head_noalloc(packed, sp, x, K, N, T, bits, y=yb)
    assert nqp.last_device_error() == 0
    return [t.cpu().numpy() for t in (ya, *ref)], [t.cpu().numpy() for t in (yb, *got)]


def _same(ref, got):
    (ya, am_a, mx_a, lse_a), (yb, am_b, mx_b, lse_b) = ref, got
    assert np.array_equal(ya.view(np.uint32), yb.view(np.uint32))
    assert np.array_equal(am_a, am_b)
    assert np.array_equal(mx_a.view(np.uint32), mx_b.view(np.uint32))
    assert np.all(np.abs(lse_a - lse_b) <= LSE_ABS + LSE_REL * np.abs(lse_a))


def test_noalloc_head_matches_workspace_head_on_two_calls_in_a_row():
    # first call: 6-bit head-like shape, 8 tokens; second: a K-split shape,
    # 3 tokens, on the scratch the first call left behind
    c1 = rtn_case((600,), 6, 3000, 5120, 8)
    p1, s1 = device_weight(nqp, torch, c1, DEV)
    c2 = uniform_case((601,), 5, 200, 17408, 3)
    p2, s2 = device_weight(nqp, torch, c2, DEV)
    for case, packed, sp, T in ((c1, p1, s1, 8), (c2, p2, s2, 3)):
        ref, got = _both(case, packed, sp, T)
        _same(ref, got)
    # and the same inputs again, back to back on the shared scratch
    for _ in range(2):
        ref, got = _both(c1, p1, s1, 8)
        _same(ref, got)


def test_noalloc_scratch_size_is_enough_for_this_device():
    assert nqp.head_workspace_bytes() <= 139520
