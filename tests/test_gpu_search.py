"""GPU checks of the searched encoder (nq_quantize_search) through the C ABI:
codes and FP16 scales bit for bit equal to the oracle's search_encode (the
choice is made in fp64 with the same operation order on both sides), with and
without an importance matrix, on random and on structured groups; and the GEMV
on search-encoded weights against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import quantized_weight_decode_gb300 as nqp
import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def built():
    nqp.build()
    nqp.lib()
    torch.cuda.set_device(0)
    assert nqp.last_device_error() == 0


def _device_search(w, bits, imp):
    wd = torch.from_numpy(w).to(DEV)
    qd = None if imp is None else torch.from_numpy(imp).to(DEV)
    c, s = nqp.quantize_search(wd, bits, qd)
    rc = nqp.last_device_error()
    return c.cpu().numpy(), s.cpu().numpy().view(np.uint16), rc


def _structured(rng, k):
    """Rows of 64-weight groups that exercise the decision: exact groups that
    need a negative / a positive scale, an all-zero group, tiny weights (FP16
    subnormal scales), a group near the FP16 limit, one dominant channel."""
    rows = []
    step = np.float32(2.0 ** -7)
    rows.append(np.tile(((np.arange(64) % 16) - 7) * step, k // 64))       # needs -step
    rows.append(np.tile(((np.arange(64) % 16) - 8) * step, k // 64))       # +step exact
    rows.append(np.zeros(k, np.float32))
    rows.append(synth.gauss_weights(rng, 1, k)[0] * np.float32(1e-5))      # subnormal scales
    rows.append(synth.gauss_weights(rng, 1, k)[0] * np.float32(4.0e5))     # near the FP16 limit
    r = synth.gauss_weights(rng, 1, k)[0]
    r[::64] *= np.float32(40.0)
    rows.append(r)
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_search_bit_exact(bits):
    rng = synth.generator(0, 910, bits)
    K = 1024
    w = np.concatenate([synth.gauss_weights(rng, 97, K), _structured(rng, K)])
    q = synth.imatrix(rng, K)
    for imp in (None, q):
        c, s, rc = _device_search(w, bits, imp)
        assert rc == 0
        c_ref, s_ref = oracle.search_encode(w, bits, imp)
        assert np.array_equal(s, s_ref), np.argwhere(s != s_ref)[:5]
        assert np.array_equal(c, c_ref)
    assert np.any(s_ref >> 15)            # some negative scales were chosen


def test_search_overflow_sets_status():
    w = np.full((16, 64), 7.0e5, np.float32)
    _, _, rc = _device_search(w, 4, None)
    assert rc == nqp.ERANGE
    assert nqp.last_device_error() == 0


@pytest.mark.parametrize("bits,T", [(4, 1), (5, 8), (6, 3), (8, 2)])
def test_gemv_on_search_encoded_weights(bits, T):
    rng = synth.generator(0, 911, bits)
    N, K = 300, 2048
    w = synth.gauss_weights(rng, N, K)
    q = synth.imatrix(rng, K)
    xb = synth.gauss_x_bf16(rng, T, K)
    codes, scales, rc = _device_search(w, bits, q)
    assert rc == 0
    packed, sp = nqp.pack_device(torch.from_numpy(codes).to(DEV),
                                 torch.from_numpy(scales.view(np.int16)).to(DEV), bits)
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    y = torch.full((T, N), float("nan"), dtype=torch.float32, device=DEV)
    nqp.gemv(packed, sp, x, y, K, N, T, bits)
    assert nqp.last_device_error() == 0
    c_ref, s_ref = oracle.search_encode(w, bits, q)
    y_ref, e_ref = oracle.gemv(c_ref, s_ref, xb)
    assert oracle.max_violation(y.cpu().numpy(), y_ref, e_ref) <= 1.0
