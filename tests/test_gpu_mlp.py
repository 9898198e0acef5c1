"""GPU checks of the decoder-layer MLP path through the C ABI: the gate+up
product with SwiGLU in its epilogue (nq_gemv_swiglu) and the layer
(nq_mlp = SwiGLU product, then the down projection).

Tolerances, derived from the GEMV bound tol = 1e-4 E + 1e-6 of each output:
act = bf16(silu(g) u) differs from the oracle's bf16(silu(g*) u*) by at most
|silu'(g) u| tol_g + |silu(g)| tol_u (first order; plus 1e-6 relative for the
fp32 silu) and one bf16 step (each side rounds once); the layer's output then
differs by the down product's own bound plus sum_k |w_k| (act error)_k."""
import numpy as np
import pytest
import torch

import oracle
import quantized_weight_decode_gb300 as nqp
import synth
from cases import oracle_inputs, rtn_case, uniform_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def built():
    nqp.build()
    nqp.lib()
    torch.cuda.set_device(0)
    assert nqp.last_device_error() == 0


def _upload(codes, sb, bits):
    hp, hs = nqp.pack(codes, sb, bits)
    return torch.from_numpy(hp).to(DEV), torch.from_numpy(hs.view(np.int16)).to(DEV)


def _act_tolerance(g, u, e_g, e_u):
    tol_g = oracle.REL_TOL * e_g + oracle.ABS_TOL
    tol_u = oracle.REL_TOL * e_u + oracle.ABS_TOL
    sig = 1.0 / (1.0 + np.exp(-np.clip(g, -700, 700)))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    silu = g * sig
    val = np.abs(silu * u)
    step = np.ldexp(1.0, np.frexp(np.maximum(val, 2.0 ** -126))[1] - 8)   # one bf16 step at val
    return np.abs(dsilu * u) * tol_g + np.abs(silu) * tol_u + 1e-6 * val + step + 1e-30


def _gate_up_case(tag, bits, I, H, T):
    """Gate and up weights (RTN codes), their interleaved packing, x."""
    rng = synth.generator(0, *tag)
    wg = synth.gauss_weights(rng, I, H)
    wu = synth.gauss_weights(rng, I, H)
    xb = synth.gauss_x_bf16(rng, T, H)
    cg, sg = oracle.rtn_encode(wg, bits)
    cu, su = oracle.rtn_encode(wu, bits)
    packed, sp = _upload(nqp.interleave_gate_up(cg, cu), nqp.interleave_gate_up(sg, su), bits)
    return cg, sg, cu, su, xb, packed, sp


def _check_act(act_bits, cg, sg, cu, su, xb, cd=None, sd=None):
    """act against oracle.mlp (gate+up in (gate; up) row order); with down
    weights, also returns the oracle's layer output and its error scale."""
    if cd is None:                      # no down product: a zero matrix of K = I
        cd = np.zeros((16, cg.shape[0]), np.int8)
        sd = np.zeros((16, cg.shape[0] // 64), np.uint16)
    act_ref, y_ref, e_ref, g, u, e_g, e_u = oracle.mlp(
        np.concatenate([cg, cu]), np.concatenate([sg, su]), cd, sd, xb)
    ref = oracle.bf16_to_f64(act_ref)
    got = oracle.bf16_to_f64(act_bits)
    tol = _act_tolerance(g, u, e_g, e_u)
    assert np.all(np.abs(got - ref) <= tol), np.max(np.abs(got - ref) / tol)
    return tol, y_ref, e_ref


@pytest.mark.parametrize("bits,T", [(4, 1), (4, 2), (4, 8), (5, 3), (6, 16), (8, 4)])
def test_swiglu_product(bits, T):
    I, H = 1000 // 8 * 8, 1024
    cg, sg, cu, su, xb, packed, sp = _gate_up_case((700, bits, T), bits, I, H, T)
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    act = torch.full((T, I), -1, dtype=torch.int16, device=DEV)
    nqp.gemv_swiglu(packed, sp, x, act, H, 2 * I, T, bits)
    assert nqp.last_device_error() == 0
    _check_act(act.cpu().numpy().view(np.uint16), cg, sg, cu, su, xb)


def test_swiglu_rejects_ragged_rows():
    cg, sg, cu, su, xb, packed, sp = _gate_up_case((701,), 4, 64, 256, 1)
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    act = torch.empty((1, 64), dtype=torch.int16, device=DEV)
    with pytest.raises(nqp.NQError) as e:
        nqp.gemv_swiglu(packed, sp, x, act, 256, 120, 1, 4)        # 120 rows: not a multiple of 16
    assert e.value.code == nqp.EINVAL


def _check_layer(I, H, Hout, bits_gu, bits_down, T, tag):
    cg, sg, cu, su, xb, packed, sp = _gate_up_case(tag, bits_gu, I, H, T)
    rng = synth.generator(0, *tag, 9)
    wd = synth.gauss_weights(rng, Hout, I)
    cd, sd = oracle.rtn_encode(wd, bits_down)
    pd, spd = _upload(cd, sd, bits_down)
    gu = nqp.QuantizedWeight(packed, sp, H, 2 * I, bits_gu)
    down = nqp.QuantizedWeight(pd, spd, I, Hout, bits_down)
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    act = torch.empty((T, I), dtype=torch.int16, device=DEV)
    y = torch.full((T, Hout), float("nan"), dtype=torch.float32, device=DEV)
    nqp.mlp(gu, down, x, act, y, T)
    assert nqp.last_device_error() == 0
    tol_act, y_ref, e_ref = _check_act(act.cpu().numpy().view(np.uint16), cg, sg, cu, su, xb, cd, sd)
    w_abs = np.abs(oracle.dequant(cd, sd))
    bound = oracle.REL_TOL * e_ref + oracle.ABS_TOL + tol_act @ w_abs.T
    err = np.abs(y.cpu().numpy() - y_ref)
    assert np.all(err <= bound), np.max(err / bound)


@pytest.mark.parametrize("T", [1, 4, 8])
def test_mlp_layer(T):
    _check_layer(I=1024, H=512, Hout=384, bits_gu=4, bits_down=5, T=T, tag=(702, T))


@pytest.mark.parametrize("bits_gu,bits_down,T", [(8, 8, 2), (6, 4, 16)])
def test_mlp_layer_other_widths(bits_gu, bits_down, T):
    _check_layer(I=1024, H=512, Hout=384, bits_gu=bits_gu, bits_down=bits_down, T=T,
                 tag=(704, bits_gu, bits_down, T))


@pytest.mark.slow
def test_mlp_layer_full_size():
    """Qwen3.8-27B-shaped layer: gate+up 5120 -> 2 x 17408 (4-bit), down
    17408 -> 5120 (5-bit), one token."""
    _check_layer(I=17408, H=5120, Hout=5120, bits_gu=4, bits_down=5, T=1, tag=(703,))
