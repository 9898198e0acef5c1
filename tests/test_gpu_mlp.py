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
    I = cg.shape[0]
    if cd is None:
        # no down product: zero rows pad gate and up to a multiple of 64 (their
        # activations are 0) and a zero down matrix takes the padded act
        pad = -I % 64
        z = lambda a: np.concatenate([a, np.zeros((pad,) + a.shape[1:], a.dtype)])
        cg, sg, cu, su = z(cg), z(sg), z(cu), z(su)
        cd = np.zeros((16, I + pad), np.int8)
        sd = np.zeros((16, (I + pad) // 64), np.uint16)
    act_ref, y_ref, e_ref, g, u, e_g, e_u = oracle.mlp(
        np.concatenate([cg, cu]), np.concatenate([sg, su]), cd, sd, xb)
    act_ref, g, u, e_g, e_u = (a[:, :I] for a in (act_ref, g, u, e_g, e_u))
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


def _check_layer(I, H, Hout, bits_gu, bits_down, T, tag, launches=None):
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
    if launches == 1:
        assert nqp.mlp_one_launch_ok(H, I, Hout, T, bits_gu, bits_down)
    nqp.mlp(gu, down, x, act, y, T, launches=launches or 0)
    assert nqp.last_device_error() == 0
    tol_act, y_ref, e_ref = _check_act(act.cpu().numpy().view(np.uint16), cg, sg, cu, su, xb, cd, sd)
    w_abs = np.abs(oracle.dequant(cd, sd))
    bound = oracle.REL_TOL * e_ref + oracle.ABS_TOL + tol_act @ w_abs.T
    err = np.abs(y.cpu().numpy() - y_ref)
    assert np.all(err <= bound), np.max(err / bound)
    return gu, down, x, act, y


@pytest.mark.parametrize("T", [1, 4, 8])
def test_mlp_layer(T):
    _check_layer(I=1024, H=512, Hout=384, bits_gu=4, bits_down=5, T=T, tag=(702, T))


@pytest.mark.parametrize("bits_gu,bits_down,T", [(8, 8, 2), (6, 4, 16)])
def test_mlp_layer_other_widths(bits_gu, bits_down, T):
    _check_layer(I=1024, H=512, Hout=384, bits_gu=bits_gu, bits_down=bits_down, T=T,
                 tag=(704, bits_gu, bits_down, T))


@pytest.mark.slow
@pytest.mark.parametrize("bits_down,T", [(5, 1), (4, 2), (5, 8)])
def test_mlp_layer_full_size(bits_down, T):
    """Qwen3.8-27B-shaped layer: gate+up 5120 -> 2 x 17408 (4-bit), down
    17408 -> 5120 (5-bit for layers 0-35, 4-bit for 36-63), in one launch."""
    _check_layer(I=17408, H=5120, Hout=5120, bits_gu=4, bits_down=bits_down, T=T,
                 tag=(703, bits_down, T), launches=1)
    _check_layer(I=17408, H=5120, Hout=5120, bits_gu=4, bits_down=bits_down, T=T,
                 tag=(703, bits_down, T), launches=2)


@pytest.mark.parametrize("bits_gu,bits_down,T,I", [(4, 5, 1, 8704), (4, 5, 2, 8704), (4, 5, 4, 8704),
                                                   (4, 5, 8, 8704), (4, 4, 3, 8704), (6, 4, 8, 8704),
                                                   (8, 8, 2, 8704), (4, 5, 1, 4352), (4, 5, 2, 4352),
                                                   (4, 4, 2, 4352)])
def test_mlp_one_launch_matches_two_launches(bits_gu, bits_down, T, I):
    """The one-launch layer (gate+up phase publishing its activations, the down
    phase in the same kernel) against the oracle, and bit for bit against the
    two-launch path (the same products in the same order).  I = 8704: the
    down product takes a K split of 2; I = 4352: no split, and the gate+up
    phase has so few tiles per CTA that the down phase's first stages reach
    the shared-memory area where the gate+up phase staged x in fp16 (T <= 2),
    which must wait until that x has been taken."""
    H, Hout = 1024, 600
    gu, down, x, act, y = _check_layer(I=I, H=H, Hout=Hout, bits_gu=bits_gu, bits_down=bits_down,
                                       T=T, tag=(705, bits_gu, bits_down, T, I), launches=1)
    act2 = torch.empty_like(act)
    y2 = torch.full_like(y, float("nan"))
    nqp.mlp(gu, down, x, act2, y2, T, launches=2)
    assert nqp.last_device_error() == 0
    assert torch.equal(act, act2)
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


def test_mlp_one_launch_limits():
    """The one-launch kernel's limits: T <= 8, gate+up K <= 5120, the
    instantiated width pairs; outside them nq_mlp_ex(launches=1) is
    NQ_EUNSUPPORTED and the default (two launches) still runs."""
    assert nqp.mlp_one_launch_ok(5120, 17408, 5120, 8, 4, 5)
    assert not nqp.mlp_one_launch_ok(5120, 17408, 5120, 9, 4, 5)
    assert not nqp.mlp_one_launch_ok(6144, 1024, 512, 1, 4, 5)
    assert not nqp.mlp_one_launch_ok(1024, 1024, 512, 1, 5, 6)
    cg, sg, cu, su, xb, packed, sp = _gate_up_case((707,), 5, 1024, 512, 1)
    gu = nqp.QuantizedWeight(packed, sp, 512, 2048, 5)
    cd = np.zeros((64, 1024), np.int8)
    sd = np.zeros((64, 16), np.uint16)
    pd, spd = _upload(cd, sd, 6)
    down = nqp.QuantizedWeight(pd, spd, 1024, 64, 6)
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    act = torch.empty((1, 1024), dtype=torch.int16, device=DEV)
    y = torch.empty((1, 64), dtype=torch.float32, device=DEV)
    with pytest.raises(nqp.NQError) as e:
        nqp.mlp(gu, down, x, act, y, 1, launches=1)
    assert e.value.code == nqp.EUNSUPPORTED
    nqp.mlp(gu, down, x, act, y, 1)
    assert nqp.last_device_error() == 0
    assert np.all(y.cpu().numpy() == 0)


def test_mlp_one_launch_repeat_and_graph():
    """Ten one-launch layers back to back on a stream, then the same ten
    captured in a CUDA graph and replayed twice: every output equals the
    first eager result bit for bit (the per-launch activation counters are
    reset by each launch)."""
    I, H, Hout, T = 4352, 1024, 600, 2
    gu, down, x, act, y = _check_layer(I=I, H=H, Hout=Hout, bits_gu=4, bits_down=5, T=T,
                                       tag=(706,), launches=1)
    ref_act, ref_y = act.clone(), y.clone()
    acts = [torch.empty_like(act) for _ in range(10)]
    ys = [torch.full_like(y, float("nan")) for _ in range(10)]
    st = torch.cuda.Stream(device=DEV)
    def run():
        for a2, y2 in zip(acts, ys):
            nqp.mlp(gu, down, x, a2, y2, T, launches=1, stream=st)
    with torch.cuda.stream(st):
        run()
    st.synchronize()
    assert nqp.last_device_error() == 0
    for a2, y2 in zip(acts, ys):
        assert torch.equal(a2, ref_act) and torch.equal(y2, ref_y)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        run()
    for _ in range(2):
        for y2 in ys:
            y2.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            g.replay()
        st.synchronize()
        assert nqp.last_device_error() == 0
        for a2, y2 in zip(acts, ys):
            assert torch.equal(a2, ref_act) and torch.equal(y2, ref_y)
