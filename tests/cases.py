"""Workload cases shared by the GPU tests: each case keeps only the raw
random draws from ``synth``; the oracle side and the CUDA side each turn them
into codes and scales with their own encoder."""
from __future__ import annotations

import numpy as np

import oracle
import synth


def rtn_case(tag, bits, N, K, T, outlier_frac=0.0, seed=0):
    """Weights N(0, 0.02) to be round-to-nearest encoded; x N(0,1) bf16."""
    rng = synth.generator(seed, *tag)
    w = synth.gauss_weights(rng, N, K)
    outl = synth.outlier_channels(rng, K, outlier_frac) if outlier_frac else None
    xb = synth.gauss_x_bf16(rng, T, K, outliers=outl)
    return {"kind": "rtn", "bits": bits, "N": N, "K": K, "T": T, "w": w, "xb": xb}


def uniform_case(tag, bits, N, K, T, outlier_frac=0.01, seed=0):
    """Down-projection style: scales = absmax/qmax of a N(0, 0.02) draw with the
    sign flipped on a random half of the groups, codes uniform over the full
    range, x N(0,1) with outlier channels x20."""
    rng = synth.generator(seed, *tag)
    w = synth.gauss_weights(rng, N, K)
    flips = synth.sign_flips(rng, N, K // 64)
    codes = synth.uniform_codes(rng, N, K, bits)
    outl = synth.outlier_channels(rng, K, outlier_frac) if outlier_frac else None
    xb = synth.gauss_x_bf16(rng, T, K, outliers=outl)
    return {"kind": "uniform", "bits": bits, "N": N, "K": K, "T": T, "w": w, "flips": flips,
            "codes": codes, "xb": xb}


def oracle_inputs(case, rows=None):
    """(codes, scale bits) on the oracle side, optionally for a subset of rows."""
    sl = slice(None) if rows is None else rows
    bits = case["bits"]
    if case["kind"] == "rtn":
        return oracle.rtn_encode(case["w"][sl], bits)
    s = oracle.rtn_scales(case["w"][sl], oracle.QMAX[bits])
    s = s ^ (case["flips"][sl].astype(np.uint16) << 15)
    return case["codes"][sl], s


def device_weight(nqp, torch, case, dev):
    """(packed, packed scales) built on the device with the library's encoder
    and packer."""
    bits = case["bits"]
    w = torch.from_numpy(case["w"]).to(dev)
    codes, scales = nqp.quantize_rtn(w, bits)
    del w
    if case["kind"] == "uniform":
        flips = torch.from_numpy(case["flips"]).to(dev)
        scales = torch.where(flips, scales ^ torch.tensor(-32768, dtype=torch.int16, device=dev),
                             scales)
        codes = torch.from_numpy(case["codes"]).to(dev)
    return nqp.pack_device(codes, scales, bits)


def device_x(torch, case, dev):
    return torch.from_numpy(case["xb"].view(np.int16)).to(dev).view(torch.bfloat16)


# Fused head (argmax / maximum / logsumexp) against the kernel's own logits:
# argmax and maximum exact, logsumexp within 4e-5 + 1e-6 |lse| of the fp64
# logsumexp of those logits (fp32 running sums, merged in a fixed order).
LSE_ABS, LSE_REL = 4e-5, 1e-6


def lse64(y):
    y = y.astype(np.float64)
    m = y.max(axis=1)
    return m + np.log(np.exp(y - m[:, None]).sum(axis=1))


def head_check_self(y, am, mx, lse):
    """argmax / max / lse against the kernel's own logits."""
    T = y.shape[0]
    ref_am = np.argmax(y, axis=1)
    assert np.array_equal(am, ref_am), (am, ref_am)
    assert np.array_equal(mx.view(np.uint32), y[np.arange(T), am].view(np.uint32))
    ref = lse64(y)
    assert np.all(np.abs(lse - ref) <= LSE_ABS + LSE_REL * np.abs(ref)), (lse, ref)
