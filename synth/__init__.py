"""Seeded synthetic inputs for the groupwise-quantized small-T GEMV.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no scale rule, no rounding to codes, no dequantisation,
no products).  Both the CPU oracle and the CUDA path take their inputs from
here, each side then applies the method by itself.

The workloads follow the shapes of a 64-layer Qwen3.8-27B-like model
(hidden 5120, intermediate 17408, vocabulary 248,320), stated on the model
card of the groupwise-int artifact ("Qwen3.8-27B for NInfer on the RTX 3090",
section "What is different from the upstream artifact") and on the ninfer-ext
model page ("Qwen3.8-27B EXL3", section "Model"):

* weights ~ N(0, 0.02) in fp32, later round-to-nearest quantised per 64-group;
* activations x ~ N(0, 1), rounded to bf16 (round to nearest even);
* for the down projection: 1 % of the input channels scaled by 20 before the
  bf16 rounding, codes drawn uniformly over the full signed range and the
  sign of a random half of the group scales flipped.

Every draw comes from a ``numpy.random.Generator`` whose seed is the tuple
(seed, config id, layer, role), so any tensor can be regenerated on its own.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "ROLE", "generator", "gauss_weights", "gauss_x_bf16", "uniform_codes",
    "sign_flips", "outlier_channels", "torch_generator",
]

# Stable integer ids of the tensor roles, used in seed tuples.
ROLE = {"gate_up": 1, "down": 2, "head": 3, "x": 4, "codes": 5, "flip": 6,
        "outliers": 7, "tiny": 8, "misc": 9}


def generator(seed: int = 0, *path: int) -> np.random.Generator:
    """Independent PCG64 stream for (seed, *path)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *path])))


def gauss_weights(rng: np.random.Generator, n: int, k: int, sigma: float = 0.02,
                  chunk_rows: int = 4096) -> np.ndarray:
    """fp32 weights W[n, k] ~ N(0, sigma^2), row-major."""
    out = np.empty((n, k), dtype=np.float32)
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        out[r0:r1] = rng.standard_normal((r1 - r0, k), dtype=np.float32)
        out[r0:r1] *= np.float32(sigma)
    return out


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the raw 16-bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def outlier_channels(rng: np.random.Generator, k: int, frac: float = 0.01) -> np.ndarray:
    """round(frac*k) distinct channel indices, sorted."""
    m = int(round(frac * k))
    return np.sort(rng.choice(k, size=m, replace=False)).astype(np.int64)


def gauss_x_bf16(rng: np.random.Generator, t: int, k: int, outliers: np.ndarray | None = None,
                 outlier_mult: float = 20.0) -> np.ndarray:
    """Activations x[t, k]: N(0,1) fp32, optional outlier channels scaled (in fp32),
    then rounded to bf16.  Returned as uint16 bit patterns."""
    x = rng.standard_normal((t, k), dtype=np.float32)
    if outliers is not None and len(outliers):
        x[:, outliers] *= np.float32(outlier_mult)
    return _f32_to_bf16_bits(x)


def uniform_codes(rng: np.random.Generator, n: int, k: int, bits: int) -> np.ndarray:
    """Signed integer codes uniform over [-2^(bits-1), 2^(bits-1) - 1], int8 [n, k]."""
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
    return rng.integers(lo, hi + 1, size=(n, k), dtype=np.int8)


def sign_flips(rng: np.random.Generator, n: int, groups: int, p: float = 0.5) -> np.ndarray:
    """Boolean mask [n, groups]: True where a group's scale sign is flipped."""
    return rng.random((n, groups)) < p


def torch_generator(seed: int, device):
    """Seeded torch generator on `device`, for drawing large tensors in place
    (used where host generation of many gigabytes would dominate run time)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def imatrix(rng: np.random.Generator, k: int, tokens: int = 64, outlier_frac: float = 0.01,
            outlier_mult: float = 20.0) -> np.ndarray:
    """A synthetic importance matrix: per channel, the mean squared value of
    `tokens` activation draws N(0, 1) with a fraction of outlier channels
    scaled by `outlier_mult` (fp32 [k]).  Stands in for an imatrix gathered
    from calibration text."""
    x = rng.standard_normal((tokens, k), dtype=np.float32)
    n_out = int(round(outlier_frac * k))
    if n_out:
        x[:, rng.choice(k, n_out, replace=False)] *= np.float32(outlier_mult)
    return np.mean(x.astype(np.float64) ** 2, axis=0).astype(np.float32)
