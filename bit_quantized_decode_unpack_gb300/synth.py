"""Seeded synthetic inputs for the quantized matrix-vector product.

This module draws raw inputs only -- integer codes, fp16 scales, fp16 biases
and fp16 activations -- and holds none of the method's arithmetic (no packing,
no decoding, no dequantisation).  Both the CUDA path and the float64 oracle are
fed from it; each packs the codes with its own packer.

Distributions (27B-class decoder layer, synthetic stand-ins for trained
weights, which this library never needs):

* codes: 1-bit uniform {0,1}; 2-bit uniform {0..3}; t5 trits with
  P(0) = P(2) = 0.3, P(1) = 0.4;
* scale = |N(0, 0.02)| + 1e-3, rounded to fp16;
* bias = -scale * U(0.3, 0.7) for 1-bit, -scale * U(1, 2) for 2-bit (formed
  in float32, rounded to fp16); t5 and the sym variants carry no bias tensor;
* x ~ N(0, 1), rounded to fp16.

Host generators use ``numpy.random.default_rng(seed)``; the device generators
(for the large rotating weight sets of the benchmark) draw the same
distributions with a seeded ``torch.Generator`` on the GPU.
"""
from __future__ import annotations

import zlib

import numpy as np

FMT_AFFINE1 = 1
FMT_AFFINE2 = 2
FMT_T5 = 3

T5_PROBS = (0.3, 0.4, 0.3)
BIAS_RANGE = {FMT_AFFINE1: (0.3, 0.7), FMT_AFFINE2: (1.0, 2.0)}

#: projection shapes (N, K) of a 27B-class dense decoder layer
LAYER_SHAPES = {
    "q_proj": (6144, 5120),
    "k_proj": (1024, 5120),
    "v_proj": (1024, 5120),
    "o_proj": (5120, 6144),
    "gate_proj": (17408, 5120),
    "up_proj": (17408, 5120),
    "down_proj": (5120, 17408),
}


def seed_for(key: str) -> int:
    """Seed 0 for the small 1-bit case, a stable CRC of the key otherwise."""
    return 0 if key == "affine1_m1_256x512_gs64" else zlib.crc32(key.encode())


def rng_for(key: str) -> np.random.Generator:
    return np.random.default_rng(seed_for(key))


def codes(rng: np.random.Generator, fmt: int, N: int, K: int) -> np.ndarray:
    if fmt == FMT_AFFINE1:
        return rng.integers(0, 2, size=(N, K), dtype=np.uint8)
    if fmt == FMT_AFFINE2:
        return rng.integers(0, 4, size=(N, K), dtype=np.uint8)
    if fmt == FMT_T5:
        return rng.choice(3, size=(N, K), p=T5_PROBS).astype(np.uint8)
    raise ValueError(f"unknown format {fmt}")


def scales(rng: np.random.Generator, N: int, G: int) -> np.ndarray:
    return (np.abs(rng.normal(0.0, 0.02, size=(N, G))) + 1e-3).astype(np.float16)


def biases(rng: np.random.Generator, fmt: int, s: np.ndarray):
    """Asymmetric bias tensor, or None for t5 (no bias tensor)."""
    if fmt == FMT_T5:
        return None
    lo, hi = BIAS_RANGE[fmt]
    u = rng.uniform(lo, hi, size=s.shape).astype(np.float32)
    return (-(s.astype(np.float32) * u)).astype(np.float16)


def activations(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    return rng.normal(0.0, 1.0, size=(M, K)).astype(np.float16)


def problem(fmt: int, M: int, N: int, K: int, gs: int, sym: bool = False,
            key: str | None = None) -> dict:
    """One seeded problem: x [M,K], codes [N,K], scales [N,G], biases|None."""
    key = key or f"fmt{fmt}_m{M}_{N}x{K}_gs{gs}_{'sym' if sym else 'asym'}"
    rng = rng_for(key)
    c = codes(rng, fmt, N, K)
    s = scales(rng, N, K // gs)
    b = None if sym else biases(rng, fmt, s)
    x = activations(rng, M, K)
    return {"x": x, "codes": c, "scales": s, "biases": b, "fmt": fmt, "gs": gs,
            "M": M, "N": N, "K": K, "sym": sym or fmt == FMT_T5, "key": key}


# ---- device-side draws (same distributions) for large weight sets ----------

def torch_codes(gen, fmt: int, N: int, K: int, device):
    import torch
    if fmt == FMT_AFFINE1:
        return torch.randint(0, 2, (N, K), generator=gen, device=device, dtype=torch.uint8)
    if fmt == FMT_AFFINE2:
        return torch.randint(0, 4, (N, K), generator=gen, device=device, dtype=torch.uint8)
    u = torch.rand((N, K), generator=gen, device=device)
    return ((u >= T5_PROBS[0]).to(torch.uint8) + (u >= T5_PROBS[0] + T5_PROBS[1]).to(torch.uint8))


def torch_scales(gen, N: int, G: int, device):
    import torch
    return (torch.randn((N, G), generator=gen, device=device).abs_() * 0.02 + 1e-3).to(torch.float16)


def torch_biases(gen, fmt: int, s, device):
    import torch
    if fmt == FMT_T5:
        return None
    lo, hi = BIAS_RANGE[fmt]
    u = torch.rand(s.shape, generator=gen, device=device) * (hi - lo) + lo
    return (-(s.float() * u)).to(torch.float16)


def torch_activations(gen, M: int, K: int, device):
    import torch
    return torch.randn((M, K), generator=gen, device=device).to(torch.float16)
