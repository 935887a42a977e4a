"""Seeded synthetic inputs shared by the tests, the bench and smoke().

This module holds no arithmetic of the method: it draws fp32 weights and fp32
activations from numpy's PCG64 generator and casts activations to bf16 with
torch's own conversion.  Quantizing the weights is done by whichever side needs
them (the oracle for parity inputs, the library for bench inputs).

Recipe (the pages measure on served models and name no dataset; these stand in
for the projection weights and decode activations of those models):
  - W[N, K] fp32 ~ N(0, 0.02), PCG64(seed).
  - X[n, K] fp32 ~ N(0, 1), PCG64(seed); optionally each entry is an outlier with
    probability ``outlier_frac`` (independent Bernoulli mask) and is multiplied
    by ``outlier_scale`` before the bf16 cast.
  - bf16 values are returned as their uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np
import torch

# Shapes of the projection workloads (output rows N, reduction K, token counts).
WORKLOADS = {
    "tiny": dict(N=256, K=512, ns=(3,), outlier_frac=0.0),
    "attn_qkv": dict(N=14336, K=5120, ns=(1, 2, 3, 4), outlier_frac=0.0),
    "o_proj": dict(N=5120, K=6144, ns=(8,), outlier_frac=0.01),
    "fused_qkv": dict(N=16384, K=5120, ns=(16,), outlier_frac=0.0),
}


def weights_f32(N: int, K: int, seed: int, std: float = 0.02) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.standard_normal((N, K), dtype=np.float32) * np.float32(std)


def activations_f32(n: int, K: int, seed: int, outlier_frac: float = 0.0,
                    outlier_scale: float = 20.0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((n, K), dtype=np.float32)
    if outlier_frac > 0.0:
        mask = rng.random((n, K)) < outlier_frac
        x = np.where(mask, x * np.float32(outlier_scale), x).astype(np.float32)
    return x


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (torch's round-to-nearest-even cast), returned as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def activations_bf16(n: int, K: int, seed: int, outlier_frac: float = 0.0,
                     outlier_scale: float = 20.0) -> np.ndarray:
    return to_bf16_bits(activations_f32(n, K, seed, outlier_frac, outlier_scale))
