"""Seeded synthetic inputs shaped like the LongLive-2.0 KV-cache workload.

This module draws random numbers and nothing else: it holds none of the
quantizer's arithmetic, and both the CUDA path's tests/benchmark and the CPU
oracle take their inputs from it.  All draws use numpy's PCG64
(``default_rng(seed)``); bf16 inputs are the fp32 draws rounded by torch's
fp32->bf16 cast.

Shapes follow the LongLive-2.0 summary page, inference step 7 (a chunk is
F_c = 8 latent frames x L_f tokens per frame) with a Wan2.2-TI2V-5B-like
attention geometry (24 heads x head_dim 128, L_f = 880).  The pages print no
KV statistics; the laws below are stated assumptions:
  * K = per-(head, channel) offset + N(0, 1) noise, a few whole channels
    scaled up (outlier channels, the reason K-smoothing exists);
  * V ~ N(0, 1);
  * weights ~ N(0, 0.02^2) with 0.1% of entries x30; activations ~ N(0, 1).
"""
from __future__ import annotations

import numpy as np

FRAMES_PER_CHUNK = 8
TOKENS_PER_FRAME = 880
HEADS = 24
HEAD_DIM = 128
CHUNK_TOKENS = FRAMES_PER_CHUNK * TOKENS_PER_FRAME  # 7040


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (torch's round-to-nearest-even cast); returns uint16 bit patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def tiny_kv(seed: int = 0):
    """Tiny oracle-check chunk: 2 frames x 32 tokens, 1 head, head_dim 64, fp32.

    K[t, c] = offset[c] + N(0,1), offset ~ N(0, 2^2); 1% of the elements (41)
    replaced by 20 * N(0,1) outliers.  V ~ N(0,1).  K then V from one stream.
    Returns float32 arrays of shape [64, 1, 64].
    """
    T, H, D = 64, 1, 64
    rng = np.random.default_rng(seed)
    off = rng.normal(0.0, 2.0, size=D)
    K = off[None, :] + rng.standard_normal((T, D))
    n_out = int(round(0.01 * T * D))
    pos = rng.choice(T * D, size=n_out, replace=False)
    K.reshape(-1)[pos] = 20.0 * rng.standard_normal(n_out)
    V = rng.standard_normal((T, D))
    return K.astype(np.float32).reshape(T, H, D), V.astype(np.float32).reshape(T, H, D)


def chunk_k(seed: int, T: int = CHUNK_TOKENS, H: int = HEADS, D: int = HEAD_DIM,
            outlier_frac: float = 0.005, outlier_gain: float = 16.0) -> np.ndarray:
    """K of one chunk, fp32 [T, H, D]: offset[h,d] ~ N(0, 3^2) + N(0,1); whole outlier channels x16."""
    rng = np.random.default_rng(seed)
    off = rng.normal(0.0, 3.0, size=(H, D)).astype(np.float32)
    K = rng.standard_normal((T, H, D), dtype=np.float32)
    K += off[None]
    n_ch = int(round(outlier_frac * H * D))
    ch = rng.choice(H * D, size=n_ch, replace=False)
    Kf = K.reshape(T, H * D)
    Kf[:, ch] *= np.float32(outlier_gain)
    return K


def chunk_v(seed: int, T: int = CHUNK_TOKENS, H: int = HEADS, D: int = HEAD_DIM) -> np.ndarray:
    """V of one chunk, fp32 [T, H, D] ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((T, H, D), dtype=np.float32)


def chunk_kv_bf16(seed_k: int = 2000, seed_v: int = 2001, T: int = CHUNK_TOKENS, H: int = HEADS,
                  D: int = HEAD_DIM):
    """One layer, one chunk (7040 x 24 x 128 by default) as bf16 bit patterns: (K, V)."""
    return to_bf16_bits(chunk_k(seed_k, T, H, D)), to_bf16_bits(chunk_v(seed_v, T, H, D))


def layer_seeds(layer: int):
    """Per-layer seeds of the full-model chunk write: K 3000 + 2l, V 3001 + 2l."""
    return 3000 + 2 * layer, 3001 + 2 * layer


def weight(i: int, M: int, N: int, seed_base: int = 5000) -> np.ndarray:
    """A Wan-like linear weight, fp32 [M, N] ~ N(0, 0.02^2) with 0.1% entries x30 (seed 5000 + i)."""
    rng = np.random.default_rng(seed_base + i)
    W = rng.standard_normal((M, N), dtype=np.float32) * np.float32(0.02)
    n_out = int(round(0.001 * M * N))
    pos = rng.choice(M * N, size=n_out, replace=False)
    W.reshape(-1)[pos] *= np.float32(30.0)
    return W


WEIGHT_SHAPES = [(3072, 3072)] * 4 + [(3072, 14336)] * 2


def activations(T: int = CHUNK_TOKENS, D: int = 3072, seed: int = 5100) -> np.ndarray:
    """Activation matrix fp32 [T, D] ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((T, D), dtype=np.float32)


def random_kv(seed: int, T: int, H: int, D: int, scale: float = 1.0, offset_sd: float = 3.0) -> np.ndarray:
    """Generic seeded [T, H, D] fp32 tensor with per-channel offsets, for shape sweeps."""
    rng = np.random.default_rng(seed)
    off = rng.normal(0.0, offset_sd, size=(H, D)).astype(np.float32)
    X = rng.standard_normal((T, H, D), dtype=np.float32) * np.float32(scale)
    X += off[None]
    return X
