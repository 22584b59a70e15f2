"""Reference for the W4A4 NVFP4 GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this module.

"LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation" (summary
page), training step 4: the GEMMs run in NVFP4 with 2-D block scales for weights and
1-D block scales for activations; inference step 6: a W4A4 model.  What a W4A4 GEMM
computes, written out: every operand element is its E2M1 value times its block's E4M3
scale (exact in binary64), the product of the two dequantized matrices is summed in
binary64, and the result is multiplied by the two fp32 tensor scales.  The decoders
are the oracle's own (``e2m1_decode``, ``e4m3_decode``), pinned elsewhere; the matrix
product is numpy's, a library primitive.
"""
from __future__ import annotations

import numpy as np

from . import e2m1_decode, e4m3_decode

_E2M1 = None
_E4M3 = None


def _tables():
    global _E2M1, _E4M3
    if _E2M1 is None:
        _E2M1 = np.array([e2m1_decode(c) for c in range(16)], dtype=np.float64)
        _E4M3 = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return _E2M1, _E4M3


def _values(codes: np.ndarray) -> np.ndarray:
    """Packed codes [R][K/2] -> E2M1 values [R][K] (element 2j = low nibble of byte j)."""
    e2m1, _ = _tables()
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty((c.shape[0], 2 * c.shape[1]), dtype=np.float64)
    out[:, 0::2] = e2m1[c & 0xF]
    out[:, 1::2] = e2m1[c >> 4]
    return out


def dequant_1d(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Activation operand: codes [M][K/2], 1-D block scales [M][K/16] -> exact values [M][K]."""
    _, e4m3 = _tables()
    v = _values(codes)
    s = e4m3[np.asarray(scales, dtype=np.uint8)]
    return v * np.repeat(s, 16, axis=1)


def dequant_2d(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Weight operand: codes [N][K/2], 16x16 tile scales [N/16][K/16] -> exact values [N][K]."""
    _, e4m3 = _tables()
    v = _values(codes)
    s = e4m3[np.asarray(scales, dtype=np.uint8)]
    return v * np.repeat(np.repeat(s, 16, axis=0), 16, axis=1)


def gemm_w4a4(x_codes, x_scales, x_g: float, w_codes, w_scales, w_g: float):
    """(Y, |Y|-bound): Y[m][n] = gX gW sum_k X[m][k] W[n][k] in binary64, and
    gX gW sum_k |X[m][k] W[n][k]| (the scale of the rounding error of any fp32 summation)."""
    X = dequant_1d(x_codes, x_scales)
    Wv = dequant_2d(w_codes, w_scales)
    g = float(x_g) * float(w_g)
    return (X @ Wv.T) * g, (np.abs(X) @ np.abs(Wv).T) * abs(g)


def rht16(x: np.ndarray, signs: int) -> np.ndarray:
    """The GEMM path's random Hadamard transform along the rows, in fp32, step by step:
    each block of 16 elements has element i negated where bit i of ``signs`` is set, then
    the radix-2 Walsh-Hadamard butterflies with strides 1, 2, 4, 8 replace each pair (a, b)
    by (fl(a + b), fl(a - b)), and the result is multiplied by 1/4."""
    v = np.array(x, dtype=np.float32, copy=True)
    rows, K = v.shape
    b = v.reshape(rows, K // 16, 16)
    for i in range(16):
        if (signs >> i) & 1:
            b[:, :, i] = -b[:, :, i]
    h = 1
    while h < 16:
        for i in range(16):
            if i & h == 0:
                a, c = b[:, :, i].copy(), b[:, :, i + h].copy()
                b[:, :, i] = a + c
                b[:, :, i + h] = a - c
        h *= 2
    return (b * np.float32(0.25)).reshape(rows, K)
