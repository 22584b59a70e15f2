"""Reference for attention over the NVFP4 KV cache -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this module.

"LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation" (summary
page), inference steps 7 and 9: attention reads the NVFP4 KV cache over the sinks and
the rolling frames.  Written out: every view token's K and V channels are dequantized
in fp32 exactly as the cache read defines them (S = fl(E g), value = fl(Q S), K's mean
added with one more rounding), then softmax(scale q . k) v is evaluated in binary64.
The decoders are the oracle's own (pinned elsewhere).
"""
from __future__ import annotations

import numpy as np

from . import e2m1_decode, e4m3_decode

_T = None


def _tables():
    global _T
    if _T is None:
        _T = (np.array([e2m1_decode(c) for c in range(16)], dtype=np.float32),
              np.array([e4m3_decode(c) for c in range(256)], dtype=np.float32))
    return _T


def dequant_fp32(codes, scales, g, mean=None):
    """codes [T][H][D/2], scales [T][H][D/16], g [T] (per token), mean [T][H][D] or None -> fp32 [T][H][D]."""
    e2m1, e4m3 = _tables()
    c = np.asarray(codes, dtype=np.uint8)
    T, H, D2 = c.shape
    q = np.empty((T, H, 2 * D2), dtype=np.float32)
    q[..., 0::2] = e2m1[c & 0xF]
    q[..., 1::2] = e2m1[c >> 4]
    S = (e4m3[np.asarray(scales, dtype=np.uint8)] * np.asarray(g, dtype=np.float32)[:, None, None]).astype(np.float32)
    v = (q * np.repeat(S, 16, axis=2)).astype(np.float32)
    if mean is not None:
        v = (v + np.asarray(mean, dtype=np.float32)).astype(np.float32)
    return v


def attention_decode(q, k, v, scale: float):
    """q [n_q][H][D], k and v [T][H][D] (fp32 values) -> (out [n_q][H][D] binary64,
    A [n_q][H] = max_t |scale| sum_d |q_d k_td|, Vmax [H] = max_t,d |v|)."""
    q64, k64, v64 = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    s = np.einsum("ihd,thd->iht", q64, k64) * float(scale)
    s -= s.max(axis=2, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=2, keepdims=True)
    out = np.einsum("iht,thd->ihd", p, v64)
    A = np.einsum("ihd,thd->iht", np.abs(q64), np.abs(k64)).max(axis=2) * abs(float(scale))
    Vmax = np.abs(v64).max(axis=(0, 2))
    return out, A, Vmax


def attention_weighted_abs(q, k, v, scale: float):
    """q [n_q][H][D], k and v [T][H][D] (fp32 values) -> (out [n_q][H][D] binary64,
    B [n_q][H][D] = sum_t p_t |v_td|), p the binary64 softmax weights of each query and head.
    B bounds how far rounding the weights moves each output: a relative error e in every
    weight moves out by at most e * B."""
    q64, k64, v64 = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    s = np.einsum("ihd,thd->iht", q64, k64) * float(scale)
    s -= s.max(axis=2, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=2, keepdims=True)
    return np.einsum("iht,thd->ihd", p, v64), np.einsum("iht,thd->ihd", p, np.abs(v64))
