"""A second, independent statement of the oracle in numpy -- TEST INFRASTRUCTURE ONLY.

It restates the quantizer of "LongLive-2.0: An NVFP4 Parallel Infrastructure for
Long Video Generation" (summary page: inference step 7, per-chunk K-smoothing
and 4/6 adaptive block scaling into the NVFP4 KV cache; the "full-stack NVFP4"
paragraph, Four-Over-Six: keep the lower-MSE of two FP8 block-scale candidates;
training step 4, 16x16 blocks for weights) from the NVFP4 definition, with the
same readings as ``nvfp4_oracle.c`` but none of its code: the minifloat
roundings are nearest-value searches over the formats' value tables, every fp32
operation is a numpy float32 operation (IEEE round to nearest even), and the
error chain's fused multiply-adds are emulated exactly in binary64.  The tests
compare the two statements bit for bit, so a slip in either shows.

Readings shared with the C oracle: mean = fl32(binary64 sum in token order / T);
Z = fl(X - mean); g = fl(amax / 2688); candidate M in {6, 4}:
s_M = fl(a_b * fl(1 / fl(M g))), e_M = E4M3(s_M), S_M = fl(E_M g), usable iff
E_M > 0, S_M > 0 and fl(1 / S_M) finite; y = fl(Z * fl(1 / S_M)), Q = E2M1(y),
err_M = fl(E_M^2 * acc) with acc = fma(y - Q, y - Q, acc) over the block's
elements in order (row-major in a 16x16 tile); 4 kept iff usable and (6 not
usable or err_4 < err_6).
"""
from __future__ import annotations

import numpy as np

f32 = np.float32

# E2M1 magnitudes in code order (codes 0..7) and E4M3 finite magnitudes (codes 0..126)
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E4M3_VALUES = np.array([(c & 7) * 2.0 ** -9 if (c >> 3) == 0 else (1 + (c & 7) / 8.0) * 2.0 ** ((c >> 3) - 7)
                        for c in range(127)], dtype=np.float64)


def _nearest_code(mag: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index of the nearest table value to each magnitude (table ascending), ties to the
    even index, magnitudes beyond the last value saturating to it."""
    mids = (table[:-1] + table[1:]) / 2.0            # exact in binary64 for both formats
    c = np.searchsorted(mids, mag, side="left")        # midpoints strictly below mag
    tie = (c < mids.size) & (mag == mids[np.minimum(c, mids.size - 1)])
    c = np.where(tie & ((c + 1) % 2 == 0), c + 1, c)   # on a midpoint: the even neighbour
    return np.minimum(c, table.size - 1)


def e2m1_encode(y: np.ndarray) -> np.ndarray:
    y = np.asarray(y, dtype=np.float32)
    code = _nearest_code(np.abs(y).astype(np.float64), E2M1_VALUES).astype(np.uint8)
    return np.where(np.signbit(y), code | 8, code).astype(np.uint8)


def e2m1_decode(code: np.ndarray) -> np.ndarray:
    code = np.asarray(code)
    v = E2M1_VALUES[code & 7]
    return np.where(code & 8, -v, v).astype(np.float32)


def e4m3_encode(s: np.ndarray) -> np.ndarray:
    s = np.asarray(s, dtype=np.float32)
    code = _nearest_code(np.abs(s).astype(np.float64), E4M3_VALUES).astype(np.uint8)
    return np.where(np.signbit(s), code | 0x80, code).astype(np.uint8)


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    code = np.asarray(code)
    mag = code & 0x7F
    v = np.where(mag == 0x7F, np.nan, E4M3_VALUES[np.minimum(mag, 126)])
    return np.where(code & 0x80, -v, v).astype(np.float32)


def _fma32(a: np.ndarray, b: np.ndarray, c: np.ndarray) -> np.ndarray:
    """fl32(a * b + c) rounded once, for float32 a, b, c: the product is exact in binary64;
    the sum's binary64 rounding error (TwoSum) decides the cases where the binary64 sum
    sits exactly on a float32 midpoint."""
    p = a.astype(np.float64) * b.astype(np.float64)
    cc = c.astype(np.float64)
    s = p + cc
    bp = s - p
    e = (p - (s - bp)) + (cc - bp)                      # s + e == p + c exactly
    r = s.astype(np.float32)
    # s on a float32 midpoint: its two float32 neighbours are equally near; the exact
    # value p + c = s + e lies on the side of e
    lo = np.nextafter(r, np.float32(-np.inf))
    hi = np.nextafter(r, np.float32(np.inf))
    below = (r.astype(np.float64) + lo.astype(np.float64)) / 2.0
    above = (r.astype(np.float64) + hi.astype(np.float64)) / 2.0
    r = np.where((s == below) & (e < 0), lo, r)         # s on the midpoint below r, exact value under it
    r = np.where((s == above) & (e > 0), hi, r)         # s on the midpoint above r, exact value over it
    return r


def _blocks(Z: np.ndarray, g: np.float32):
    """Four-Over-Six on blocks Z[nb][n] (float32); returns (codes uint8 [nb][n], scale bytes [nb])."""
    nb, n = Z.shape
    ab = np.max(np.abs(Z), axis=1).astype(np.float32)
    res = {}
    for M in (6, 4):
        with np.errstate(divide="ignore", over="ignore"):
            k = f32(f32(1.0) / f32(f32(M) * g))   # inf when M g is subnormal: a_b * k is then inf or NaN
        e = e4m3_encode((ab * k).astype(np.float32))
        E = e4m3_decode(e)
        S = (E * g).astype(np.float32)
        with np.errstate(divide="ignore", over="ignore"):
            inv = (f32(1.0) / S).astype(np.float32)
        ok = (E > 0) & (S > 0) & np.isfinite(inv)
        inv_used = np.where(ok, inv, f32(0.0)).astype(np.float32)
        y = (Z * inv_used[:, None]).astype(np.float32)
        q = e2m1_encode(y)
        d = (y - e2m1_decode(q)).astype(np.float32)    # exact: y and Q within a factor of two
        acc = np.zeros(nb, dtype=np.float32)
        for i in range(n):                              # element order
            acc = _fma32(d[:, i], d[:, i], acc)
        err = ((E * E).astype(np.float32) * acc).astype(np.float32)
        res[M] = (e, q, ok, err)
    e6, q6, ok6, err6 = res[6]
    e4, q4, ok4, err4 = res[4]
    pick4 = ok4 & (~ok6 | (err4 < err6))
    codes = np.where(pick4[:, None], q4, np.where(ok6[:, None], q6, 0)).astype(np.uint8)
    scale = np.where(pick4, e4, np.where(ok6, e6, 0)).astype(np.uint8)
    zero = ab == 0
    codes[zero] = 0
    scale[zero] = 0
    return codes, scale


def _widen(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32)
    return np.asarray(x, dtype=np.float32)


def _pack(codes: np.ndarray) -> np.ndarray:
    c = codes.reshape(-1, 2)
    return (c[:, 0] | (c[:, 1] << 4)).astype(np.uint8)


def kv_smooth_quant(x: np.ndarray, smooth: bool):
    """x [T][H][D] (bf16 bits as uint16, or float32) -> dict(codes, scales, g, mean, status)."""
    X = _widen(x)
    T, H, D = X.shape
    C = H * D
    Xf = X.reshape(T, C)
    mean = None
    if smooth:
        total = np.cumsum(Xf.astype(np.float64), axis=0)[-1] if T else np.zeros(C)  # binary64, token order
        mean = (total / T).astype(np.float32) if T else np.zeros(C, np.float32)
        Z = (Xf - mean[None, :]).astype(np.float32)
    else:
        Z = Xf
    amax = np.float32(np.max(np.abs(Z))) if Z.size else np.float32(0.0)
    if not np.isfinite(amax):
        return dict(codes=np.zeros((T, H, D // 2), np.uint8), scales=np.full((T, H, D // 16), 0x7F, np.uint8),
                    g=np.float32(np.nan), mean=mean, status=1)
    g = f32(amax / f32(2688.0))
    blocks = Z.reshape(-1, 16)
    if g == 0:
        codes = np.zeros(blocks.shape, np.uint8)
        scales = np.zeros(blocks.shape[0], np.uint8)
    else:
        codes, scales = _blocks(blocks, g)
    return dict(codes=_pack(codes.reshape(-1)).reshape(T, H, D // 2), scales=scales.reshape(T, H, D // 16), g=g,
                mean=mean, status=0)


def weight_quant_2d(w: np.ndarray):
    """w [M][N] (bf16 bits or float32) -> dict(codes [M][N/2], scales [M/16][N/16], g, status); 16x16 tiles,
    each tile's error chain in row-major order."""
    W = _widen(w)
    M, N = W.shape
    amax = np.float32(np.max(np.abs(W))) if W.size else np.float32(0.0)
    if not np.isfinite(amax):
        return dict(codes=np.zeros((M, N // 2), np.uint8), scales=np.full((M // 16, N // 16), 0x7F, np.uint8),
                    g=np.float32(np.nan), status=1)
    g = f32(amax / f32(2688.0))
    tiles = W.reshape(M // 16, 16, N // 16, 16).transpose(0, 2, 1, 3).reshape(-1, 256)
    if g == 0:
        codes = np.zeros(tiles.shape, np.uint8)
        scales = np.zeros(tiles.shape[0], np.uint8)
    else:
        codes, scales = _blocks(tiles, g)
    grid = codes.reshape(M // 16, N // 16, 16, 16).transpose(0, 2, 1, 3).reshape(M, N)
    return dict(codes=_pack(grid.reshape(-1)).reshape(M, N // 2), scales=scales.reshape(M // 16, N // 16), g=g,
                status=0)
