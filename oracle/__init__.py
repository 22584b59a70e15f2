"""CPU oracle for the NVFP4 KV-cache quantizer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and this package never imports the
product.

The arithmetic lives in ``nvfp4_oracle.c`` (plain C, fp32 IEEE operations in
the order the method's definition states, no FMA contraction).  This module
compiles it with gcc on first use and wraps it with ctypes + numpy.  The
method follows the LongLive-2.0 summary page ("LongLive-2.0: An NVFP4 Parallel
Infrastructure for Long Video Generation"): inference step 7 (per-chunk
K-smoothing, then 4/6 adaptive block scaling into the NVFP4 KV cache), the
"full-stack NVFP4" paragraph (Four-Over-Six: keep the lower-MSE of two FP8
block-scale candidates) and training step 4 (2-D block scales for weights).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

OK = 0
NONFINITE = 1
EINVAL = 2

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c_void_p, c_int, c_int64, c_float = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        P = ctypes.POINTER
        lib.oracle_e2m1_encode.argtypes = [c_float]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint]
        lib.oracle_e2m1_decode.restype = c_float
        lib.oracle_e4m3_encode.argtypes = [c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint]
        lib.oracle_e4m3_decode.restype = c_float
        lib.oracle_e2m1_encode_n.argtypes = [c_void_p, c_void_p, c_int64]
        lib.oracle_e2m1_encode_n.restype = None
        lib.oracle_e4m3_encode_n.argtypes = [c_void_p, c_void_p, c_int64]
        lib.oracle_e4m3_encode_n.restype = None
        lib.oracle_bf16_rne.argtypes = [c_float]
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_tensor_scale.argtypes = [c_float]
        lib.oracle_tensor_scale.restype = c_float
        lib.oracle_channel_mean.argtypes = [c_void_p, c_int, c_int64, c_int64, c_void_p]
        lib.oracle_channel_mean.restype = None
        lib.oracle_block_detail.argtypes = [c_void_p, c_int, c_float, c_void_p] + [c_void_p] * 10
        lib.oracle_block_detail.restype = c_int
        lib.oracle_kv_smooth_quant.argtypes = [c_void_p, c_int, c_int64, c_int64, c_int64, c_int,
                                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
        lib.oracle_kv_smooth_quant.restype = c_int
        lib.oracle_kv_smooth_quant_headroom.argtypes = [c_void_p, c_int, c_int64, c_int64, c_int64, c_int,
                                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
        lib.oracle_kv_smooth_quant_headroom.restype = c_int
        lib.oracle_kv_smooth_quant_threads.argtypes = [c_void_p, c_int, c_int64, c_int64, c_int64, c_int,
                                                       c_void_p, c_void_p, c_void_p, c_void_p, c_int]
        lib.oracle_kv_smooth_quant_threads.restype = c_int
        lib.oracle_tensor_scale_headroom.argtypes = [c_float]
        lib.oracle_tensor_scale_headroom.restype = c_float
        lib.oracle_kv_dequant.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64,
                                          c_int64, c_int64, c_void_p]
        lib.oracle_kv_dequant.restype = c_int
        lib.oracle_weight_quant_2d.argtypes = [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p,
                                               c_void_p, c_void_p]
        lib.oracle_weight_quant_2d.restype = c_int
        lib.oracle_weight_dequant_2d.argtypes = [c_void_p, c_void_p, c_float, c_int64, c_int64, c_void_p]
        lib.oracle_weight_dequant_2d.restype = c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_input(x: np.ndarray):
    """Return (array, dtype code): uint16 arrays are bf16 bit patterns, float32 arrays fp32."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, 0
    if x.dtype == np.float32:
        return x, 1
    raise TypeError(f"oracle input must be bf16 bits (uint16) or float32, got {x.dtype}")


# ---------------------------------------------------------------- scalar casts
def e2m1_encode(y: float) -> int:
    return int(_load().oracle_e2m1_encode(float(y)))


def e2m1_decode(code: int) -> float:
    return float(_load().oracle_e2m1_decode(int(code)))


def e4m3_encode(s: float) -> int:
    return int(_load().oracle_e4m3_encode(float(s)))


def e4m3_decode(code: int) -> float:
    return float(_load().oracle_e4m3_decode(int(code)))


def e2m1_encode_array(y: np.ndarray) -> np.ndarray:
    """E2M1 codes (uint8) of a float32 array, element by element."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    _load().oracle_e2m1_encode_n(_ptr(y), _ptr(out), y.size)
    return out


def e4m3_encode_array(s: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8) of a float32 array, element by element."""
    s = np.ascontiguousarray(s, dtype=np.float32)
    out = np.empty(s.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_n(_ptr(s), _ptr(out), s.size)
    return out


def bf16_rne(x: float) -> int:
    return int(_load().oracle_bf16_rne(float(x)))


def tensor_scale(amax: float) -> float:
    return float(_load().oracle_tensor_scale(float(amax)))


# ---------------------------------------------------------------- tensors
def channel_mean(x: np.ndarray) -> np.ndarray:
    """Per-channel token mean of x[T, C] (bf16 bits or fp32), rounded once to fp32."""
    x, dt = _as_input(x)
    T = x.shape[0]
    C = int(np.prod(x.shape[1:]))
    out = np.zeros(C, dtype=np.float32)
    _load().oracle_channel_mean(_ptr(x), dt, T, C, _ptr(out))
    return out


def block_detail(z: np.ndarray, g: float) -> dict:
    """Both Four-Over-Six candidates for one block z (16 or 256 values, R8 order)."""
    z = np.ascontiguousarray(z, dtype=np.float32).ravel()
    n = z.size
    codes = np.zeros(n, dtype=np.uint32)
    u = [np.zeros(1, dtype=np.uint32) for _ in range(3)]  # scale, e6, e4
    i = [np.zeros(1, dtype=np.int32) for _ in range(3)]  # chose4, ok6, ok4
    f = [np.zeros(1, dtype=np.float32) for _ in range(4)]  # err6, err4, sum6, sum4
    rc = _load().oracle_block_detail(_ptr(z), n, float(g), _ptr(codes), _ptr(u[0]), _ptr(i[0]), _ptr(u[1]),
                                     _ptr(u[2]), _ptr(i[1]), _ptr(i[2]), _ptr(f[0]), _ptr(f[1]), _ptr(f[2]),
                                     _ptr(f[3]))
    if rc != OK:
        raise ValueError(f"oracle_block_detail rc={rc}")
    return dict(codes=codes.astype(np.uint8), scale=int(u[0][0]), chose4=bool(i[0][0]), e6=int(u[1][0]),
                e4=int(u[2][0]), ok6=bool(i[1][0]), ok4=bool(i[2][0]), err6=float(f[0][0]), err4=float(f[1][0]),
                sum6=float(f[2][0]), sum4=float(f[3][0]))


def kv_smooth_quant(x: np.ndarray, smooth: bool, mean_in: np.ndarray | None = None,
                    headroom: bool = False) -> dict:
    """Quantize x[T, H, D] (bf16 bits as uint16, or float32).

    headroom: take the tensor scale g = amax / 1792 (4 x 448) instead of amax / 2688.
    Returns dict(codes [T, H, D/2] uint8, scales [T, H, D/16] uint8, g float,
    mean [H, D] float32 or None, chose4 [T, H, D/16] uint8, status int).
    """
    x, dt = _as_input(x)
    T, H, D = x.shape
    codes = np.zeros((T, H, D // 2), dtype=np.uint8)
    scales = np.zeros((T, H, D // 16), dtype=np.uint8)
    chose4 = np.zeros((T, H, D // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    mean_out = np.zeros((H, D), dtype=np.float32) if smooth else None
    mi = None if mean_in is None else np.ascontiguousarray(mean_in, dtype=np.float32).reshape(H, D)
    lib = _load()
    fn = lib.oracle_kv_smooth_quant_headroom if headroom else lib.oracle_kv_smooth_quant
    rc = fn(_ptr(x), dt, T, H, D, int(bool(smooth)), _ptr(mi), _ptr(mean_out),
            _ptr(codes), _ptr(scales), _ptr(g), _ptr(chose4))
    if rc == EINVAL:
        raise ValueError("oracle_kv_smooth_quant: invalid arguments")
    return dict(codes=codes, scales=scales, g=float(g[0]), mean=mean_out, chose4=chose4, status=rc)


def kv_smooth_quant_threads(x: np.ndarray, smooth: bool, threads: int) -> dict:
    """kv_smooth_quant on `threads` host threads (channel, element and block ranges split among
    them; bit for bit the single-threaded results).  For timing the baseline on all cores.
    Returns dict(codes, scales, g, mean, status) as kv_smooth_quant (no chose4)."""
    x, dt = _as_input(x)
    T, H, D = x.shape
    codes = np.zeros((T, H, D // 2), dtype=np.uint8)
    scales = np.zeros((T, H, D // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    mean_out = np.zeros((H, D), dtype=np.float32) if smooth else None
    rc = _load().oracle_kv_smooth_quant_threads(_ptr(x), dt, T, H, D, int(bool(smooth)), _ptr(mean_out),
                                                _ptr(codes), _ptr(scales), _ptr(g), int(threads))
    if rc == EINVAL:
        raise ValueError("oracle_kv_smooth_quant_threads: invalid arguments")
    return dict(codes=codes, scales=scales, g=float(g[0]), mean=mean_out, status=rc)


def kv_dequant(codes: np.ndarray, scales: np.ndarray, g, mean=None, tokens_per_group: int | None = None) -> np.ndarray:
    """Dequantize to bf16 bit patterns (uint16) of shape [T, H, D]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    T, H, D2 = codes.shape
    D = 2 * D2
    g = np.ascontiguousarray(np.atleast_1d(np.asarray(g, dtype=np.float32)))
    tpg = T if tokens_per_group is None else int(tokens_per_group)
    tpg = max(tpg, 1)
    m = None if mean is None else np.ascontiguousarray(mean, dtype=np.float32)
    out = np.zeros((T, H, D), dtype=np.uint16)
    rc = _load().oracle_kv_dequant(_ptr(codes), _ptr(scales), _ptr(g), _ptr(m), tpg, T, H, D, _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_kv_dequant rc={rc}")
    return out


def weight_quant_2d(w: np.ndarray) -> dict:
    """Quantize w[M, N] with 16x16 tiles.  Returns codes [M, N/2], scales [M/16, N/16], g, chose4, status."""
    w, dt = _as_input(w)
    M, N = w.shape
    codes = np.zeros((M, N // 2), dtype=np.uint8)
    scales = np.zeros((M // 16, N // 16), dtype=np.uint8)
    chose4 = np.zeros((M // 16, N // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    rc = _load().oracle_weight_quant_2d(_ptr(w), dt, M, N, _ptr(codes), _ptr(scales), _ptr(g), _ptr(chose4))
    if rc == EINVAL:
        raise ValueError("oracle_weight_quant_2d: invalid arguments")
    return dict(codes=codes, scales=scales, g=float(g[0]), chose4=chose4, status=rc)


def weight_dequant_2d(codes: np.ndarray, scales: np.ndarray, g: float) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    M, N2 = codes.shape
    out = np.zeros((M, 2 * N2), dtype=np.uint16)
    rc = _load().oracle_weight_dequant_2d(_ptr(codes), _ptr(scales), float(g), M, 2 * N2, _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_weight_dequant_2d rc={rc}")
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
