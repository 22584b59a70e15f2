"""NVFP4 KV-cache quantizer for GB300 (sm_103a): thin PyTorch-facing binding.

Every computation runs in the CUDA library (``_build/libnvfp4_gb300.so``,
C ABI in ``include/nvfp4.h``); this module only allocates output tensors with
torch, marshals pointers and sizes, and raises on a non-OK status.  There is no
CPU path: without the built library every call raises.

Method: "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video
Generation" (summary page) -- inference step 7 (per-chunk K-smoothing, then
Four-Over-Six NVFP4 KV cache) and training step 4 (2-D block scales for
weights, 1-D for activations).
"""
from __future__ import annotations

import ctypes
from typing import NamedTuple, Optional, Sequence

from . import _lib
from ._lib import NVFP4_IN_BF16, NVFP4_IN_FP32, NVFP4Error, nvfp4_kv_job, nvfp4_w2d_job

__all__ = [
    "NVFP4Error", "KvQuantized", "W2dQuantized", "kv_workspace", "kv_smooth_quant", "kv_smooth_quant_batched",
    "kv_stats_batched", "kv_quant_batched",
    "kv_dequant", "KvCache", "KvCachePool", "kv_gather_dequant", "kv_attention_decode", "mma_scales", "rht16", "ActQuantized", "act_quant_mma", "GemmPlan",
    "gemm_w4a4",
    "w2d_workspace", "weight_quant_2d", "w2d_batched_workspace", "weight_quant_2d_batched",
    "weight_dequant_2d", "load_library",
]


def load_library():
    """Load the CUDA library (raises if it has not been built)."""
    return _lib.load()


class KvQuantized(NamedTuple):
    codes: "torch.Tensor"         # uint8 [T, H, D/2]
    scales: "torch.Tensor"        # uint8 [T, H, D/16] (E4M3 bytes)
    tensor_scale: "torch.Tensor"  # float32 [1]
    mean: Optional["torch.Tensor"]  # float32 [H, D] (smoothed tensors) or None
    status: "torch.Tensor"        # int32 [1] device status word


class W2dQuantized(NamedTuple):
    codes: "torch.Tensor"         # uint8 [M, N/2]
    scales: "torch.Tensor"        # uint8 [M/16, N/16]
    tensor_scale: "torch.Tensor"  # float32 [1]
    status: "torch.Tensor"        # int32 [1]


def _torch():
    import torch

    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dt(x) -> int:
    torch = _torch()
    if x.dtype == torch.bfloat16:
        return NVFP4_IN_BF16
    if x.dtype == torch.float32:
        return NVFP4_IN_FP32
    raise TypeError(f"input must be bfloat16 or float32, got {x.dtype}")


def _check_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def kv_workspace(T: int, H: int, D: int, n_jobs: int = 1, device=None):
    """Allocate (with torch) the zero-filled device workspace a KV quantize call of this shape needs.

    The library's counters in it return to zero at the end of every call, so it can be reused by
    later calls on the same stream without clearing.
    """
    torch = _torch()
    nbytes = _lib.nvfp4_kv_batched_workspace_bytes(n_jobs, T, H, D)
    if nbytes == 0:
        raise NVFP4Error(_lib.NVFP4_ESHAPE, "kv_workspace")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def _kv_outputs(T, H, D, smooth, device):
    torch = _torch()
    codes = torch.empty((T, H, D // 2), dtype=torch.uint8, device=device)
    scales = torch.empty((T, H, D // 16), dtype=torch.uint8, device=device)
    g = torch.empty(1, dtype=torch.float32, device=device)
    mean = torch.empty((H, D), dtype=torch.float32, device=device) if smooth else None
    return codes, scales, g, mean


def kv_smooth_quant(x, smooth: bool, mean_in=None, workspace=None, out: Optional[KvQuantized] = None,
                    stream=None) -> KvQuantized:
    """Quantize x[T, H, D] (bf16 or fp32, CUDA) into NVFP4 with Four-Over-Six block scales.

    smooth=True subtracts the per-(head, channel) token mean first (keys); the mean used is
    returned.  Asynchronous on `stream`; `status` is a device int (NVFP4_DEV_*).
    """
    torch = _torch()
    _check_cuda(x, mean_in)
    T, H, D = x.shape
    if out is None:
        codes, scales, g, mean = _kv_outputs(T, H, D, smooth, x.device)
        status = torch.empty(1, dtype=torch.int32, device=x.device)
    else:
        codes, scales, g, mean, status = out
    if workspace is None:
        workspace = kv_workspace(T, H, D, 1, x.device)
    st = _lib.nvfp4_kv_smooth_quant(_ptr(x), _dt(x), T, H, D, int(bool(smooth)), _ptr(mean_in),
                                    _ptr(mean) if smooth else None, _ptr(codes), _ptr(scales), _ptr(g),
                                    _ptr(status), _ptr(workspace), workspace.numel(), _stream(stream))
    _lib.check(st, "nvfp4_kv_smooth_quant")
    return KvQuantized(codes, scales, g, mean, status)


def _batch_jobs(xs, smooth, outs, status):
    torch = _torch()
    n = len(xs)
    if n == 0 or len(smooth) != n:
        raise ValueError("need one smooth flag per tensor")
    x0 = xs[0]
    T, H, D = x0.shape
    for x in xs:
        _check_cuda(x)
        if tuple(x.shape) != (T, H, D) or x.dtype != x0.dtype:
            raise ValueError("all tensors of a batch share shape and dtype")
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=x0.device)
    if outs is None:
        outs = []
        for sm in smooth:
            c, s, g, m = _kv_outputs(T, H, D, sm, x0.device)
            outs.append(KvQuantized(c, s, g, m, status))
    jobs = (nvfp4_kv_job * n)()
    for i, (x, sm, o) in enumerate(zip(xs, smooth, outs)):
        jobs[i].x = x.data_ptr()
        jobs[i].smooth = int(bool(sm))
        jobs[i].mean_in = None
        jobs[i].mean_out = o.mean.data_ptr() if (sm and o.mean is not None) else None
        jobs[i].codes = o.codes.data_ptr()
        jobs[i].scales = o.scales.data_ptr()
        jobs[i].tensor_scale = o.tensor_scale.data_ptr()
    return jobs, outs, status, (T, H, D)


def kv_smooth_quant_batched(xs: Sequence, smooth: Sequence[bool], workspace=None, outs=None, status=None,
                            stream=None, headroom: bool = False):
    """Quantize several same-shape chunk tensors (e.g. K and V of every layer) in one enqueue.

    Returns (list of KvQuantized, status) with one shared device status word (OR over tensors).
    headroom=True takes the tensor scale g = amax / 1792 instead of amax / 2688
    (nvfp4_kv_smooth_quant_headroom).
    """
    jobs, outs, status, (T, H, D) = _batch_jobs(xs, smooth, outs, status)
    if workspace is None:
        workspace = kv_workspace(T, H, D, len(xs), xs[0].device)
    fn = _lib.nvfp4_kv_smooth_quant_headroom if headroom else _lib.nvfp4_kv_smooth_quant_batched
    st = fn(jobs, len(xs), _dt(xs[0]), T, H, D, _ptr(status), _ptr(workspace), workspace.numel(), _stream(stream))
    _lib.check(st, "nvfp4_kv_smooth_quant_headroom" if headroom else "nvfp4_kv_smooth_quant_batched")
    return outs, status


def kv_stats_batched(xs: Sequence, smooth: Sequence[bool], workspace, outs, stream=None):
    """First pass of kv_smooth_quant_batched alone: channel means (into outs[i].mean) and amax, kept in `workspace`.

    Must be followed by kv_quant_batched with the same tensors, outputs and workspace.
    """
    jobs, outs, _, (T, H, D) = _batch_jobs(xs, smooth, outs, outs[0].status)
    st = _lib.nvfp4_kv_stats_batched(jobs, len(xs), _dt(xs[0]), T, H, D, _ptr(workspace), workspace.numel(),
                                     _stream(stream))
    _lib.check(st, "nvfp4_kv_stats_batched")
    return outs


def kv_quant_batched(xs: Sequence, smooth: Sequence[bool], workspace, outs, status, stream=None):
    """Second pass of kv_smooth_quant_batched: quantize with the statistics kv_stats_batched left in `workspace`."""
    jobs, outs, status, (T, H, D) = _batch_jobs(xs, smooth, outs, status)
    st = _lib.nvfp4_kv_quant_batched(jobs, len(xs), _dt(xs[0]), T, H, D, _ptr(status), _ptr(workspace),
                                     workspace.numel(), _stream(stream))
    _lib.check(st, "nvfp4_kv_quant_batched")
    return outs, status


def kv_dequant(codes, scales, tensor_scale, mean=None, tokens_per_group: Optional[int] = None, out=None,
               stream=None):
    """Dequantize NVFP4 codes/scales [T, H, D/2] / [T, H, D/16] to bf16 [T, H, D]."""
    torch = _torch()
    _check_cuda(codes, scales, tensor_scale, mean)
    T, H, D2 = codes.shape
    D = 2 * D2
    tpg = T if tokens_per_group is None else int(tokens_per_group)
    tpg = max(tpg, 1)
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=codes.device)
    st = _lib.nvfp4_kv_dequant(_ptr(codes), _ptr(scales), _ptr(tensor_scale), _ptr(mean), tpg, T, H, D, _ptr(out),
                               _stream(stream))
    _lib.check(st, "nvfp4_kv_dequant")
    return out


def selftest_cvt(x, stream=None):
    """Run the quantizers' conversion instructions on a CUDA fp32 tensor ``x``: returns
    (E2M1 code bytes [n] -- the code in both nibbles, E4M3 codes [n] uint16 -- the code in
    both bytes, the f16 pair decode of every byte [256] int32, every E4M3 code's value [256])."""
    torch = _torch()
    _check_cuda(x)
    x = x.contiguous().view(-1)
    n = x.numel()
    e2m1 = torch.empty(n, dtype=torch.uint8, device=x.device)
    e4m3 = torch.empty(n, dtype=torch.int16, device=x.device)
    dec = torch.empty(256, dtype=torch.int32, device=x.device)
    val = torch.empty(256, dtype=torch.float32, device=x.device)
    st = _lib.nvfp4_selftest_cvt(_ptr(x), n, _ptr(e2m1), _ptr(e4m3), _ptr(dec), _ptr(val), _stream(stream))
    _lib.check(st, "nvfp4_selftest_cvt")
    return e2m1, e4m3, dec, val


def kv_shard_bytes(T: int, H: int, D: int, P: int, with_mean: bool) -> int:
    """Bytes of one head-shard segment (nvfp4_kv_shard_bytes); 0 for invalid shapes."""
    return int(_lib.nvfp4_kv_shard_bytes(T, H, D, P, int(bool(with_mean))))


def kv_pack_head_shards(q: "KvQuantized", P: int, out=None, stream=None):
    """Pack a quantized tensor into P head-shard segments (uint8 [P, segment bytes])."""
    torch = _torch()
    _check_cuda(q.codes, q.scales, q.tensor_scale, q.mean)
    T, H, D2 = q.codes.shape
    D = 2 * D2
    seg = kv_shard_bytes(T, H, D, P, q.mean is not None)
    if seg == 0:
        raise ValueError("invalid shard shape (H % P must be 0)")
    if out is None:
        out = torch.empty((P, seg), dtype=torch.uint8, device=q.codes.device)
    st = _lib.nvfp4_kv_pack_head_shards(_ptr(q.codes), _ptr(q.scales), _ptr(q.tensor_scale), _ptr(q.mean), T, H, D,
                                        P, _ptr(out), _stream(stream))
    _lib.check(st, "nvfp4_kv_pack_head_shards")
    return out


def kv_unpack_head_shards(segments, T: int, H: int, D: int, P: int, with_mean: bool, stream=None):
    """Unpack P received segments into this rank's head shard of a P-group cache: returns
    (codes [P T, H/P, D/2], scales [P T, H/P, D/16], tensor scales [P], means [P, H/P, D] or None)."""
    torch = _torch()
    _check_cuda(segments)
    hs = H // P
    dev = segments.device
    codes = torch.empty((P * T, hs, D // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((P * T, hs, D // 16), dtype=torch.uint8, device=dev)
    gs = torch.empty(P, dtype=torch.float32, device=dev)
    means = torch.empty((P, hs, D), dtype=torch.float32, device=dev) if with_mean else None
    st = _lib.nvfp4_kv_unpack_head_shards(_ptr(segments), T, H, D, P, int(bool(with_mean)), _ptr(codes),
                                          _ptr(scales), _ptr(gs), _ptr(means), _stream(stream))
    _lib.check(st, "nvfp4_kv_unpack_head_shards")
    return codes, scales, gs, means


def kv_exchange_head_shards(segments, group=None):
    """All-to-all of packed head-shard segments ([P, segment bytes], equal splits): segment p
    goes to rank p and row r of the result came from rank r.  Uses torch.distributed
    (NCCL between GPUs; any backend with all_to_all_single)."""
    torch = _torch()
    import torch.distributed as dist

    out = torch.empty_like(segments)
    dist.all_to_all_single(out.view(-1), segments.contiguous().view(-1), group=group)
    return out


class KvCache:
    """Host bookkeeping of a multi-shot NVFP4 KV cache (``nvfp4_kvcache_*``): which chunk
    slot holds which chunk, the global sink, the shot sink (START/LEN) and the rolling
    window.  No device memory: pair it with one ``KvCachePool`` per cached tensor."""

    def __init__(self, frames_per_chunk: int, tokens_per_frame: int, global_sink: int, shot_sink: int, window: int,
                 n_slots: Optional[int] = None):
        if n_slots is None:
            n_slots = _lib.nvfp4_kvcache_slots_needed(frames_per_chunk, global_sink, shot_sink, window)
        self.state = _lib.nvfp4_kvcache()
        _lib.check(_lib.nvfp4_kvcache_init(self.state, frames_per_chunk, tokens_per_frame, global_sink, shot_sink,
                                           window, n_slots), "nvfp4_kvcache_init")

    @property
    def n_slots(self) -> int:
        return self.state.n_slots

    @property
    def n_chunks(self) -> int:
        return self.state.n_chunks

    def append(self) -> int:
        """Slot for the next chunk (releases dead slots first)."""
        slot = ctypes.c_int(-1)
        _lib.check(_lib.nvfp4_kvcache_append(self.state, slot), "nvfp4_kvcache_append")
        return slot.value

    def new_shot(self) -> None:
        _lib.check(_lib.nvfp4_kvcache_new_shot(self.state), "nvfp4_kvcache_new_shot")

    def view(self):
        """(frame_index, frame_row, frame_slot) numpy arrays of the next chunk's view."""
        import numpy as np

        cap = self.state.global_sink + self.state.shot_sink + self.state.window
        fi, fr = np.zeros(cap, np.int64), np.zeros(cap, np.int64)
        fs = np.zeros(cap, np.int32)
        n = _lib.nvfp4_kvcache_view(self.state, fi.ctypes.data, fr.ctypes.data, fs.ctypes.data, cap)
        if n < 0:
            raise NVFP4Error(_lib.NVFP4_EINVAL, "nvfp4_kvcache_view")
        return fi[:n], fr[:n], fs[:n]


class KvCachePool(NamedTuple):
    """Device storage of one cached tensor: ``n_slots`` chunk slots of F_c * L_f tokens."""
    codes: "torch.Tensor"   # uint8 [n_slots * F_c * L_f, H, D/2]
    scales: "torch.Tensor"  # uint8 [n_slots * F_c * L_f, H, D/16]
    g: "torch.Tensor"       # float32 [n_slots]
    mean: Optional["torch.Tensor"]  # float32 [n_slots, H, D] (smoothed tensors) or None

    @staticmethod
    def allocate(cache: KvCache, H: int, D: int, smooth: bool, device=None) -> "KvCachePool":
        torch = _torch()
        st = cache.state
        rows = st.n_slots * st.frames_per_chunk * st.tokens_per_frame
        dev = device or "cuda"
        return KvCachePool(torch.zeros((rows, H, D // 2), dtype=torch.uint8, device=dev),
                           torch.zeros((rows, H, D // 16), dtype=torch.uint8, device=dev),
                           torch.zeros(st.n_slots, dtype=torch.float32, device=dev),
                           torch.zeros((st.n_slots, H, D), dtype=torch.float32, device=dev) if smooth else None)

    def slot_outputs(self, cache: KvCache, slot: int, status=None) -> "KvQuantized":
        """The quantizer's outputs for a chunk written straight into ``slot`` (views, no copy)."""
        torch = _torch()
        rows = cache.state.frames_per_chunk * cache.state.tokens_per_frame
        r0 = slot * rows
        if status is None:
            status = torch.zeros(1, dtype=torch.int32, device=self.codes.device)
        return KvQuantized(self.codes[r0:r0 + rows], self.scales[r0:r0 + rows], self.g[slot:slot + 1],
                           None if self.mean is None else self.mean[slot], status)


def kv_gather_dequant(pool: KvCachePool, frame_row, frame_slot, tokens_per_frame: int, with_mean: bool = True,
                      out=None, stream=None):
    """Expand a view (frame_row, frame_slot: host int arrays from ``KvCache.view``) to bf16
    [n_frames * L_f, H, D], each frame with its slot's tensor scale (and mean when
    ``with_mean`` and the pool has means)."""
    import numpy as np

    torch = _torch()
    _check_cuda(pool.codes, pool.scales, pool.g, pool.mean)
    rows, H, D2 = pool.codes.shape
    D = 2 * D2
    fr = np.ascontiguousarray(frame_row, dtype=np.int64)
    fs = np.ascontiguousarray(frame_slot, dtype=np.int32)
    n = int(fr.shape[0])
    if out is None:
        out = torch.empty((n * tokens_per_frame, H, D), dtype=torch.bfloat16, device=pool.codes.device)
    mean = pool.mean if with_mean else None
    st = _lib.nvfp4_kv_gather_dequant(_ptr(pool.codes), _ptr(pool.scales), _ptr(pool.g), _ptr(mean), rows,
                                      int(pool.g.numel()), fr.ctypes.data, fs.ctypes.data, n, tokens_per_frame, H, D,
                                      _ptr(out), _stream(stream))
    _lib.check(st, "nvfp4_kv_gather_dequant")
    return out


def kv_attention_prefill(q, k_pool: KvCachePool, v_pool: KvCachePool, frame_row, frame_slot, tokens_per_frame: int,
                         scale: float, out=None, status=None, stream=None, workspace=None, split: bool = True):
    """Attention of a block of queries q [n_q, H, 128] (bf16) over a cache view read straight from the
    NVFP4 pools, on the tensor cores (``nvfp4_kv_attention_prefill``); K's means are re-added when its
    pool has them.  Returns fp32 [n_q, H, 128]; ``status`` (int32 [1], optional) collects
    NVFP4_DEV_TIMEOUT.  With ``split`` the last, partial wave of CTAs is split along the keys, in
    ``workspace`` (uint8 on the device, allocated here when None); ``split=False`` runs every unit
    whole."""
    import numpy as np

    torch = _torch()
    _check_cuda(q, k_pool.codes, v_pool.codes)
    if q.dtype != torch.bfloat16:
        raise TypeError("kv_attention_prefill: q must be bf16")
    n_q, H, D = q.shape
    fr = np.ascontiguousarray(frame_row, dtype=np.int64)
    fs = np.ascontiguousarray(frame_slot, dtype=np.int32)
    if out is None:
        out = torch.empty((n_q, H, D), dtype=torch.float32, device=q.device)
    ws_bytes = 0
    if split:
        need = _lib.nvfp4_kv_attention_prefill_workspace_bytes(n_q, H, int(fr.shape[0]), tokens_per_frame)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    else:
        workspace = None
    st = _lib.nvfp4_kv_attention_prefill(_ptr(q), n_q, _ptr(k_pool.codes), _ptr(k_pool.scales), _ptr(k_pool.g),
                                         _ptr(k_pool.mean), _ptr(v_pool.codes), _ptr(v_pool.scales), _ptr(v_pool.g),
                                         k_pool.codes.shape[0], int(k_pool.g.numel()), fr.ctypes.data,
                                         fs.ctypes.data, int(fr.shape[0]), tokens_per_frame, H, D, float(scale),
                                         _ptr(out), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream))
    _lib.check(st, "nvfp4_kv_attention_prefill")
    return out


def mma_scales(scales, K: int, tile2d: bool = False, out=None, stream=None):
    """Block scales in the tensor cores' layout (``nvfp4_scales_to_mma`` / ``nvfp4_w2d_scales_to_mma``).

    ``scales``: uint8 [rows, K/16] (1-D activation scales) or, with ``tile2d``, the
    16x16-tile weight scales [N/16, K/16]; returns a flat uint8 tensor."""
    torch = _torch()
    _check_cuda(scales)
    rows = scales.shape[0] * (16 if tile2d else 1)
    n = _lib.nvfp4_mma_scales_bytes(rows, K)
    if out is None:
        out = torch.empty(max(n, 16), dtype=torch.uint8, device=scales.device)
    fn = _lib.nvfp4_w2d_scales_to_mma if tile2d else _lib.nvfp4_scales_to_mma
    _lib.check(fn(_ptr(scales), rows, K, _ptr(out), _stream(stream)), fn.__name__)
    return out


def rht16(x, signs: int, out=None, stream=None):
    """Random Hadamard transform of every 16-element block along the last dim (``nvfp4_rht16``):
    x [rows, K] bf16 or fp32 -> fp32 [rows, K]."""
    torch = _torch()
    _check_cuda(x)
    K = x.shape[-1]
    rows = x.numel() // K
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    _lib.check(_lib.nvfp4_rht16(_ptr(x), _dt(x), rows, K, int(signs), _ptr(out), _stream(stream)), "nvfp4_rht16")
    return out


class ActQuantized(NamedTuple):
    codes: "torch.Tensor"         # uint8 [M, K/2]
    scales_mma: "torch.Tensor"    # uint8, tensor-core layout
    tensor_scale: "torch.Tensor"  # float32 [1]
    status: "torch.Tensor"        # int32 [1]


def act_quant_mma(x, rht_signs: Optional[int] = None, workspace=None, out: Optional[ActQuantized] = None,
                  stream=None) -> ActQuantized:
    """Activation x [M, K] bf16 -> NVFP4 codes and tensor-core-layout scales in one call pair
    (``nvfp4_act_quant_mma``), with the random Hadamard transform first when ``rht_signs`` is given."""
    torch = _torch()
    _check_cuda(x)
    M, K = x.shape
    if out is None:
        out = ActQuantized(torch.empty((M, K // 2), dtype=torch.uint8, device=x.device),
                           torch.empty(max(_lib.nvfp4_mma_scales_bytes(M, K), 16), dtype=torch.uint8,
                                       device=x.device),
                           torch.empty(1, dtype=torch.float32, device=x.device),
                           torch.empty(1, dtype=torch.int32, device=x.device))
    if workspace is None:
        workspace = torch.empty(_lib.nvfp4_act_quant_workspace_bytes(), dtype=torch.uint8, device=x.device)
    st = _lib.nvfp4_act_quant_mma(_ptr(x), M, K, 0 if rht_signs is None else 1, int(rht_signs or 0),
                                  _ptr(out.codes), _ptr(out.scales_mma), _ptr(out.tensor_scale), _ptr(out.status),
                                  _ptr(workspace), workspace.numel(), _stream(stream))
    _lib.check(st, "nvfp4_act_quant_mma")
    return out


class GemmPlan:
    """Caller-owned W4A4 GEMM plan for one (M, N, K) (``nvfp4_gemm_plan_create``)."""

    def __init__(self, M: int, N: int, K: int):
        self.M, self.N, self.K = M, N, K
        self._p = ctypes.c_void_p()
        _lib.check(_lib.nvfp4_gemm_plan_create(M, N, K, self._p), "nvfp4_gemm_plan_create")

    def close(self):
        """Free the plan now (it is also freed when the object is collected)."""
        p, self._p = getattr(self, "_p", None), None
        if p is not None and p.value:
            _lib.nvfp4_gemm_plan_destroy(p)

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: the library may already be unloaded
            pass


def gemm_workspace(device=None):
    torch = _torch()
    return torch.zeros(_lib.nvfp4_gemm_workspace_bytes(), dtype=torch.uint8, device=device or "cuda")


def gemm_w4a4(plan: GemmPlan, x_codes, x_scales_mma, x_tensor_scale, w_codes, w_scales_mma, w_tensor_scale,
              workspace, out=None, stream=None):
    """Y [M, N] bf16 = X W^T from NVFP4 operands (``nvfp4_gemm_w4a4``): X codes [M, K/2], W codes
    [N, K/2], scales already in the tensor-core layout (``mma_scales``)."""
    torch = _torch()
    _check_cuda(x_codes, x_scales_mma, x_tensor_scale, w_codes, w_scales_mma, w_tensor_scale, workspace)
    if out is None:
        out = torch.empty((plan.M, plan.N), dtype=torch.bfloat16, device=x_codes.device)
    st = _lib.nvfp4_gemm_w4a4(plan._p, _ptr(x_codes), _ptr(x_scales_mma), _ptr(x_tensor_scale), _ptr(w_codes),
                              _ptr(w_scales_mma), _ptr(w_tensor_scale), _ptr(out), _ptr(workspace),
                              workspace.numel(), _stream(stream))
    _lib.check(st, "nvfp4_gemm_w4a4")
    return out


def kv_attention_decode(q, k_pool: KvCachePool, v_pool: KvCachePool, frame_row, frame_slot, tokens_per_frame: int,
                        scale: float, workspace=None, out=None, stream=None):
    """Attention of q [n_q, H, D] (fp32) over a cache view read straight from the NVFP4 pools
    (``nvfp4_kv_attention_decode``); K's means are re-added when its pool has them.  fp32 [n_q, H, D]."""
    import numpy as np

    torch = _torch()
    _check_cuda(q, k_pool.codes, v_pool.codes)
    n_q, H, D = q.shape
    fr = np.ascontiguousarray(frame_row, dtype=np.int64)
    fs = np.ascontiguousarray(frame_slot, dtype=np.int32)
    n = int(fr.shape[0])
    if workspace is None:
        workspace = torch.empty(max(_lib.nvfp4_kv_attention_workspace_bytes(n, tokens_per_frame, H, D, n_q), 256),
                                dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((n_q, H, D), dtype=torch.float32, device=q.device)
    st = _lib.nvfp4_kv_attention_decode(_ptr(q), n_q, _ptr(k_pool.codes), _ptr(k_pool.scales), _ptr(k_pool.g),
                                        _ptr(k_pool.mean), _ptr(v_pool.codes), _ptr(v_pool.scales), _ptr(v_pool.g),
                                        k_pool.codes.shape[0], int(k_pool.g.numel()), fr.ctypes.data,
                                        fs.ctypes.data, n, tokens_per_frame, H, D, float(scale), _ptr(out),
                                        _ptr(workspace), workspace.numel(), _stream(stream))
    _lib.check(st, "nvfp4_kv_attention_decode")
    return out


def w2d_workspace(M: int, N: int, device=None):
    torch = _torch()
    nbytes = _lib.nvfp4_w2d_workspace_bytes(M, N)
    if nbytes == 0:
        raise NVFP4Error(_lib.NVFP4_ESHAPE, "w2d_workspace")
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def weight_quant_2d(w, workspace=None, out: Optional[W2dQuantized] = None, stream=None) -> W2dQuantized:
    """Quantize a weight matrix w[M, N] with 16x16 NVFP4 tiles and Four-Over-Six scales."""
    torch = _torch()
    _check_cuda(w)
    M, N = w.shape
    if out is None:
        codes = torch.empty((M, N // 2), dtype=torch.uint8, device=w.device)
        scales = torch.empty((M // 16, N // 16), dtype=torch.uint8, device=w.device)
        g = torch.empty(1, dtype=torch.float32, device=w.device)
        status = torch.empty(1, dtype=torch.int32, device=w.device)
    else:
        codes, scales, g, status = out
    if workspace is None:
        workspace = w2d_workspace(M, N, w.device)
    st = _lib.nvfp4_weight_quant_2d(_ptr(w), _dt(w), M, N, _ptr(codes), _ptr(scales), _ptr(g), _ptr(status),
                                    _ptr(workspace), workspace.numel(), _stream(stream))
    _lib.check(st, "nvfp4_weight_quant_2d")
    return W2dQuantized(codes, scales, g, status)


def w2d_batched_workspace(n_jobs: int, device=None):
    torch = _torch()
    nbytes = _lib.nvfp4_w2d_batched_workspace_bytes(n_jobs)
    if nbytes == 0:
        raise NVFP4Error(_lib.NVFP4_EINVAL, "w2d_batched_workspace")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")  # must start zero-filled


def weight_quant_2d_batched(ws: Sequence, workspace=None, outs=None, status=None, stream=None):
    """Quantize several weight matrices (shapes may differ, dtype shared) in one amax and one quantizer launch.

    Returns (list of W2dQuantized, status) with one shared device status word (OR over matrices).
    """
    torch = _torch()
    n = len(ws)
    if n == 0:
        raise ValueError("need at least one matrix")
    w0 = ws[0]
    for w in ws:
        _check_cuda(w)
        if w.dim() != 2 or w.dtype != w0.dtype:
            raise ValueError("all matrices of a batch are 2-D and share a dtype")
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=w0.device)
    if outs is None:
        outs = []
        for w in ws:
            M, N = w.shape
            outs.append(W2dQuantized(torch.empty((M, N // 2), dtype=torch.uint8, device=w.device),
                                     torch.empty((M // 16, N // 16), dtype=torch.uint8, device=w.device),
                                     torch.empty(1, dtype=torch.float32, device=w.device), status))
    if workspace is None:
        workspace = w2d_batched_workspace(n, w0.device)
    jobs = (nvfp4_w2d_job * n)()
    for i, (w, o) in enumerate(zip(ws, outs)):
        jobs[i].w = w.data_ptr()
        jobs[i].M, jobs[i].N = w.shape
        jobs[i].codes = o.codes.data_ptr()
        jobs[i].scales = o.scales.data_ptr()
        jobs[i].tensor_scale = o.tensor_scale.data_ptr()
    st = _lib.nvfp4_weight_quant_2d_batched(jobs, n, _dt(w0), _ptr(status), _ptr(workspace), workspace.numel(),
                                            _stream(stream))
    _lib.check(st, "nvfp4_weight_quant_2d_batched")
    return outs, status


def weight_dequant_2d(codes, scales, tensor_scale, out=None, stream=None):
    """Dequantize 16x16-tiled NVFP4 weights to bf16 [M, N]."""
    torch = _torch()
    _check_cuda(codes, scales, tensor_scale)
    M, N2 = codes.shape
    if out is None:
        out = torch.empty((M, 2 * N2), dtype=torch.bfloat16, device=codes.device)
    st = _lib.nvfp4_weight_dequant_2d(_ptr(codes), _ptr(scales), _ptr(tensor_scale), M, 2 * N2, _ptr(out),
                                      _stream(stream))
    _lib.check(st, "nvfp4_weight_dequant_2d")
    return out
