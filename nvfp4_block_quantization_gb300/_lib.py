"""ctypes binding of the C ABI in include/nvfp4.h (argument marshalling only).

Every function here has the name and argument order of its C entry point.  The
library must have been built (``nvfp4_block_quantization_gb300.build.build()``
or ``__graft_entry__.build()``); there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

NVFP4_OK, NVFP4_EINVAL, NVFP4_ESHAPE, NVFP4_EALIGN, NVFP4_EWORKSPACE, NVFP4_ECUDA, NVFP4_ECAPACITY = range(7)
NVFP4_KVCACHE_MAX_SLOTS = 64
NVFP4_MAX_VIEW_FRAMES = 512
NVFP4_IN_BF16, NVFP4_IN_FP32 = 0, 1
NVFP4_DEV_OK, NVFP4_DEV_NONFINITE, NVFP4_DEV_TIMEOUT = 0, 1, 2

# Every entry point declared in include/nvfp4.h.
EXPORTS = (
    "nvfp4_status_string",
    "nvfp4_version",
    "nvfp4_kv_workspace_bytes",
    "nvfp4_kv_smooth_quant",
    "nvfp4_kv_batched_workspace_bytes",
    "nvfp4_kv_smooth_quant_batched",
    "nvfp4_kv_smooth_quant_headroom",
    "nvfp4_kv_stats_batched",
    "nvfp4_kv_quant_batched",
    "nvfp4_kv_dequant",
    "nvfp4_selftest_cvt",
    "nvfp4_kv_shard_bytes",
    "nvfp4_kv_pack_head_shards",
    "nvfp4_kv_unpack_head_shards",
    "nvfp4_kvcache_slots_needed",
    "nvfp4_kvcache_init",
    "nvfp4_kvcache_append",
    "nvfp4_kvcache_new_shot",
    "nvfp4_kvcache_view",
    "nvfp4_kv_gather_dequant",
    "nvfp4_kv_attention_workspace_bytes",
    "nvfp4_kv_attention_decode",
    "nvfp4_kv_attention_prefill_workspace_bytes",
    "nvfp4_kv_attention_prefill",
    "nvfp4_mma_scales_bytes",
    "nvfp4_scales_to_mma",
    "nvfp4_w2d_scales_to_mma",
    "nvfp4_rht16",
    "nvfp4_act_quant_workspace_bytes",
    "nvfp4_act_quant_mma",
    "nvfp4_gemm_workspace_bytes",
    "nvfp4_gemm_plan_create",
    "nvfp4_gemm_plan_destroy",
    "nvfp4_gemm_w4a4",
    "nvfp4_w2d_workspace_bytes",
    "nvfp4_weight_quant_2d",
    "nvfp4_w2d_batched_workspace_bytes",
    "nvfp4_weight_quant_2d_batched",
    "nvfp4_weight_quant_2d_static",
    "nvfp4_weight_dequant_2d",
)


class nvfp4_kv_job(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p),
        ("smooth", ctypes.c_int),
        ("mean_in", ctypes.c_void_p),
        ("mean_out", ctypes.c_void_p),
        ("codes", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("tensor_scale", ctypes.c_void_p),
    ]


class nvfp4_w2d_job(ctypes.Structure):
    _fields_ = [
        ("w", ctypes.c_void_p),
        ("M", ctypes.c_int64),
        ("N", ctypes.c_int64),
        ("codes", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("tensor_scale", ctypes.c_void_p),
    ]


class nvfp4_kvcache(ctypes.Structure):
    _fields_ = [
        ("frames_per_chunk", ctypes.c_int),
        ("global_sink", ctypes.c_int),
        ("shot_sink", ctypes.c_int),
        ("window", ctypes.c_int),
        ("n_slots", ctypes.c_int),
        ("tokens_per_frame", ctypes.c_int64),
        ("n_chunks", ctypes.c_int64),
        ("shot_start", ctypes.c_int64),
        ("slot_chunk", ctypes.c_int64 * NVFP4_KVCACHE_MAX_SLOTS),
    ]


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


_lib = None


def load(path: str | None = None):
    """Load the CUDA library; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"NVFP4 CUDA library not built ({path} missing): run "
                           "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.nvfp4_status_string.argtypes = [i32]
    lib.nvfp4_status_string.restype = ctypes.c_char_p
    lib.nvfp4_version.argtypes = []
    lib.nvfp4_version.restype = i32
    lib.nvfp4_kv_workspace_bytes.argtypes = [i64, i32, i32]
    lib.nvfp4_kv_workspace_bytes.restype = sz
    lib.nvfp4_kv_smooth_quant.argtypes = [vp, i32, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.nvfp4_kv_smooth_quant.restype = i32
    lib.nvfp4_kv_batched_workspace_bytes.argtypes = [i32, i64, i32, i32]
    lib.nvfp4_kv_batched_workspace_bytes.restype = sz
    lib.nvfp4_kv_smooth_quant_batched.argtypes = [ctypes.POINTER(nvfp4_kv_job), i32, i32, i64, i32, i32, vp, vp,
                                                  sz, vp]
    lib.nvfp4_kv_smooth_quant_batched.restype = i32
    lib.nvfp4_kv_smooth_quant_headroom.argtypes = [ctypes.POINTER(nvfp4_kv_job), i32, i32, i64, i32, i32, vp, vp,
                                                   sz, vp]
    lib.nvfp4_kv_smooth_quant_headroom.restype = i32
    lib.nvfp4_kv_stats_batched.argtypes = [ctypes.POINTER(nvfp4_kv_job), i32, i32, i64, i32, i32, vp, sz, vp]
    lib.nvfp4_kv_stats_batched.restype = i32
    lib.nvfp4_kv_quant_batched.argtypes = [ctypes.POINTER(nvfp4_kv_job), i32, i32, i64, i32, i32, vp, vp, sz, vp]
    lib.nvfp4_kv_quant_batched.restype = i32
    lib.nvfp4_kv_dequant.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, vp, vp]
    lib.nvfp4_kv_dequant.restype = i32
    lib.nvfp4_selftest_cvt.argtypes = [vp, i64, vp, vp, vp, vp, vp]
    lib.nvfp4_selftest_cvt.restype = i32
    lib.nvfp4_kv_shard_bytes.argtypes = [i64, i32, i32, i32, i32]
    lib.nvfp4_kv_shard_bytes.restype = sz
    lib.nvfp4_kv_pack_head_shards.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, vp, vp]
    lib.nvfp4_kv_pack_head_shards.restype = i32
    lib.nvfp4_kv_unpack_head_shards.argtypes = [vp, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.nvfp4_kv_unpack_head_shards.restype = i32
    P = ctypes.POINTER
    lib.nvfp4_kvcache_slots_needed.argtypes = [i32, i32, i32, i32]
    lib.nvfp4_kvcache_slots_needed.restype = i32
    lib.nvfp4_kvcache_init.argtypes = [P(nvfp4_kvcache), i32, i64, i32, i32, i32, i32]
    lib.nvfp4_kvcache_init.restype = i32
    lib.nvfp4_kvcache_append.argtypes = [P(nvfp4_kvcache), P(i32)]
    lib.nvfp4_kvcache_append.restype = i32
    lib.nvfp4_kvcache_new_shot.argtypes = [P(nvfp4_kvcache)]
    lib.nvfp4_kvcache_new_shot.restype = i32
    lib.nvfp4_kvcache_view.argtypes = [P(nvfp4_kvcache), vp, vp, vp, i32]
    lib.nvfp4_kvcache_view.restype = i32
    lib.nvfp4_kv_gather_dequant.argtypes = [vp, vp, vp, vp, i64, i32, vp, vp, i32, i64, i32, i32, vp, vp]
    lib.nvfp4_kv_gather_dequant.restype = i32
    lib.nvfp4_kv_attention_workspace_bytes.argtypes = [i32, i64, i32, i32, i32]
    lib.nvfp4_kv_attention_workspace_bytes.restype = sz
    lib.nvfp4_kv_attention_decode.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, i64, i32, vp, vp, i32, i64, i32,
                                              i32, ctypes.c_float, vp, vp, sz, vp]
    lib.nvfp4_kv_attention_decode.restype = i32
    lib.nvfp4_kv_attention_prefill_workspace_bytes.argtypes = [i64, i32, i32, i64]
    lib.nvfp4_kv_attention_prefill_workspace_bytes.restype = sz
    lib.nvfp4_kv_attention_prefill.argtypes = [vp, i64, vp, vp, vp, vp, vp, vp, vp, i64, i32, vp, vp, i32, i64, i32,
                                               i32, ctypes.c_float, vp, vp, sz, vp, vp]
    lib.nvfp4_kv_attention_prefill.restype = i32
    lib.nvfp4_mma_scales_bytes.argtypes = [i64, i64]
    lib.nvfp4_mma_scales_bytes.restype = i64
    lib.nvfp4_scales_to_mma.argtypes = [vp, i64, i64, vp, vp]
    lib.nvfp4_scales_to_mma.restype = i32
    lib.nvfp4_w2d_scales_to_mma.argtypes = [vp, i64, i64, vp, vp]
    lib.nvfp4_w2d_scales_to_mma.restype = i32
    lib.nvfp4_rht16.argtypes = [vp, i32, i64, i64, ctypes.c_uint32, vp, vp]
    lib.nvfp4_rht16.restype = i32
    lib.nvfp4_act_quant_workspace_bytes.argtypes = []
    lib.nvfp4_act_quant_workspace_bytes.restype = sz
    lib.nvfp4_act_quant_mma.argtypes = [vp, i64, i64, i32, ctypes.c_uint32, vp, vp, vp, vp, vp, sz, vp]
    lib.nvfp4_act_quant_mma.restype = i32
    lib.nvfp4_gemm_workspace_bytes.argtypes = []
    lib.nvfp4_gemm_workspace_bytes.restype = sz
    lib.nvfp4_gemm_plan_create.argtypes = [i64, i64, i64, P(vp)]
    lib.nvfp4_gemm_plan_create.restype = i32
    lib.nvfp4_gemm_plan_destroy.argtypes = [vp]
    lib.nvfp4_gemm_plan_destroy.restype = None
    lib.nvfp4_gemm_w4a4.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.nvfp4_gemm_w4a4.restype = i32
    lib.nvfp4_w2d_workspace_bytes.argtypes = [i64, i64]
    lib.nvfp4_w2d_workspace_bytes.restype = sz
    lib.nvfp4_weight_quant_2d.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp, vp, sz, vp]
    lib.nvfp4_weight_quant_2d.restype = i32
    lib.nvfp4_w2d_batched_workspace_bytes.argtypes = [i32]
    lib.nvfp4_w2d_batched_workspace_bytes.restype = sz
    lib.nvfp4_weight_quant_2d_batched.argtypes = [ctypes.POINTER(nvfp4_w2d_job), i32, i32, vp, vp, sz, vp]
    lib.nvfp4_weight_quant_2d_batched.restype = i32
    lib.nvfp4_weight_quant_2d_static.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp, vp]
    lib.nvfp4_weight_quant_2d_static.restype = i32
    lib.nvfp4_weight_dequant_2d.argtypes = [vp, vp, vp, i64, i64, vp, vp]
    lib.nvfp4_weight_dequant_2d.restype = i32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().nvfp4_status_string(int(status)).decode()


def check(status: int, what: str):
    if status != NVFP4_OK:
        raise NVFP4Error(status, what)


def nvfp4_version():
    return load().nvfp4_version()


def nvfp4_kv_workspace_bytes(T, H, D):
    return load().nvfp4_kv_workspace_bytes(T, H, D)


def nvfp4_kv_smooth_quant(x, dt, T, H, D, smooth, mean_in, mean_out, codes, scales, tensor_scale, dev_status,
                          workspace, workspace_bytes, stream):
    return load().nvfp4_kv_smooth_quant(x, dt, T, H, D, smooth, mean_in, mean_out, codes, scales, tensor_scale,
                                        dev_status, workspace, workspace_bytes, stream)


def nvfp4_kv_batched_workspace_bytes(n_jobs, T, H, D):
    return load().nvfp4_kv_batched_workspace_bytes(n_jobs, T, H, D)


def nvfp4_kv_smooth_quant_batched(jobs, n_jobs, dt, T, H, D, dev_status, workspace, workspace_bytes, stream):
    return load().nvfp4_kv_smooth_quant_batched(jobs, n_jobs, dt, T, H, D, dev_status, workspace, workspace_bytes,
                                                stream)


def nvfp4_kv_smooth_quant_headroom(jobs, n_jobs, dt, T, H, D, dev_status, workspace, workspace_bytes, stream):
    return load().nvfp4_kv_smooth_quant_headroom(jobs, n_jobs, dt, T, H, D, dev_status, workspace, workspace_bytes,
                                                 stream)


def nvfp4_kv_stats_batched(jobs, n_jobs, dt, T, H, D, workspace, workspace_bytes, stream):
    return load().nvfp4_kv_stats_batched(jobs, n_jobs, dt, T, H, D, workspace, workspace_bytes, stream)


def nvfp4_kv_quant_batched(jobs, n_jobs, dt, T, H, D, dev_status, workspace, workspace_bytes, stream):
    return load().nvfp4_kv_quant_batched(jobs, n_jobs, dt, T, H, D, dev_status, workspace, workspace_bytes, stream)


def nvfp4_kv_dequant(codes, scales, tensor_scale, mean, tokens_per_group, T, H, D, out_bf16, stream):
    return load().nvfp4_kv_dequant(codes, scales, tensor_scale, mean, tokens_per_group, T, H, D, out_bf16, stream)


def nvfp4_selftest_cvt(x, n, e2m1_codes, e4m3_codes, e2m1_pair_f16x2, e4m3_values, stream):
    return load().nvfp4_selftest_cvt(x, n, e2m1_codes, e4m3_codes, e2m1_pair_f16x2, e4m3_values, stream)


def nvfp4_kv_shard_bytes(T, H, D, P, with_mean):
    return load().nvfp4_kv_shard_bytes(T, H, D, P, with_mean)


def nvfp4_kv_pack_head_shards(codes, scales, tensor_scale, mean, T, H, D, P, out, stream):
    return load().nvfp4_kv_pack_head_shards(codes, scales, tensor_scale, mean, T, H, D, P, out, stream)


def nvfp4_kv_unpack_head_shards(src, T, H, D, P, with_mean, codes, scales, tensor_scales, means, stream):
    return load().nvfp4_kv_unpack_head_shards(src, T, H, D, P, with_mean, codes, scales, tensor_scales, means,
                                              stream)


def nvfp4_kvcache_slots_needed(frames_per_chunk, global_sink, shot_sink, window):
    return load().nvfp4_kvcache_slots_needed(frames_per_chunk, global_sink, shot_sink, window)


def nvfp4_kvcache_init(c, frames_per_chunk, tokens_per_frame, global_sink, shot_sink, window, n_slots):
    return load().nvfp4_kvcache_init(ctypes.byref(c), frames_per_chunk, tokens_per_frame, global_sink, shot_sink,
                                     window, n_slots)


def nvfp4_kvcache_append(c, slot):
    return load().nvfp4_kvcache_append(ctypes.byref(c), ctypes.byref(slot))


def nvfp4_kvcache_new_shot(c):
    return load().nvfp4_kvcache_new_shot(ctypes.byref(c))


def nvfp4_kvcache_view(c, frame_index, frame_row, frame_slot, max_frames):
    return load().nvfp4_kvcache_view(ctypes.byref(c), frame_index, frame_row, frame_slot, max_frames)


def nvfp4_kv_gather_dequant(codes_pool, scales_pool, g_pool, mean_pool, pool_rows, n_meta, frame_row, frame_meta,
                            n_frames, tokens_per_frame, H, D, out_bf16, stream):
    return load().nvfp4_kv_gather_dequant(codes_pool, scales_pool, g_pool, mean_pool, pool_rows, n_meta, frame_row,
                                          frame_meta, n_frames, tokens_per_frame, H, D, out_bf16, stream)


def nvfp4_kv_attention_workspace_bytes(n_frames, tokens_per_frame, H, D, n_q):
    return load().nvfp4_kv_attention_workspace_bytes(n_frames, tokens_per_frame, H, D, n_q)


def nvfp4_kv_attention_decode(q, n_q, k_codes, k_scales, k_g, k_mean, v_codes, v_scales, v_g, pool_rows, n_meta,
                              frame_row, frame_meta, n_frames, tokens_per_frame, H, D, scale, out, workspace,
                              workspace_bytes, stream):
    return load().nvfp4_kv_attention_decode(q, n_q, k_codes, k_scales, k_g, k_mean, v_codes, v_scales, v_g,
                                            pool_rows, n_meta, frame_row, frame_meta, n_frames, tokens_per_frame,
                                            H, D, scale, out, workspace, workspace_bytes, stream)


def nvfp4_kv_attention_prefill_workspace_bytes(n_q, H, n_frames, tokens_per_frame):
    return load().nvfp4_kv_attention_prefill_workspace_bytes(n_q, H, n_frames, tokens_per_frame)


def nvfp4_kv_attention_prefill(q, n_q, k_codes, k_scales, k_g, k_mean, v_codes, v_scales, v_g, pool_rows, n_meta,
                               frame_row, frame_meta, n_frames, tokens_per_frame, H, D, scale, out, workspace,
                               workspace_bytes, dev_status, stream):
    return load().nvfp4_kv_attention_prefill(q, n_q, k_codes, k_scales, k_g, k_mean, v_codes, v_scales, v_g,
                                             pool_rows, n_meta, frame_row, frame_meta, n_frames, tokens_per_frame,
                                             H, D, scale, out, workspace, workspace_bytes, dev_status, stream)


def nvfp4_mma_scales_bytes(rows, K):
    return load().nvfp4_mma_scales_bytes(rows, K)


def nvfp4_scales_to_mma(scales, rows, K, out, stream):
    return load().nvfp4_scales_to_mma(scales, rows, K, out, stream)


def nvfp4_w2d_scales_to_mma(scales, N, K, out, stream):
    return load().nvfp4_w2d_scales_to_mma(scales, N, K, out, stream)


def nvfp4_rht16(x, dt, rows, K, signs, out, stream):
    return load().nvfp4_rht16(x, dt, rows, K, signs, out, stream)


def nvfp4_act_quant_workspace_bytes():
    return load().nvfp4_act_quant_workspace_bytes()


def nvfp4_act_quant_mma(x, M, K, use_rht, signs, codes, scales_mma, tensor_scale, dev_status, workspace,
                        workspace_bytes, stream):
    return load().nvfp4_act_quant_mma(x, M, K, use_rht, signs, codes, scales_mma, tensor_scale, dev_status,
                                      workspace, workspace_bytes, stream)


def nvfp4_gemm_workspace_bytes():
    return load().nvfp4_gemm_workspace_bytes()


def nvfp4_gemm_plan_create(M, N, K, plan):
    return load().nvfp4_gemm_plan_create(M, N, K, ctypes.byref(plan))


def nvfp4_gemm_plan_destroy(plan):
    load().nvfp4_gemm_plan_destroy(plan)


def nvfp4_gemm_w4a4(plan, x_codes, x_scales_mma, x_tensor_scale, w_codes, w_scales_mma, w_tensor_scale, y_bf16,
                    workspace, workspace_bytes, stream):
    return load().nvfp4_gemm_w4a4(plan, x_codes, x_scales_mma, x_tensor_scale, w_codes, w_scales_mma, w_tensor_scale,
                                  y_bf16, workspace, workspace_bytes, stream)


def nvfp4_w2d_workspace_bytes(M, N):
    return load().nvfp4_w2d_workspace_bytes(M, N)


def nvfp4_weight_quant_2d(w, dt, M, N, codes, scales, tensor_scale, dev_status, workspace, workspace_bytes, stream):
    return load().nvfp4_weight_quant_2d(w, dt, M, N, codes, scales, tensor_scale, dev_status, workspace,
                                        workspace_bytes, stream)


def nvfp4_weight_quant_2d_static(w, dt, M, N, codes, scales, tensor_scale, dev_status, stream):
    return load().nvfp4_weight_quant_2d_static(w, dt, M, N, codes, scales, tensor_scale, dev_status, stream)


def nvfp4_weight_dequant_2d(codes, scales, tensor_scale, M, N, out_bf16, stream):
    return load().nvfp4_weight_dequant_2d(codes, scales, tensor_scale, M, N, out_bf16, stream)


def nvfp4_w2d_batched_workspace_bytes(n_jobs):
    return load().nvfp4_w2d_batched_workspace_bytes(n_jobs)


def nvfp4_weight_quant_2d_batched(jobs, n_jobs, dt, dev_status, workspace, workspace_bytes, stream):
    return load().nvfp4_weight_quant_2d_batched(jobs, n_jobs, dt, dev_status, workspace, workspace_bytes, stream)
