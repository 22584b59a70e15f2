/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 KV-cache quantizer.
 *
 * The method is the KV-cache write of "LongLive-2.0: An NVFP4 Parallel
 * Infrastructure for Long Video Generation" (summary page,
 * paper.rainbus.top/paper/2605.18739):
 *   - inference pipeline, step 7: each chunk of F_c = 8 latent frames
 *     (T_c = F_c * L_f tokens) has K smoothed, K <- K - mean(K) over the
 *     chunk's tokens, and is then quantized into the NVFP4 KV cache with
 *     4/6 adaptive block scales;
 *   - "full-stack NVFP4" paragraph: Four-Over-Six compares the MSE of two
 *     candidate FP8 block scales, keeping the +-6 range or switching to +-4;
 *   - training pipeline, step 4: 2-D block scales for weights, 1-D block
 *     scales for activations.
 * NVFP4: E2M1 elements {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6} in blocks of
 * 16, one E4M3 scale per block (round-to-nearest-even, saturating at 448) and
 * one fp32 scale per tensor, g = amax / 2688 (2688 = 6 * 448).  Per block the
 * candidate scales e_M = E4M3(a_b * fl(1 / fl(M * g))), M in {6, 4}, map the
 * block's absolute maximum a_b to 6 and to 4; the block is quantized under
 * both (y = Z * fl(1 / fl(E_M * g)), codes round to nearest even, sign kept),
 * each candidate's error is E_M^2 * sum (y - Q)^2 (fused multiply-add per
 * element, element order), and the lower error wins, ties going to 6.
 *
 * Conventions for every entry point:
 *   - Device pointers name GPU global memory owned by the caller; the library
 *     never allocates device memory, never frees, synchronizes or prints, and
 *     keeps no mutable global state (it is safe to call from several host
 *     threads).  Two entry points say otherwise where they are declared: the
 *     GEMM plan is a host object the library allocates for the caller, and
 *     nvfp4_weight_quant_2d_static uses a scratch array inside the library.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously; outputs are valid once the stream
 *     reaches that point.
 *   - Argument errors are returned synchronously and nothing is enqueued.
 *     A failed launch returns NVFP4_ECUDA (cudaGetLastError is consumed).
 *   - Data-dependent conditions are written by the kernels to *dev_status (a
 *     device int, optional): NVFP4_DEV_OK, or NVFP4_DEV_NONFINITE when a
 *     smoothed value is NaN or infinite.  Then every scale byte is 0x7F
 *     (E4M3 NaN), every code 0 and the tensor scale NaN, so a later dequant
 *     yields NaN rather than plausible numbers.
 *   - Quantizer inputs x must be 32-byte aligned; codes, scales and dequant
 *     outputs 16-byte aligned (NVFP4_EALIGN otherwise); float pointers 4-byte
 *     aligned.
 *   - Sizes are 64-bit; T may be 0 (nothing but the tensor scale, 0, and the
 *     mean, 0, is written).
 *
 * Layouts (row-major):
 *   input  x       [T][H][D]   bf16 or fp32, D contiguous, D % 16 == 0
 *   codes          [T][H][D/2] byte j of a row = element 2j (low nibble) and
 *                              element 2j+1 (high nibble), E2M1 sign-magnitude
 *   scales         [T][H][D/16] one E4M3 byte per 16 consecutive d
 *   tensor_scale   one fp32 per quantized tensor (g)
 *   mean           [H][D] fp32 per chunk (the mean that K-smoothing removed)
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_EINVAL = 1,     /* a required pointer is NULL, or an enum/flag is out of range */
  NVFP4_ESHAPE = 2,     /* a size is out of range (D % 16, H <= 0, T < 0, M/N % 16, ...) */
  NVFP4_EALIGN = 3,     /* a pointer is not aligned as required */
  NVFP4_EWORKSPACE = 4, /* workspace NULL, too small, or not 256-byte aligned */
  NVFP4_ECUDA = 5,      /* a CUDA runtime call or kernel launch failed */
  NVFP4_ECAPACITY = 6   /* the KV-cache pool has no free chunk slot */
} nvfp4_status;

typedef enum nvfp4_in_dtype {
  NVFP4_IN_BF16 = 0, /* bfloat16 elements, widened to fp32 exactly */
  NVFP4_IN_FP32 = 1  /* fp32 elements */
} nvfp4_in_dtype;

#define NVFP4_DEV_OK 0
#define NVFP4_DEV_NONFINITE 1 /* bit: a smoothed value was NaN or infinite */
#define NVFP4_DEV_TIMEOUT 2   /* bit: a bounded cross-CTA wait ran out */

/* Human-readable name of a status code (static string, never NULL). */
const char* nvfp4_status_string(nvfp4_status s);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int nvfp4_version(void);

/* ------------------------------------------------------------------------ */
/* KV chunk quantizer (LongLive-2.0 summary page, inference step 7, and the */
/* "full-stack NVFP4" paragraph).                                            */
/* ------------------------------------------------------------------------ */

/* Bytes of device workspace one nvfp4_kv_smooth_quant call needs for this
 * shape on the current device.  Returns 0 for invalid shapes. */
size_t nvfp4_kv_workspace_bytes(int64_t T, int H, int D);

/* Quantize one chunk tensor x[T][H][D] into NVFP4 with Four-Over-Six scales.
 *   x            device, [T][H][D] of `dt`, 32-byte aligned
 *   smooth       1: K-smoothing -- subtract mean[h][d] = (sum over the chunk's
 *                T tokens of x[t][h][d]) / T, rounded once to fp32, before
 *                quantizing (keys); 0: no smoothing (values, activations)
 *   mean_in      device [H*D] or NULL; when set (smooth must be 1) it is used
 *                as the mean instead of computing it
 *   mean_out     device [H*D] or NULL (smooth must be 1); receives the mean used
 *   codes        device [T*H*D/2] output, packed E2M1 nibbles
 *   scales       device [T*H*D/16] output, E4M3 bytes
 *   tensor_scale device [1] output, g = amax / 2688 of the smoothed tensor
 *   dev_status   device int or NULL, see the conventions above
 *   workspace    device scratch of at least nvfp4_kv_workspace_bytes(T, H, D)
 *                bytes, 256-byte aligned, ZERO-FILLED before its first use
 *                (e.g. cudaMemset).  It holds the cross-CTA counters of the
 *                fused kernel, which every completed call returns to zero, so
 *                the same workspace serves later calls on one stream without
 *                clearing.  Calls that share a workspace must not overlap.
 *   stream       cudaStream_t
 * Implementation: a cooperative statistics grid (one CTA per SM: channel sums,
 * minima and maxima, the means and the tensor's absolute maximum) followed by a
 * quantization grid launched as its programmatic dependent, whose CTAs wait
 * for their own tensor's statistics.  Both grids' cross-CTA waits are bounded
 * (about 2 s); if one runs out, *dev_status gets NVFP4_DEV_TIMEOUT, the
 * affected outputs are left unwritten and the workspace must be zero-filled
 * again before reuse.
 * Errors: NVFP4_EINVAL (NULL x/codes/scales/tensor_scale, bad dt or smooth,
 * mean pointers with smooth == 0), NVFP4_ESHAPE (also T*H*D > 2^46),
 * NVFP4_EALIGN, NVFP4_EWORKSPACE, NVFP4_ECUDA. */
nvfp4_status nvfp4_kv_smooth_quant(const void* x, nvfp4_in_dtype dt, int64_t T, int H, int D, int smooth,
                                   const float* mean_in, float* mean_out, uint8_t* codes, uint8_t* scales,
                                   float* tensor_scale, int* dev_status, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* One tensor of a batched call (all tensors of a batch share T, H, D, dt). */
typedef struct nvfp4_kv_job {
  const void* x;        /* device [T][H][D] input */
  int smooth;           /* 1 = K (smoothed), 0 = V */
  const float* mean_in; /* device [H*D] or NULL */
  float* mean_out;      /* device [H*D] or NULL */
  uint8_t* codes;       /* device [T*H*D/2] */
  uint8_t* scales;      /* device [T*H*D/16] */
  float* tensor_scale;  /* device [1] */
} nvfp4_kv_job;

/* Workspace for nvfp4_kv_smooth_quant_batched with n_jobs tensors. */
size_t nvfp4_kv_batched_workspace_bytes(int n_jobs, int64_t T, int H, int D);

/* Quantize n_jobs independent chunk tensors (e.g. K and V of every layer of
 * one chunk) in one enqueue; each job gets exactly the result the single
 * call would give it.  `jobs` is a HOST array read before the call returns.
 * *dev_status is the OR over jobs.  Errors as nvfp4_kv_smooth_quant, plus
 * NVFP4_EINVAL for n_jobs < 1 or a bad job. */
nvfp4_status nvfp4_kv_smooth_quant_batched(const nvfp4_kv_job* jobs, int n_jobs, nvfp4_in_dtype dt,
                                           int64_t T, int H, int D, int* dev_status, void* workspace,
                                           size_t workspace_bytes, void* stream);

/* nvfp4_kv_smooth_quant_batched with E4M3 headroom in the tensor scale:
 * g = fl(amax / 1792), 1792 = 4 * 448, instead of amax / 2688.  The pages fix
 * no per-tensor scale formula.  With 2688 (the standard two-level NVFP4 scale)
 * a block above 2/3 of the tensor amax has its 4-candidate saturate at 448, so
 * the block holding the amax always keeps 6; 1792 is the largest denominator
 * at which every block's 4-candidate fits under 448, so every block can choose
 * between the two ranges ("LongLive-2.0" summary page, "full-stack NVFP4"
 * paragraph: Four-Over-Six).  Everything else -- candidates, errors, ties,
 * layouts, dequant -- is unchanged; the dequant of these outputs is
 * nvfp4_kv_dequant with the tensor scale this call writes.  Arguments,
 * workspace and errors as nvfp4_kv_smooth_quant_batched. */
nvfp4_status nvfp4_kv_smooth_quant_headroom(const nvfp4_kv_job* jobs, int n_jobs, nvfp4_in_dtype dt, int64_t T,
                                            int H, int D, int* dev_status, void* workspace,
                                            size_t workspace_bytes, void* stream);

/* The two passes of nvfp4_kv_smooth_quant_batched as separate enqueues, for a
 * caller that wants to schedule them apart (e.g. the statistics of one tensor
 * on one stream while another tensor is quantized on a second stream).
 * nvfp4_kv_stats_batched computes, for every job, the channel means (written to
 * mean_out when set) and the tensor's absolute maximum, and leaves them in the
 * workspace; nvfp4_kv_quant_batched then quantizes with them, writes codes,
 * scales and tensor scales, publishes *dev_status (covering both passes) and
 * returns the workspace to its idle state.  The quantization call must follow
 * the statistics call on the same stream (or after an event that orders it),
 * with the same jobs in the same order, the same shape and dtype, and the same
 * workspace; nothing else may use that workspace in between.  A statistics call
 * without its quantization call leaves the workspace dirty (zero-fill it
 * again).  Arguments and errors as nvfp4_kv_smooth_quant_batched. */
nvfp4_status nvfp4_kv_stats_batched(const nvfp4_kv_job* jobs, int n_jobs, nvfp4_in_dtype dt, int64_t T, int H,
                                    int D, void* workspace, size_t workspace_bytes, void* stream);
nvfp4_status nvfp4_kv_quant_batched(const nvfp4_kv_job* jobs, int n_jobs, nvfp4_in_dtype dt, int64_t T, int H,
                                    int D, int* dev_status, void* workspace, size_t workspace_bytes, void* stream);

/* Dequantize an NVFP4 KV cache back to bf16 (the cache read that attention
 * performs; LongLive-2.0 summary page, inference steps 7 and 9).
 *   codes, scales     device, layouts above, for T tokens
 *   tensor_scale      device [G], G = ceil(T / tokens_per_group): token t uses
 *                     tensor_scale[t / tokens_per_group] (one chunk: pass
 *                     tokens_per_group = T; a cache assembled from frames of
 *                     different chunks: per-frame groups, e.g. 880)
 *   mean              device [G][H][D] or NULL; when set the group's mean is
 *                     added back (undoes K-smoothing)
 *   out_bf16          device [T][H][D] bf16 output:
 *                     bf16_rne(fl(fl(Q * fl(E * g)) + mean))
 * Errors: NVFP4_EINVAL, NVFP4_ESHAPE (tokens_per_group < 1 ...), NVFP4_EALIGN,
 * NVFP4_ECUDA. */
nvfp4_status nvfp4_kv_dequant(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                              const float* mean, int64_t tokens_per_group, int64_t T, int H, int D,
                              void* out_bf16, void* stream);

/* Self-test of the conversion instructions (the pages have no counterpart):
 * runs, on caller-provided values, exactly the rounding and decoding steps the
 * quantizers above use, so that a test can compare them with a software
 * statement of the formats.
 *   x                device [n] fp32 inputs (4-byte aligned)
 *   e2m1_codes       device [n]: byte i holds x[i]'s E2M1 code (round to nearest
 *                    even, saturating at 6, sign kept) in both nibbles -- one per
 *                    lane of the paired conversion the quantizers use
 *   e4m3_codes       device [n] uint16: x[i]'s E4M3 code (round to nearest even,
 *                    saturating at 448; NaN in, NaN code out) in both bytes
 *   e2m1_pair_f16x2  device [256]: entry b is byte b decoded as two E2M1 codes,
 *                    f16 pair (low half = low nibble)
 *   e4m3_values      device [256]: entry b is E4M3 code b as fp32 (0x7F/0xFF: NaN)
 * Errors: NVFP4_ESHAPE (n < 0), NVFP4_EINVAL (NULL pointers), NVFP4_EALIGN,
 * NVFP4_ECUDA. */
nvfp4_status nvfp4_selftest_cvt(const float* x, int64_t n, uint8_t* e2m1_codes, uint16_t* e4m3_codes,
                                uint32_t* e2m1_pair_f16x2, float* e4m3_values, void* stream);

/* ------------------------------------------------------------------------ */
/* Head shards of a quantized KV tensor for a sequence-parallel exchange     */
/* ("LongLive-2.0" summary page: Ulysses SP all-to-all; the page credits the */
/* 4-bit KV cache with the time saved at SP = 2 and 4, Table 6).             */
/* ------------------------------------------------------------------------ */
/* A quantized tensor [T][H][..] (codes, scales, tensor scale, optional mean)
 * is cut into P head shards of H / P heads.  Shard p is one contiguous,
 * 16-byte aligned segment of nvfp4_kv_shard_bytes(T, H, D, P, with_mean)
 * bytes, so one all-to-all of P equal segments sends shard p to rank p:
 *   [16 B: tensor scale g (fp32), then zeros]
 *   [the shard's mean, (H / P) * D fp32, only with_mean]
 *   [codes of the shard, [T][H/P][D/2], padded to a multiple of 16 bytes]
 *   [scales of the shard, [T][H/P][D/16], padded to a multiple of 16 bytes]
 * Returns 0 for invalid shapes (H % P != 0 among them). */
size_t nvfp4_kv_shard_bytes(int64_t T, int H, int D, int P, int with_mean);

/* Packs codes [T][H][D/2], scales [T][H][D/16], tensor_scale (device [1]) and
 * mean (device [H][D] or NULL) into out (device, P segments, 16-byte aligned).
 * Errors: NVFP4_ESHAPE (also H % P != 0), NVFP4_EINVAL, NVFP4_EALIGN,
 * NVFP4_ECUDA. */
nvfp4_status nvfp4_kv_pack_head_shards(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                                       const float* mean, int64_t T, int H, int D, int P, void* out, void* stream);

/* Unpacks P segments (segment r from rank r, each holding that rank's T tokens
 * of this rank's H / P heads) by stacking them along the token axis:
 * codes [P*T][H/P][D/2], scales [P*T][H/P][D/16], tensor_scales device [P]
 * (segment r's g), means device [P][H/P][D] (with_mean) or NULL.  The result
 * is a cache of P groups of T tokens: nvfp4_kv_dequant with tokens_per_group
 * = T reads it.  Errors as nvfp4_kv_pack_head_shards. */
nvfp4_status nvfp4_kv_unpack_head_shards(const void* in, int64_t T, int H, int D, int P, int with_mean,
                                         uint8_t* codes, uint8_t* scales, float* tensor_scales, float* means,
                                         void* stream);

/* ------------------------------------------------------------------------ */
/* Multi-shot NVFP4 KV cache (LongLive-2.0 summary page, inference step 9:  */
/* attention over a Global Sink, the first S_g frames of the video, plus a  */
/* Shot-Level Sink, the first S_s frames of the current shot, held as       */
/* START/LEN pointers into frames already cached; a prompt switch rebinds   */
/* the shot sink.  Step 7: the cache is written one chunk of F_c frames at  */
/* a time).                                                                 */
/* ------------------------------------------------------------------------ */
/* The local part of the attention is read as a rolling window of the W
 * frames right before the chunk being generated.  The view of chunk n (first
 * frame cur = n * F_c) is the union, in ascending frame order and without
 * repeats, of [0, S_g), [START, START + S_s) and [cur - W, cur), each clipped
 * to the cached frames [0, cur).
 *
 * Storage, per cached tensor (each layer's K, each layer's V), is a pool of
 * chunk slots that the caller allocates on the device:
 *   codes   [n_slots * F_c * L_f][H][D/2]    scales [n_slots * F_c * L_f][H][D/16]
 *   g       [n_slots] fp32                   mean   [n_slots][H][D] fp32 (K only)
 * Slot s holds one chunk; its frame i is pool rows [(s F_c + i) L_f, (s F_c + i + 1) L_f).
 * The quantizer writes a chunk straight into its slot: x of F_c * L_f tokens,
 * codes and scales at pool row s * F_c * L_f, tensor_scale = g + s,
 * mean_out = mean + s * H * D.  Nothing is copied.
 *
 * The manager is host bookkeeping in a caller-owned struct: it makes no CUDA
 * call and touches no device memory.  Release rule: when chunk n is written,
 * a slot is freed if none of its chunk's frames can be in the view of chunk
 * n + 1 or a later one (windows only move forward; a new shot sink covers only
 * frames not yet written).  So a view stays valid until the next append. */
#define NVFP4_KVCACHE_MAX_SLOTS 64
typedef struct nvfp4_kvcache {
  int frames_per_chunk;     /* F_c */
  int global_sink;          /* S_g frames */
  int shot_sink;            /* S_s frames */
  int window;               /* W frames */
  int n_slots;              /* chunk slots in the pool, <= NVFP4_KVCACHE_MAX_SLOTS */
  int64_t tokens_per_frame; /* L_f */
  int64_t n_chunks;         /* chunks written so far; the next one is chunk n_chunks */
  int64_t shot_start;       /* START: first frame of the current shot */
  int64_t slot_chunk[NVFP4_KVCACHE_MAX_SLOTS]; /* chunk held by each slot, -1 = free */
} nvfp4_kvcache;

/* Chunk slots that always suffice: ceil(S_g/F_c) + ceil(S_s/F_c) +
 * max(1, ceil(W/F_c)); -1 for invalid sizes or more than the maximum. */
int nvfp4_kvcache_slots_needed(int frames_per_chunk, int global_sink, int shot_sink, int window);

/* An empty cache (one shot starting at frame 0).  NVFP4_ESHAPE for sizes out
 * of range (F_c < 1, L_f < 1, negative sinks or window, n_slots outside
 * [1, NVFP4_KVCACHE_MAX_SLOTS]); NVFP4_EINVAL for a NULL struct. */
nvfp4_status nvfp4_kvcache_init(nvfp4_kvcache* c, int frames_per_chunk, int64_t tokens_per_frame, int global_sink,
                                int shot_sink, int window, int n_slots);

/* Chunk n_chunks is about to be written: frees the slots the release rule
 * allows, stores the new chunk in the lowest free slot (*slot) and counts it.
 * NVFP4_ECAPACITY (nothing changed but the releases) when every slot is live. */
nvfp4_status nvfp4_kvcache_append(nvfp4_kvcache* c, int* slot);

/* Prompt switch: the next chunk is the first of a new shot (START = its first
 * frame); the old shot's sink frames become releasable. */
nvfp4_status nvfp4_kvcache_new_shot(nvfp4_kvcache* c);

/* The view of chunk n_chunks: per frame, in order, its video frame index, its
 * first pool row and its slot (each output array optional, host memory).
 * Returns the frame count (at most S_g + S_s + W), or -1 when max_frames is
 * too small (nothing written) or the struct is inconsistent. */
int nvfp4_kvcache_view(const nvfp4_kvcache* c, int64_t* frame_index, int64_t* frame_row, int* frame_slot,
                       int max_frames);

/* Frames one gathered read can take (its frame table is a kernel parameter). */
#define NVFP4_MAX_VIEW_FRAMES 512

/* Gathered cache read: expands n_frames view frames of tokens_per_frame (L_f)
 * tokens each from a chunk-slot pool into out_bf16 [n_frames * L_f][H][D],
 * frame i's tokens from pool rows [frame_row[i], frame_row[i] + L_f) with the
 * tensor scale g_pool[frame_meta[i]] and, when mean_pool is set, the mean
 * mean_pool[frame_meta[i]][H][D] added back: bf16_rne(fl(fl(Q * fl(E * g)) + mean))
 * per element, as nvfp4_kv_dequant.
 *   codes_pool, scales_pool  device, pool_rows rows (layouts above)
 *   g_pool, mean_pool        device, n_meta entries (mean_pool may be NULL)
 *   frame_row, frame_meta    HOST arrays of n_frames entries (the view of
 *                            nvfp4_kvcache_view: frame_meta = frame_slot)
 * Every frame must lie inside the pool and every frame_meta inside [0, n_meta):
 * NVFP4_ESHAPE otherwise, checked before anything is enqueued.  n_frames = 0
 * enqueues nothing.  Alignment and other errors as nvfp4_kv_dequant. */
nvfp4_status nvfp4_kv_gather_dequant(const uint8_t* codes_pool, const uint8_t* scales_pool, const float* g_pool,
                                     const float* mean_pool, int64_t pool_rows, int n_meta, const int64_t* frame_row,
                                     const int* frame_meta, int n_frames, int64_t tokens_per_frame, int H, int D,
                                     void* out_bf16, void* stream);

/* Attention that reads the cache (inference steps 7 and 9): n_q query tokens
 * per head attend over one view, K and V dequantized in registers from their
 * pools, so the cache is read at 0.5625 bytes per element.  Per view token t
 * (pool row frame_row[t / L_f] + t % L_f, slot frame_meta[t / L_f]) and channel d,
 * with S = fl(E * g[slot]) the scale of d's 16-channel block:
 *   k = Q S_k + k_mean[slot][h][d]   (k_mean may be NULL),   v = Q S_v
 *   out[i][h][:] = sum_t softmax_t(scale * q[i][h] . k_t) v_t
 * all in fp32: over each block q . k is taken as S_k (q . Q) + q . mean and p v
 * as (p S_v) Q; the softmax is online over token ranges (256 to 2048 tokens,
 * sized so that heads x ranges is one wave of the CTAs the GPU holds at once),
 * merged exactly as a softmax of the union; out fp32.
 *   q          device [n_q][H][D] fp32, n_q in 1..4, D 64 or 128
 *   k_*, v_*   the pools of nvfp4_kv_gather_dequant (pool_rows rows, n_meta slots;
 *              codes 16-byte aligned, k_mean 16-byte aligned)
 *   frame_row, frame_meta  HOST arrays of n_frames (<= NVFP4_MAX_VIEW_FRAMES)
 *              entries, validated before anything is enqueued (NVFP4_ESHAPE)
 *   workspace  device, nvfp4_kv_attention_workspace_bytes(...), 256-byte aligned */
size_t nvfp4_kv_attention_workspace_bytes(int n_frames, int64_t tokens_per_frame, int H, int D, int n_q);
nvfp4_status nvfp4_kv_attention_decode(const float* q, int n_q, const uint8_t* k_codes, const uint8_t* k_scales,
                                       const float* k_g, const float* k_mean, const uint8_t* v_codes,
                                       const uint8_t* v_scales, const float* v_g, int64_t pool_rows, int n_meta,
                                       const int64_t* frame_row, const int* frame_meta, int n_frames,
                                       int64_t tokens_per_frame, int H, int D, float scale, float* out,
                                       void* workspace, size_t workspace_bytes, void* stream);

/* Attention of a block of query tokens (prefill: a whole new chunk) over one
 * view of the cache on the tensor cores (inference steps 7 and 9).  Per view
 * token t (pool row frame_row[t / L_f] + t % L_f, slot frame_meta[t / L_f]) and
 * channel d, as nvfp4_kv_attention_decode:
 *   k = Q S_k + k_mean[slot][h][d] (k_mean may be NULL),   v = Q S_v,
 *   out[i][h][:] = sum_t softmax_t(scale * q[i][h] . k_t) v_t.
 * Computed as: K' = Q E_k and V' = Q E_v, exact in bf16, in shared memory;
 * s = scale * (g_k (q . K') + q . mean) with q . K' summed in fp32 by
 * tcgen05.mma and q . mean in fp32; one pass over the view in tiles of 64
 * keys with a running maximum m that moves when a tile exceeds it by more
 * than 8 (base 2; O and l are then rescaled); P' = bf16(2^(s log2 e - m)
 * g_v / G), G the largest g_v of the view, accumulated as O += P' V' in fp32
 * on the tensor cores, l = sum 2^(s log2 e - m) in fp32; out = G O / l in
 * fp32.  P' is the only value rounded below fp32 (relative 2^-9); 2^x is the
 * hardware approximation (relative error below 2^-22).
 *   q_bf16     device [n_q][H][D] bf16, 16-byte aligned; D = 128
 *   k_*, v_*   the pools of nvfp4_kv_gather_dequant: codes 16-byte aligned,
 *              scales 8-byte aligned, k_mean 4-byte aligned (NVFP4_EALIGN)
 *   frame_row, frame_meta  HOST arrays of n_frames (<= NVFP4_MAX_VIEW_FRAMES)
 *              entries, validated before anything is enqueued; at most 16
 *              distinct slots in one view (NVFP4_ESHAPE otherwise)
 *   out        device [n_q][H][D] fp32, 16-byte aligned
 *   workspace  device scratch, 16-byte aligned, or NULL: with at least
 *              nvfp4_kv_attention_prefill_workspace_bytes(...) bytes (else
 *              NVFP4_EINVAL) the (query tile, head) units of the last, partial
 *              wave of CTAs run as two CTAs over the two halves of the view's
 *              keys each, merged by a second kernel on the same stream:
 *              out = (o_0 w_0 + o_1 w_1) / (w_0 + w_1), o_i = G O_i / l_i of
 *              half i, w_i = l_i 2^(m_i - max(m_0, m_1)).  NULL: every unit runs
 *              whole.  Owned by the caller, free again once the call's work on
 *              `stream` is done.
 *   dev_status device int or NULL: NVFP4_DEV_TIMEOUT is OR-ed in when a
 *              bounded wait for the tensor cores gave up (out then incomplete)
 * One CTA per 256 queries and head (a split unit: two). */
/* Workspace bytes for nvfp4_kv_attention_prefill on the current device: 0
 * when no unit would be split (or the shape is invalid). */
size_t nvfp4_kv_attention_prefill_workspace_bytes(int64_t n_q, int H, int n_frames, int64_t tokens_per_frame);
nvfp4_status nvfp4_kv_attention_prefill(const void* q_bf16, int64_t n_q, const uint8_t* k_codes,
                                        const uint8_t* k_scales, const float* k_g, const float* k_mean,
                                        const uint8_t* v_codes, const uint8_t* v_scales, const float* v_g,
                                        int64_t pool_rows, int n_meta, const int64_t* frame_row,
                                        const int* frame_meta, int n_frames, int64_t tokens_per_frame, int H, int D,
                                        float scale, float* out, void* workspace, size_t workspace_bytes,
                                        int* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Weights with 16x16 2-D blocks (LongLive-2.0 summary page, training        */
/* pipeline step 4: "2-D block scales for weights").                         */
/* ------------------------------------------------------------------------ */

/* Workspace for nvfp4_weight_quant_2d on an M x N matrix (current device). */
size_t nvfp4_w2d_workspace_bytes(int64_t M, int64_t N);

/* Quantize w[M][N] (M, N multiples of 16) with one E4M3 scale per 16x16 tile
 * and Four-Over-Six selection; each tile's error sums its 256 elements in
 * row-major order.  No smoothing.
 *   codes        device [M][N/2], same nibble packing as the KV codes
 *   scales       device [M/16][N/16] E4M3 bytes
 *   tensor_scale device [1]
 * Errors as nvfp4_kv_smooth_quant (NVFP4_ESHAPE also for M * N > 2^46). */
nvfp4_status nvfp4_weight_quant_2d(const void* w, nvfp4_in_dtype dt, int64_t M, int64_t N, uint8_t* codes,
                                   uint8_t* scales, float* tensor_scale, int* dev_status, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* One matrix of a batched weight call (the matrices may differ in shape). */
typedef struct nvfp4_w2d_job {
  const void* w;        /* device [M][N] input */
  int64_t M, N;         /* multiples of 16; M may be 0 */
  uint8_t* codes;       /* device [M][N/2] */
  uint8_t* scales;      /* device [M/16][N/16] */
  float* tensor_scale;  /* device [1], this matrix's g */
} nvfp4_w2d_job;

/* Workspace for nvfp4_weight_quant_2d_batched (a few hundred bytes, the same
 * for every n_jobs >= 1); 0 for n_jobs < 1. */
size_t nvfp4_w2d_batched_workspace_bytes(int n_jobs);

/* Quantize n_jobs independent weight matrices (e.g. all linear layers of a
 * block) in one enqueue: each matrix gets exactly the result
 * nvfp4_weight_quant_2d would give it, with its own tensor scale.  `jobs` is a
 * HOST array read before the call returns; matrices beyond 64 go into further
 * launch pairs on the same stream.  *dev_status is the OR over matrices.
 * Implementation: an amax grid takes the matrices one after another (smallest
 * first) and publishes each one's amax when complete; the quantization grid
 * runs beside it and starts on a matrix as soon as its amax is published
 * (bounded waits of about 2 s; if one runs out, *dev_status gets
 * NVFP4_DEV_TIMEOUT, that matrix is written as for a non-finite amax and the
 * workspace must be zero-filled again).
 * The workspace (at least nvfp4_w2d_batched_workspace_bytes(n_jobs) bytes,
 * 256-byte aligned) must be ZERO-FILLED before its first use; every completed
 * call leaves it zero, so later calls on one stream reuse it without clearing.
 * Calls that share it must not overlap.
 * Errors: NVFP4_EINVAL (NULL jobs, n_jobs < 1, bad dt or a NULL pointer in a
 * job), NVFP4_ESHAPE, NVFP4_EALIGN, NVFP4_EWORKSPACE, NVFP4_ECUDA. */
nvfp4_status nvfp4_weight_quant_2d_batched(const nvfp4_w2d_job* jobs, int n_jobs, nvfp4_in_dtype dt,
                                           int* dev_status, void* workspace, size_t workspace_bytes, void* stream);

/* nvfp4_weight_quant_2d without a workspace.  The pages have no counterpart:
 * this call exists for callers that cannot allocate device memory or hand the
 * library a scratch buffer -- e.g. a runtime that passes the library only the
 * tensors it reads and writes, or code that must not call into an allocator
 * at that point.  Its scratch (the per-CTA amax partials, 4 per SM) is a
 * file-scope device array inside the library of 4096 entries: the call returns
 * NVFP4_EWORKSPACE on a device with more than 1024 SMs.  Every call looks up
 * the array's device address (cudaGetSymbolAddress with the caller's device
 * current), so a call after a device reset uses the array of the new context.
 * The first call on a device may load the library's device code: make it
 * before capturing a stream.  All calls on a
 * device share the one array, so calls that overlap in time (several streams
 * or host threads) race: order them.  Results, arguments and other errors are
 * those of nvfp4_weight_quant_2d. */
nvfp4_status nvfp4_weight_quant_2d_static(const void* w, nvfp4_in_dtype dt, int64_t M, int64_t N, uint8_t* codes,
                                          uint8_t* scales, float* tensor_scale, int* dev_status, void* stream);

/* Dequantize 16x16-tiled NVFP4 weights to bf16 out[M][N]
 * (bf16_rne(fl(Q * fl(E * g)))).  tensor_scale is device [1]. */
nvfp4_status nvfp4_weight_dequant_2d(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                                     int64_t M, int64_t N, void* out_bf16, void* stream);

/* ------------------------------------------------------------------------ */
/* W4A4 NVFP4 GEMM (LongLive-2.0 summary page, training step 4: NVFP4 GEMMs  */
/* with 2-D block scales for weights and 1-D for activations; inference     */
/* step 6: a W4A4 model).                                                   */
/* ------------------------------------------------------------------------ */
/* Y[M][N] = bf16_rne(fl(gX * gW) * sum_k (QX * EX)[m][k] * (QW * EW)[n][k]), the
 * sum accumulated in fp32 by the tensor cores (a hand-written tcgen05 kernel:
 * E2M1 operands with one UE4M3 block scale per 16 elements of K, fp32
 * accumulation in TMEM).  X is an activation quantized by the 1-D quantizer
 * (nvfp4_kv_smooth_quant with H = 1, D = K, no smoothing): codes [M][K/2],
 * scales [M][K/16].  W is a weight quantized by nvfp4_weight_quant_2d: codes
 * [N][K/2], scales [N/16][K/16].
 *
 * The tensor cores read block scales in their own layout: per operand, tiles
 * of 128 rows x 4 blocks (64 elements of K), 512 bytes each, K tiles fastest;
 * inside a tile, block c of row r sits at byte (r % 32) * 16 + (r / 32) * 4 + c.
 * Rows past the operand and blocks past K/16 are zero. */

/* Bytes of an operand's scales in that layout: roundup(rows, 128) *
 * roundup(K / 16, 4); 0 for invalid sizes. */
int64_t nvfp4_mma_scales_bytes(int64_t rows, int64_t K);

/* Row-major 1-D block scales [rows][K/16] (device) -> the tensor-core layout
 * (device, nvfp4_mma_scales_bytes(rows, K) bytes, 16-byte aligned, padding
 * zeroed). */
nvfp4_status nvfp4_scales_to_mma(const uint8_t* scales, int64_t rows, int64_t K, uint8_t* out, void* stream);

/* 16x16-tile weight scales [N/16][K/16] (device) -> per-row block scales in the
 * tensor-core layout for N rows (each tile's scale repeated for its 16 rows). */
nvfp4_status nvfp4_w2d_scales_to_mma(const uint8_t* scales, int64_t N, int64_t K, uint8_t* out, void* stream);

/* Random Hadamard transform against outliers (the GEMM path's RHT): along each
 * row of x[rows][K] (bf16 or fp32, 32-byte aligned, K % 16 == 0), every block
 * of 16 elements becomes y = (x D) H / 4 in fp32: D = diag(+-1), element i
 * negated where bit i of `signs` (the random draw, 16 bits, an input) is set;
 * H the 16-point Sylvester Hadamard matrix, applied by the radix-2 butterflies
 * with strides 1, 2, 4, 8, each pair (a, b) -> (fl(a + b), fl(a - b)); the
 * final * 1/4 is exact.  The transform is orthogonal, so transforming both
 * GEMM operands along K with the same signs leaves X W^T unchanged:
 * quantize rht16(X) and rht16(W) and multiply as usual.  out: device fp32
 * [rows][K], 16-byte aligned.  NVFP4_EINVAL for signs above 0xFFFF. */
nvfp4_status nvfp4_rht16(const void* x, nvfp4_in_dtype dt, int64_t rows, int64_t K, uint32_t signs, float* out,
                         void* stream);

/* The activation side of a W4A4 layer in one call pair: optionally the
 * transform above (use_rht = 1, with `signs`), then the 1-D Four-Over-Six
 * quantizer, with the block scales written straight into the tensor-core
 * layout.  Bit for bit the same as nvfp4_rht16 (if used), then
 * nvfp4_kv_smooth_quant (H = 1, D = K, no smoothing) on the fp32 result (on x
 * itself without the transform), then nvfp4_scales_to_mma; the transformed
 * values never leave registers.
 *   x           device [M][K] bf16, 32-byte aligned, M >= 1, K % 16 == 0
 *   codes       device [M][K/2]
 *   scales_mma  device, nvfp4_mma_scales_bytes(M, K) bytes, padding written
 *   tensor_scale, dev_status  as nvfp4_kv_smooth_quant
 *   workspace   device, nvfp4_act_quant_workspace_bytes(), 256-byte aligned,
 *               no zero-fill needed (one amax partial per CTA) */
size_t nvfp4_act_quant_workspace_bytes(void);
nvfp4_status nvfp4_act_quant_mma(const void* x, int64_t M, int64_t K, int use_rht, uint32_t signs, uint8_t* codes,
                                 uint8_t* scales_mma, float* tensor_scale, int* dev_status, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Device workspace of nvfp4_gemm_w4a4 (256-byte aligned).  Its first int32 is
 * an error flag: the kernel sets it to 1 when one of its bounded waits (about
 * two seconds each) gave up, in which case Y is incomplete.  The kernel never
 * clears it: zero the workspace once, before the first call, to read it. */
size_t nvfp4_gemm_workspace_bytes(void);

/* A GEMM plan for one shape: the shape, the SM count (the kernel is
 * persistent, one CTA per SM) and the driver's tensor-map encoder.  It is the
 * one object the library allocates, in host memory; the caller owns it and
 * frees it with nvfp4_gemm_plan_destroy.  A plan serves one host thread at a
 * time.  M >= 1, N a multiple of 16, K a multiple of 32, M * N <= 2^46
 * (NVFP4_ESHAPE otherwise); NVFP4_ECUDA when the device or the driver's
 * encoder is unavailable. */
typedef struct nvfp4_gemm_plan nvfp4_gemm_plan;
nvfp4_status nvfp4_gemm_plan_create(int64_t M, int64_t N, int64_t K, nvfp4_gemm_plan** plan);
void nvfp4_gemm_plan_destroy(nvfp4_gemm_plan* plan);

/* Y = X W^T as above, enqueued on `stream`.
 *   x_codes, w_codes          device, 16-byte aligned
 *   x_scales_mma, w_scales_mma device, the tensor-core layout, 16-byte aligned
 *   x_tensor_scale, w_tensor_scale  device fp32 [1] (gX, gW)
 *   y_bf16                    device [M][N] bf16, 16-byte aligned
 *   workspace                 device, nvfp4_gemm_workspace_bytes(), the error flag above
 * The codes are read through TMA tensor maps encoded on the host at each call
 * (boxes of 128 bytes of K by 128 or 256 rows); NVFP4_ECUDA if encoding or the
 * launch fails. */
nvfp4_status nvfp4_gemm_w4a4(nvfp4_gemm_plan* plan, const uint8_t* x_codes, const uint8_t* x_scales_mma,
                             const float* x_tensor_scale, const uint8_t* w_codes, const uint8_t* w_scales_mma,
                             const float* w_tensor_scale, void* y_bf16, void* workspace, size_t workspace_bytes,
                             void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GB300_H */
