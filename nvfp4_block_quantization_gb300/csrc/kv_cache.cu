// kv_cache.cu -- the multi-shot NVFP4 KV cache (sm_103a): host-side frame
// bookkeeping over a caller-owned pool of chunk slots, and the gathered cache
// read that expands one attention view to bf16.
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page):
//   - inference step 7: the NVFP4 KV cache is written one chunk of F_c latent
//     frames at a time (K smoothed, then 4/6 adaptive block scales), so a chunk
//     slot holds one chunk's codes, scales, tensor scale and mean;
//   - inference step 9: attention reads a Global Sink (the first S_g frames of
//     the video) plus a Shot-Level Sink (the first S_s frames of the current
//     shot, kept as START/LEN pointers into frames already cached: no memory of
//     its own); a prompt switch rebinds the shot sink.
// The local part of the attention is read as a rolling window of the W frames
// right before the chunk being generated; a chunk slot is released once none of
// its frames can be in the next chunk's view or a later one (windows only move
// forward and a new shot sink only covers frames not yet written).
//
// The gathered read is the dequant of the plain cache read with one level of
// indirection: output row t belongs to view frame t / L_f, whose rows sit at
// pool row frame_row[t / L_f] and whose tensor scale and mean are those of its
// slot.  The frame table travels as a kernel parameter (validated on the host),
// so no device table is needed and no index is ever out of the pool.
#include <algorithm>
#include <cstring>

#include "nvfp4.h"
#include "common.cuh"

namespace nvfp4 {
namespace {

// ---------------------------------------------------------------- host bookkeeping

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// True when frame f can be in the view of a chunk whose first frame is >= cur.
bool frame_live(const nvfp4_kvcache& c, int64_t f, int64_t cur) {
  if (f < c.global_sink) return true;
  if (f >= c.shot_start && f < c.shot_start + c.shot_sink) return true;
  return f >= cur - c.window;
}

bool config_ok(const nvfp4_kvcache& c) {
  return c.frames_per_chunk >= 1 && c.tokens_per_frame >= 1 && c.global_sink >= 0 && c.shot_sink >= 0 &&
         c.window >= 0 && c.n_slots >= 1 && c.n_slots <= NVFP4_KVCACHE_MAX_SLOTS && c.n_chunks >= 0 &&
         c.shot_start >= 0 && c.shot_start <= c.n_chunks * c.frames_per_chunk;
}

// ---------------------------------------------------------------- gathered read

struct ViewTable {
  int64_t row[NVFP4_MAX_VIEW_FRAMES];  // first pool row of each view frame
  int meta[NVFP4_MAX_VIEW_FRAMES];     // its slot: tensor scale g[meta], mean [meta][C]
};

constexpr int kAhead = 4;

__device__ __forceinline__ void st_v8_cs(void* p, const uint32_t w[8]) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Launch: grid (gx, gy), CTAs of cw * rpp threads.  Thread (c, r) owns block
// column blockIdx.x * cw + c (16 channels) of the contiguous output row range
// [blockIdx.y * R, (blockIdx.y + 1) * R), rows r, r + rpp, ...  Its frame's pool
// offset, tensor scale and 16 means stay in registers and change only when a row
// crosses into the next view frame.  Codes and scale bytes of kAhead rows are
// loaded before any of them is expanded; each block's 16 bf16 values leave in one
// 32-byte streaming store when the output is 32-byte aligned.
template <bool kMean, bool kWide>
__global__ void __launch_bounds__(256) kv_gather_dequant_kernel(const uint8_t* __restrict__ codes,
                                                                const uint8_t* __restrict__ scales,
                                                                const float* __restrict__ g_pool,
                                                                const float* __restrict__ mean_pool, int64_t L,
                                                                int64_t T, int C, int cw, int rpp,
                                                                int64_t rows_per_cta, __nv_bfloat16* __restrict__ out,
                                                                const __grid_constant__ ViewTable tab) {
  const int nbr = C / 16;
  const int c = threadIdx.x % cw, rl = threadIdx.x / cw;
  const int cb = blockIdx.x * cw + c;
  if (cb >= nbr || rl >= rpp) return;
  const int64_t ra = (int64_t)blockIdx.y * rows_per_cta;
  const int64_t rb = ra + rows_per_cta < T ? ra + rows_per_cta : T;
  const uint2* c8 = reinterpret_cast<const uint2*>(codes) + cb;
  const uint8_t* s8 = scales + cb;
  uint4* o = reinterpret_cast<uint4*>(out + (size_t)cb * 16);
  const size_t orow = (size_t)C / 8;  // uint4 per output row
  int64_t fend = -1, delta = 0;       // first output row of the next frame; pool row - output row
  int fmeta = 0;                      // slot of the current frame
  int gmeta = -1;                     // slot whose tensor scale and means are in registers
  float g = 0.0f, mu[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) mu[i] = 0.0f;
  for (int64_t r = ra + rl; r < rb; r += (int64_t)kAhead * rpp) {
    uint2 cwd[kAhead];
    uint32_t sc[kAhead];
    int meta[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int64_t row = r + (int64_t)u * rpp;
      meta[u] = fmeta;
      if (row < rb) {
        if (row >= fend) {  // entering the next view frame
          const int64_t f = row / L;
          fend = (f + 1) * L;
          delta = tab.row[f] - f * L;
          fmeta = tab.meta[f];
          meta[u] = fmeta;
        }
        const int64_t src = row + delta;
        cwd[u] = __ldg(c8 + (size_t)src * nbr);
        sc[u] = __ldg(s8 + (size_t)src * nbr);
      }
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int64_t row = r + (int64_t)u * rpp;
      if (row >= rb) break;
      if (meta[u] != gmeta) {  // a frame of another chunk: its tensor scale and means
        gmeta = meta[u];
        g = __ldg(g_pool + gmeta);
        if (kMean) {
          const float* m = mean_pool + (size_t)gmeta * C + (size_t)cb * 16;
          if ((reinterpret_cast<uintptr_t>(m) & 15) == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 v = __ldg(reinterpret_cast<const float4*>(m) + i);
              mu[4 * i] = v.x; mu[4 * i + 1] = v.y; mu[4 * i + 2] = v.z; mu[4 * i + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) mu[i] = __ldg(m + i);
          }
        }
      }
      const float S = __fmul_rn(e4m3_value(sc[u]), g);
      uint32_t w[8];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const uint32_t byte = ((p < 4 ? cwd[u].x : cwd[u].y) >> (8 * (p & 3))) & 0xFFu;
        const uint32_t q = e2m1x2_to_f16x2(byte);
        float v0 = __fmul_rn(f16lo(q), S);
        float v1 = __fmul_rn(f16hi(q), S);
        if (kMean) {
          v0 = __fadd_rn(v0, mu[2 * p]);
          v1 = __fadd_rn(v1, mu[2 * p + 1]);
        }
        __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
        w[p] = *reinterpret_cast<uint32_t*>(&h);
      }
      uint4* dst = o + (size_t)row * orow;
      if (kWide) {
        st_v8_cs(dst, w);
      } else {
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
  }
}

cudaError_t launch_gather(const uint8_t* codes, const uint8_t* scales, const float* g_pool, const float* mean_pool,
                          int64_t L, int64_t T, int C, const ViewTable& tab, void* out, int sms, cudaStream_t s) {
  const int nbr = C / 16;
  const int cw = nbr < 256 ? nbr : 256;
  const int rpp = 256 / cw;
  const int gx = (nbr + cw - 1) / cw;
  // the plain cache read's grid: 16 CTAs per SM with the means re-added, 32 without
  const int per_sm = mean_pool ? 16 : 32;
  int64_t gy = ((int64_t)per_sm * (sms > 0 ? sms : 1) + gx - 1) / gx;
  const int64_t max_gy = (T + rpp - 1) / rpp;
  if (gy > max_gy) gy = max_gy;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  const int64_t rows_per_cta = (T + gy - 1) / gy;
  gy = (T + rows_per_cta - 1) / rows_per_cta;
  const dim3 grid(gx, (unsigned)gy);
  const dim3 block(cw * rpp);
  auto* o = static_cast<__nv_bfloat16*>(out);
  const bool wide = (reinterpret_cast<uintptr_t>(out) % 32) == 0;
  if (mean_pool && wide)
    kv_gather_dequant_kernel<true, true><<<grid, block, 0, s>>>(codes, scales, g_pool, mean_pool, L, T, C, cw, rpp,
                                                                rows_per_cta, o, tab);
  else if (mean_pool)
    kv_gather_dequant_kernel<true, false><<<grid, block, 0, s>>>(codes, scales, g_pool, mean_pool, L, T, C, cw, rpp,
                                                                 rows_per_cta, o, tab);
  else if (wide)
    kv_gather_dequant_kernel<false, true><<<grid, block, 0, s>>>(codes, scales, g_pool, mean_pool, L, T, C, cw, rpp,
                                                                 rows_per_cta, o, tab);
  else
    kv_gather_dequant_kernel<false, false><<<grid, block, 0, s>>>(codes, scales, g_pool, mean_pool, L, T, C, cw,
                                                                  rpp, rows_per_cta, o, tab);
  return cudaGetLastError();
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace nvfp4

using nvfp4::ceil_div;

extern "C" {

int nvfp4_kvcache_slots_needed(int frames_per_chunk, int global_sink, int shot_sink, int window) {
  if (frames_per_chunk < 1 || global_sink < 0 || shot_sink < 0 || window < 0) return -1;
  // chunks that can hold live frames while one more is written: the global sink's,
  // the current shot sink's (its START is a chunk's first frame), and those that a
  // window of W frames ending at a chunk boundary overlaps (at least the new chunk)
  const int64_t n = ceil_div(global_sink, frames_per_chunk) + ceil_div(shot_sink, frames_per_chunk) +
                    std::max<int64_t>(1, ceil_div(window, frames_per_chunk));
  return n > NVFP4_KVCACHE_MAX_SLOTS ? -1 : (int)n;
}

nvfp4_status nvfp4_kvcache_init(nvfp4_kvcache* c, int frames_per_chunk, int64_t tokens_per_frame, int global_sink,
                                int shot_sink, int window, int n_slots) {
  if (!c) return NVFP4_EINVAL;
  nvfp4_kvcache t;
  std::memset(&t, 0, sizeof(t));
  t.frames_per_chunk = frames_per_chunk;
  t.tokens_per_frame = tokens_per_frame;
  t.global_sink = global_sink;
  t.shot_sink = shot_sink;
  t.window = window;
  t.n_slots = n_slots;
  t.n_chunks = 0;
  t.shot_start = 0;
  for (int i = 0; i < NVFP4_KVCACHE_MAX_SLOTS; ++i) t.slot_chunk[i] = -1;
  if (!nvfp4::config_ok(t)) return NVFP4_ESHAPE;
  *c = t;
  return NVFP4_OK;
}

nvfp4_status nvfp4_kvcache_append(nvfp4_kvcache* c, int* slot) {
  if (!c || !slot) return NVFP4_EINVAL;
  if (!nvfp4::config_ok(*c)) return NVFP4_ESHAPE;
  const int64_t F = c->frames_per_chunk;
  const int64_t next = (c->n_chunks + 1) * F;  // first frame of the chunk after this one
  // release the chunks none of whose frames the next view (or a later one) can hold
  for (int s = 0; s < c->n_slots; ++s) {
    const int64_t k = c->slot_chunk[s];
    if (k < 0) continue;
    bool live = false;
    for (int64_t f = k * F; f < (k + 1) * F && !live; ++f) live = nvfp4::frame_live(*c, f, next);
    if (!live) c->slot_chunk[s] = -1;
  }
  for (int s = 0; s < c->n_slots; ++s) {
    if (c->slot_chunk[s] < 0) {
      c->slot_chunk[s] = c->n_chunks++;
      *slot = s;
      return NVFP4_OK;
    }
  }
  return NVFP4_ECAPACITY;
}

nvfp4_status nvfp4_kvcache_new_shot(nvfp4_kvcache* c) {
  if (!c) return NVFP4_EINVAL;
  if (!nvfp4::config_ok(*c)) return NVFP4_ESHAPE;
  c->shot_start = c->n_chunks * c->frames_per_chunk;
  return NVFP4_OK;
}

int nvfp4_kvcache_view(const nvfp4_kvcache* c, int64_t* frame_index, int64_t* frame_row, int* frame_slot,
                       int max_frames) {
  if (!c || !nvfp4::config_ok(*c) || max_frames < 0) return -1;
  const int64_t F = c->frames_per_chunk;
  const int64_t cur = c->n_chunks * F;
  // the three ranges, clipped to the cached frames [0, cur), merged in ascending order
  int64_t lo[3] = {0, c->shot_start, cur - c->window};
  int64_t hi[3] = {(int64_t)c->global_sink, c->shot_start + c->shot_sink, cur};
  for (int i = 0; i < 3; ++i) {
    lo[i] = std::max<int64_t>(lo[i], 0);
    hi[i] = std::min<int64_t>(hi[i], cur);
  }
  for (int i = 0; i < 3; ++i)  // sort the ranges by start (three elements)
    for (int j = i + 1; j < 3; ++j)
      if (lo[j] < lo[i]) {
        std::swap(lo[i], lo[j]);
        std::swap(hi[i], hi[j]);
      }
  // count first, then write: nothing is written when max_frames is too small
  for (int pass = 0; pass < 2; ++pass) {
    int64_t n = 0, next = 0;  // next: first frame not yet emitted
    for (int i = 0; i < 3; ++i) {
      for (int64_t f = std::max(lo[i], next); f < hi[i]; ++f, ++n) {
        if (pass == 1) {
          const int64_t k = f / F;
          int s = -1;
          for (int t = 0; t < c->n_slots; ++t)
            if (c->slot_chunk[t] == k) s = t;
          if (s < 0) return -1;  // not resident: the struct was modified by hand
          if (frame_index) frame_index[n] = f;
          if (frame_row) frame_row[n] = ((int64_t)s * F + (f - k * F)) * c->tokens_per_frame;
          if (frame_slot) frame_slot[n] = s;
        }
      }
      next = std::max(next, hi[i]);
    }
    if (pass == 0 && n > max_frames) return -1;
    if (pass == 1) return (int)n;
  }
  return -1;
}

nvfp4_status nvfp4_kv_gather_dequant(const uint8_t* codes_pool, const uint8_t* scales_pool, const float* g_pool,
                                     const float* mean_pool, int64_t pool_rows, int n_meta, const int64_t* frame_row,
                                     const int* frame_meta, int n_frames, int64_t tokens_per_frame, int H, int D,
                                     void* out_bf16, void* stream) {
  if (H < 1 || D < 16 || (D % 16) != 0 || (int64_t)H * D > (1 << 24)) return NVFP4_ESHAPE;
  if (n_frames < 0 || n_frames > NVFP4_MAX_VIEW_FRAMES || tokens_per_frame < 1 || pool_rows < 0) return NVFP4_ESHAPE;
  if (n_frames == 0) return NVFP4_OK;
  const int64_t C = (int64_t)H * D;
  if (pool_rows > 0 && C > ((int64_t)1 << 46) / pool_rows) return NVFP4_ESHAPE;
  if (tokens_per_frame > ((int64_t)1 << 46) / NVFP4_MAX_VIEW_FRAMES) return NVFP4_ESHAPE;
  if (!codes_pool || !scales_pool || !g_pool || !frame_row || !frame_meta || !out_bf16) return NVFP4_EINVAL;
  if (n_meta < 1) return NVFP4_ESHAPE;
  if (!nvfp4::aligned_to(codes_pool, 16) || !nvfp4::aligned_to(scales_pool, 16) ||
      !nvfp4::aligned_to(out_bf16, 16))
    return NVFP4_EALIGN;
  if (!nvfp4::aligned_to(g_pool, 4) || !nvfp4::aligned_to(mean_pool, 4)) return NVFP4_EALIGN;
  nvfp4::ViewTable tab;
  std::memset(&tab, 0, sizeof(tab));
  for (int i = 0; i < n_frames; ++i) {  // every frame inside the pool, every slot inside the metadata
    if (frame_row[i] < 0 || frame_row[i] > pool_rows - tokens_per_frame) return NVFP4_ESHAPE;
    if (frame_meta[i] < 0 || frame_meta[i] >= n_meta) return NVFP4_ESHAPE;
    tab.row[i] = frame_row[i];
    tab.meta[i] = frame_meta[i];
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ECUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return NVFP4_ECUDA;
  const cudaError_t e = nvfp4::launch_gather(codes_pool, scales_pool, g_pool, mean_pool, tokens_per_frame,
                                             (int64_t)n_frames * tokens_per_frame, (int)C, tab, out_bf16, sms,
                                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

}  // extern "C"
