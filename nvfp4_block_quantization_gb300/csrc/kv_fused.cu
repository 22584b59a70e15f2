// kv_fused.cu -- one persistent, cooperative kernel that K-smooths and
// Four-Over-Six-quantizes a batch of same-shape KV chunk tensors (sm_103a).
//
// Method: "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video
// Generation" (summary page), inference step 7 (per-chunk K-smoothing, then
// 4/6 adaptive block scales into the NVFP4 KV cache) and the "full-stack NVFP4"
// paragraph (keep the lower-MSE of two FP8 block-scale candidates).
//
// Work split.  Each tensor [T][C] (C = H*D) is cut into channel groups of W
// channels (W = 128 when C allows); the ngroups*T (group, row) units are dealt
// out in contiguous ranges to the P resident CTAs, so a CTA holds a few long
// row segments of one or two groups.  A segment is read in tiles of 64 rows x W
// channels by 2-D TMA (cp.async.bulk.tensor) into shared-memory stages that
// complete on mbarriers.
//
// Roles inside every CTA (warp-specialized, no block-wide barrier between them):
//   stats warps  stream job j: per-channel TwoSum-compensated sums, min and max
//                (smoothed tensors) or the absolute maximum (unsmoothed).  The
//                last CTA to finish a channel group combines the group's
//                partials in binary64, rounds the mean once to fp32 and folds
//                the group's max |x - mean| into the job amax.
//   quant warps  wait (bounded) until job j's amax is complete, build the
//                per-tensor reciprocal table, then quantize their tiles of job
//                j (re-read through L2 by their own TMA pipeline, which starts
//                prefetching before the wait): two 16-element blocks per
//                thread, both candidates, fused error chains in packed f32x2,
//                choice, packed stores.
// Stats of job j+1 overlap the quantization of job j; the stats warps stay at
// most two jobs ahead of their own CTA's quant warps so the re-read hits L2.
//
// Every wait (mbarrier, cross-CTA counter, intra-CTA progress) is bounded;
// the cross-CTA counters live in the caller's zero-filled workspace and the
// last CTA to exit zeroes them again.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kv_kernels.cuh"

namespace nvfp4 {

namespace {

constexpr int kST = kFusedStatsWarps * 32;  // stats threads
constexpr int kQT = kFusedQuantWarps * 32;  // quant threads
constexpr int kBarStats = 1, kBarQuant = 2;
constexpr int kTileRows = 64;
constexpr unsigned kStatusNonfinite = 1u, kStatusTimeout = 2u;

template <bool kBF16>
struct Cfg {
  static constexpr int kEsize = kBF16 ? 2 : 4;
  static constexpr int kStagesS = kBF16 ? 8 : 3;  // stats stream (HBM): deep, covers ~2 us round trips
  static constexpr int kStagesQ = kBF16 ? 4 : 2;  // quant stream (L2 re-read)
  static constexpr int kStageBytes = kTileRows * kFusedMaxW * kEsize;
  static constexpr int kDynSmem = (kStagesS + kStagesQ) * kStageBytes;
};

struct StatsSmem {
  float wred[kFusedStatsWarps][4][kFusedMaxW];  // per-warp partials: sum, low part, min, max
  float red[32];
  int last;
};

struct QuantSmem {
  float2 tab[128];  // {fl(1 / fl(E * g)) or 0 when unusable, E * E} per E4M3 code
  unsigned amax_bits;
  int abort;
};

struct Smem {
  uint64_t full_s[8];   // stats stages: data landed (TMA transaction count)
  uint64_t empty_s[8];  // stats stages: every stats warp finished reading
  uint64_t full_q[4];   // quant stages: data landed
  uint64_t empty_q[4];  // quant stages: every quant warp finished reading
  StatsSmem st;
  QuantSmem qu;
  volatile int quant_done;  // jobs this CTA's quant warps have finished
  unsigned status;
  int exit_last;
};

// ------------------------------------------------------------------ partition
__device__ __forceinline__ int64_t range_start(const FusedGeom& G, int c) { return (int64_t)c * G.U / G.P; }
__device__ __forceinline__ int owner_of(const FusedGeom& G, int64_t u) { return (int)(((u + 1) * G.P - 1) / G.U); }
__device__ __forceinline__ unsigned group_arrivals(const FusedGeom& G, int k) {
  if (G.U < G.P) return (unsigned)G.T;  // every non-empty CTA owns exactly one unit
  return (unsigned)(owner_of(G, (int64_t)k * G.T + G.T - 1) - owner_of(G, (int64_t)k * G.T) + 1);
}

// Segments of [u0, u1): group k, rows [r0, r1).
struct Seg {
  int k;
  int64_t r0, r1;
};
__device__ __forceinline__ Seg seg_at(const FusedGeom& G, int64_t u, int64_t u1) {
  Seg s;
  s.k = (int)(u / G.T);
  s.r0 = u - (int64_t)s.k * G.T;
  s.r1 = min(G.T, s.r0 + (u1 - u));
  return s;
}
__device__ __forceinline__ int tiles_in(const Seg& s) { return (int)((s.r1 - s.r0 + kTileRows - 1) / kTileRows); }

__device__ int tiles_per_job(const FusedGeom& G, int64_t u0, int64_t u1) {
  int n = 0;
  for (int64_t u = u0; u < u1;) {
    const Seg s = seg_at(G, u, u1);
    n += tiles_in(s);
    u += s.r1 - s.r0;
  }
  return n;
}

// Issue-side cursor over a role's tile stream: jobs in order, each job's segments
// in order, 64-row tiles within a segment.  Advancing is O(1) except at segment
// boundaries (one 64-bit division).
struct TileCursor {
  int j;        // job of the next tile
  int64_t u;    // first unit of the current segment
  int k;        // channel group of the current segment
  int64_t row;  // next tile's first row
  int64_t r1;   // end row of the current segment
};

__device__ __forceinline__ void cursor_seek(TileCursor& c, const FusedGeom& G, int64_t u1) {
  const Seg s = seg_at(G, c.u, u1);
  c.k = s.k;
  c.row = s.r0;
  c.r1 = s.r1;
}

__device__ __forceinline__ void cursor_init(TileCursor& c, const FusedGeom& G, int64_t u0, int64_t u1) {
  c.j = 0;
  c.u = u0;
  if (u0 < u1) cursor_seek(c, G, u1);
}

__device__ __forceinline__ void cursor_next(TileCursor& c, const FusedGeom& G, int64_t u0, int64_t u1) {
  c.row += kTileRows;
  if (c.row < c.r1) return;
  c.u = (int64_t)c.k * G.T + c.r1;  // first unit after this segment
  if (c.u >= u1) {
    ++c.j;
    c.u = u0;
  }
  cursor_seek(c, G, u1);
}

// ------------------------------------------------------------------ sync primitives
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitNs = 2000000000ull;  // every wait gives up after about 2 s

__device__ __forceinline__ bool wait_geq(const unsigned* p, unsigned target, unsigned spin_limit) {
  const uint64_t t0 = global_timer_ns();
  for (unsigned it = 0; ld_acquire_u32(p) < target; ++it) {
    if (it >= spin_limit || global_timer_ns() - t0 > kWaitNs) return false;
    __nanosleep(it < 64 ? 32 : 256);
  }
  return true;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait for phase `parity` of an mbarrier; false after about 2 s.  try_wait
// itself suspends the thread in hardware until the phase completes (or a short
// system time limit passes), so the loop only re-polls; the clock is read every
// 1024 polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, unsigned spin_limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (unsigned it = 1; !mbar_try_wait(bar, parity); ++it) {
    if ((it & 1023u) == 0 && (it >= spin_limit || global_timer_ns() - t0 > kWaitNs)) return false;
  }
  return true;
}

// One 2-D TMA tile (box W x 64 rows of the tensor map) into `dst`, completing on `bar`.
__device__ __forceinline__ void tma_tile(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                         unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Issue the cursor's tile into stage `st` and advance the cursor.
__device__ __forceinline__ void issue_next(const FusedBatch& b, const FusedGeom& G, int64_t u0, int64_t u1,
                                           TileCursor& c, uint8_t* stages, int st, unsigned stage_bytes,
                                           unsigned box_bytes, uint64_t* bars) {
  tma_tile(stages + (size_t)st * stage_bytes, &b.map[c.j], c.k * G.W, (int)c.row, &bars[st], box_bytes);
  cursor_next(c, G, u0, u1);
}

// ------------------------------------------------------------------ stats role
// (s, n) pairs carry sum = s + n (n: the low part lost by s).
__device__ __forceinline__ void comp_add(float& s, float& n, float s2, float n2) {
  float t, e;
  two_sum(s, s2, t, e);
  s = t;
  n = __fadd_rn(n, __fadd_rn(n2, e));
}

__device__ __forceinline__ float warp_max_nan(float v) {
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Max over the stats threads; result valid in every stats thread.
__device__ __forceinline__ float stats_max(float v, StatsSmem& sm) {
  v = warp_max_nan(v);
  const int s = threadIdx.x;
  if ((s & 31) == 0) sm.red[s >> 5] = v;
  named_barrier(kBarStats, kST);
  float r = 0.0f;
#pragma unroll
  for (int w = 0; w < kFusedStatsWarps; ++w) r = max_nan(r, sm.red[w]);
  named_barrier(kBarStats, kST);
  return r;
}

// The last CTA to finish group k of job J: binary64 combine of the partials,
// mean, channel amax; publishes mean[] and the group's amax.
__device__ void group_reduce(const FusedJob& J, const FusedGeom& G, int k, StatsSmem& sm) {
  const int s = threadIdx.x;
  float cam = 0.0f;
  if (s < G.W) {
    const int ch = k * G.W + s;
    const int cf = owner_of(G, (int64_t)k * G.T), cl = owner_of(G, (int64_t)k * G.T + G.T - 1);
    double S = 0.0;
    float mn = __int_as_float(0x7f800000), mx = -mn;
    for (int c = cf; c <= cl; ++c) {
      const int64_t a = range_start(G, c), e = range_start(G, c + 1);
      if (a == e) continue;  // empty CTA (only when units < CTAs)
      const int seg = k - (int)(a / G.T);
      const float4 p = __ldcg(J.part + ((int64_t)c * G.smax + seg) * G.W + s);
      S += (double)p.x;
      S += (double)p.y;
      mn = min_nan(mn, p.z);
      mx = max_nan(mx, p.w);
    }
    const float mu = J.mean_in ? J.mean_in[ch] : (float)(S / (double)G.T);
    J.mean[ch] = mu;
    if (J.mean_out) J.mean_out[ch] = mu;
    cam = max_nan(__fsub_rn(mx, mu), __fsub_rn(mu, mn));
  }
  __threadfence();
  const float gmax = stats_max(cam, sm);
  if (s == 0) {
    atomicMax(J.ctr + 0, __float_as_uint(gmax) & 0x7fffffffu);
    __threadfence();
    atomicAdd(J.ctr + 1, 1u);
  }
}

// Accumulate one tile (rows [row0, row0+64) of the segment, clipped to r1) into the
// thread's channel statistics.
template <bool kBF16>
__device__ __forceinline__ void stats_tile(const uint8_t* tile, int W, int64_t row0, int64_t r1, int ro, int rpp,
                                           int ls, bool smooth, float2 sum[4], float2 low[4], uint32_t mnw[4],
                                           uint32_t mxw[4], float mn[8], float mx[8], float& vmax,
                                           uint32_t vmaxw[4]) {
  const float2 m1 = make_float2(-1.0f, -1.0f);
  const int nrows = (int)min((int64_t)kTileRows, r1 - row0);
  for (int tr = ro; tr < nrows; tr += rpp) {
    float v[8];
    const uint8_t* p = tile + ((size_t)tr * W + 8 * ls) * Cfg<kBF16>::kEsize;
    if (kBF16) {
      const uint4 w = *reinterpret_cast<const uint4*>(p);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
      if (!smooth) {
#pragma unroll
        for (int m = 0; m < 4; ++m) vmaxw[m] = bf16x2_max_nan(vmaxw[m], ww[m] & 0x7fff7fffu);
        continue;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        v[2 * m] = bf16lo(ww[m]);
        v[2 * m + 1] = bf16hi(ww[m]);
        mnw[m] = bf16x2_min_nan(mnw[m], ww[m]);
        mxw[m] = bf16x2_max_nan(mxw[m], ww[m]);
      }
    } else {
      const uint4 a = *reinterpret_cast<const uint4*>(p);
      const uint4 c = *reinterpret_cast<const uint4*>(p + 16);
      v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
      v[4] = __uint_as_float(c.x); v[5] = __uint_as_float(c.y); v[6] = __uint_as_float(c.z); v[7] = __uint_as_float(c.w);
      if (!smooth) {
#pragma unroll
        for (int i = 0; i < 8; ++i) vmax = max_nan(vmax, fabsf(v[i]));
        continue;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) { mn[i] = min_nan(mn[i], v[i]); mx[i] = max_nan(mx[i], v[i]); }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      // TwoSum on the channel pair (2m, 2m+1): t + e == sum + x exactly; e accumulates into low
      const float2 x2 = make_float2(v[2 * m], v[2 * m + 1]);
      const float2 t = __fadd2_rn(sum[m], x2);
      const float2 bp = __ffma2_rn(sum[m], m1, t);   // t - sum
      const float2 ap = __ffma2_rn(bp, m1, t);       // t - bp
      const float2 da = __ffma2_rn(ap, m1, sum[m]);  // sum - ap
      const float2 db = __ffma2_rn(bp, m1, x2);      // x - bp
      low[m] = __fadd2_rn(low[m], __fadd2_rn(da, db));
      sum[m] = t;
    }
  }
}

template <bool kBF16>
__device__ void stats_role(const FusedBatch& b, const FusedGeom& G, int64_t u0, int64_t u1, Smem& sm,
                           uint8_t* stages) {
  using CF = Cfg<kBF16>;
  const int s = threadIdx.x;
  const int tpr = G.W / 8;  // threads per row (8 channels each)
  const int rpp = kST / tpr;  // rows per pass
  const int ls = s % tpr, ro = s / tpr;
  const int warp = s >> 5, lane = s & 31;
  int f = 0;
  for (int j = 0; j < b.n; ++j) {
    const FusedJob& J = b.job[j];
    float vmax = 0.0f;
    uint32_t vmaxw[4] = {0u, 0u, 0u, 0u};
    for (int64_t u = u0; u < u1;) {
      const Seg sg = seg_at(G, u, u1);
      float2 sum[4], low[4];
      float mn[8], mx[8];
      uint32_t mnw[4], mxw[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        sum[m] = make_float2(0.f, 0.f);
        low[m] = make_float2(0.f, 0.f);
        mnw[m] = 0x7f807f80u;  // (+inf, +inf)
        mxw[m] = 0xff80ff80u;  // (-inf, -inf)
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) { mn[i] = __int_as_float(0x7f800000); mx[i] = -mn[i]; }
      for (int64_t row0 = sg.r0; row0 < sg.r1; row0 += kTileRows, ++f) {
        const int st = f % CF::kStagesS;
        if (!mbar_wait(&sm.full_s[st], (unsigned)(f / CF::kStagesS) & 1u, G.spin_limit) && s == 0)
          atomicOr(&sm.status, kStatusTimeout);
        stats_tile<kBF16>(stages + (size_t)st * CF::kStageBytes, G.W, row0, sg.r1, ro, rpp, ls, J.smooth != 0, sum,
                          low, mnw, mxw, mn, mx, vmax, vmaxw);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty_s[st]);
      }
      if (J.smooth) {
        if (kBF16) {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            mn[2 * m] = bf16lo(mnw[m]); mn[2 * m + 1] = bf16hi(mnw[m]);
            mx[2 * m] = bf16lo(mxw[m]); mx[2 * m + 1] = bf16hi(mxw[m]);
          }
        }
        float S[8], L[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) { S[2 * m] = sum[m].x; S[2 * m + 1] = sum[m].y; L[2 * m] = low[m].x; L[2 * m + 1] = low[m].y; }
        // combine the lanes of a warp that share channels (lanes ls, ls + tpr, ...)
        for (int o = tpr; o < 32; o <<= 1) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float s2 = __shfl_xor_sync(0xffffffffu, S[i], o), l2 = __shfl_xor_sync(0xffffffffu, L[i], o);
            const float a2 = __shfl_xor_sync(0xffffffffu, mn[i], o), b2 = __shfl_xor_sync(0xffffffffu, mx[i], o);
            comp_add(S[i], L[i], s2, l2);
            mn[i] = min_nan(mn[i], a2);
            mx[i] = max_nan(mx[i], b2);
          }
        }
        if (lane < tpr) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            sm.st.wred[warp][0][8 * ls + i] = S[i];
            sm.st.wred[warp][1][8 * ls + i] = L[i];
            sm.st.wred[warp][2][8 * ls + i] = mn[i];
            sm.st.wred[warp][3][8 * ls + i] = mx[i];
          }
        }
        named_barrier(kBarStats, kST);
        if (s < G.W) {
          float Sc = sm.st.wred[0][0][s], Lc = sm.st.wred[0][1][s], mnc = sm.st.wred[0][2][s], mxc = sm.st.wred[0][3][s];
          for (int w = 1; w < kFusedStatsWarps; ++w) {
            comp_add(Sc, Lc, sm.st.wred[w][0][s], sm.st.wred[w][1][s]);
            mnc = min_nan(mnc, sm.st.wred[w][2][s]);
            mxc = max_nan(mxc, sm.st.wred[w][3][s]);
          }
          const int seg = sg.k - (int)(u0 / G.T);
          J.part[((int64_t)blockIdx.x * G.smax + seg) * G.W + s] = make_float4(Sc, Lc, mnc, mxc);
          __threadfence();
        }
        named_barrier(kBarStats, kST);
        if (s == 0) sm.st.last = (atomicAdd(J.ctr + 2 + sg.k, 1u) + 1u == group_arrivals(G, sg.k));
        named_barrier(kBarStats, kST);
        if (sm.st.last) {
          __threadfence();
          group_reduce(J, G, sg.k, sm.st);
        }
      }
      u += sg.r1 - sg.r0;
    }
    if (!J.smooth) {
      if (kBF16) {
        const uint32_t w01 = bf16x2_max_nan(vmaxw[0], vmaxw[1]), w23 = bf16x2_max_nan(vmaxw[2], vmaxw[3]);
        const uint32_t w = bf16x2_max_nan(w01, w23);
        vmax = max_nan(bf16lo(w), bf16hi(w));
      }
      const float m = stats_max(vmax, sm.st);
      if (s == 0) {
        atomicMax(J.ctr + 0, __float_as_uint(m) & 0x7fffffffu);
        __threadfence();
        atomicAdd(J.ctr + 1, 1u);
      }
    }
  }
}

// ------------------------------------------------------------------ quant role
// One 16-element block from a shared-memory tile, smoothed (z = fl(x - mu)) or widened.
template <bool kBF16, bool kSmooth>
__device__ __forceinline__ void tile_block(const uint8_t* p, const float mu[16], float z[16]) {
  if (kBF16) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const uint4 c = *reinterpret_cast<const uint4*>(p + 16);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (kSmooth) bf16x2_minus(w[i], mu[2 * i], mu[2 * i + 1], z[2 * i], z[2 * i + 1]);
      else { z[2 * i] = bf16lo(w[i]); z[2 * i + 1] = bf16hi(w[i]); }
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 a = *reinterpret_cast<const float4*>(p + 16 * q);
      const float xs[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) z[4 * q + i] = kSmooth ? __fsub_rn(xs[i], mu[4 * q + i]) : xs[i];
    }
  }
}

// Four-Over-Six on one block.  The two candidates' sequential error chains run
// side by side in one packed f32x2 accumulator (lane x: scale 6, lane y: scale 4);
// each lane is exactly the element-order fused chain of its candidate.
__device__ __forceinline__ void quant_block(const float z[16], const float2* tab, float k6, float k4, bool nonfinite,
                                            uint2& code, uint32_t& sc) {
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = fmaxf(fabsf(z[2 * i]), fabsf(z[2 * i + 1]));
  const float ma = fmaxf(fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])), fmaxf(fmaxf(a[4], a[5]), fmaxf(a[6], a[7])));
  const float2 s2 = __fmul2_rn(make_float2(ma, ma), make_float2(k6, k4));
  const uint32_t e = e4m3x2(s2.x, s2.y);
  const uint32_t e6 = e & 0x7Fu, e4 = (e >> 8) & 0x7Fu;
  const float2 t6 = tab[e6], t4 = tab[e4];
  const float2 i6 = make_float2(t6.x, t6.x), i4 = make_float2(t4.x, t4.x);
  float2 acc = make_float2(0.0f, 0.0f);
  uint32_t c6[2], c4[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float y6[8], y4[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 zz = make_float2(z[8 * h + 2 * p], z[8 * h + 2 * p + 1]);
      const float2 a6 = __fmul2_rn(zz, i6), a4 = __fmul2_rn(zz, i4);
      y6[2 * p] = a6.x; y6[2 * p + 1] = a6.y;
      y4[2 * p] = a4.x; y4[2 * p + 1] = a4.y;
    }
    uint32_t q6[4], q4[4];
    c6[h] = e2m1x8(y6, q6);
    c4[h] = e2m1x8(y4, q4);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      float d60, d61, d40, d41;
      f16x2_minus(q6[p], y6[2 * p], y6[2 * p + 1], d60, d61);
      f16x2_minus(q4[p], y4[2 * p], y4[2 * p + 1], d40, d41);
      const float2 d0 = make_float2(d60, d40);
      acc = __ffma2_rn(d0, d0, acc);
      const float2 d1 = make_float2(d61, d41);
      acc = __ffma2_rn(d1, d1, acc);
    }
  }
  const float2 err = __fmul2_rn(make_float2(t6.y, t4.y), acc);
  const bool ok6 = t6.x > 0.0f, ok4 = t4.x > 0.0f;
  const bool pick4 = ok4 && (!ok6 || err.y < err.x);
  code = pick4 ? make_uint2(c4[0], c4[1]) : (ok6 ? make_uint2(c6[0], c6[1]) : make_uint2(0u, 0u));
  sc = nonfinite ? 0x7Fu : (pick4 ? e4 : (ok6 ? e6 : 0u));
}

template <bool kBF16, bool kSmooth>
__device__ __forceinline__ void quant_tile(const FusedJob& J, const FusedGeom& G, const uint8_t* tile, int ch_base,
                                           int64_t row0, int64_t r1, const float mu[16], const float2* tab, float k6,
                                           float k4, bool nonfinite) {
  const int q = threadIdx.x - kST;
  const int bpr = G.W / 16;
  const int bc = q % bpr, tr = q / bpr;
  if (tr >= kTileRows) return;
  const int64_t r = row0 + tr;
  if (r >= r1) return;
  constexpr int es = Cfg<kBF16>::kEsize;
  float z[16];
  tile_block<kBF16, kSmooth>(tile + ((size_t)tr * G.W + 16 * bc) * es, mu, z);
  uint2 code;
  uint32_t sc;
  quant_block(z, tab, k6, k4, nonfinite, code, sc);
  const int64_t e = r * G.C + ch_base + 16 * bc;
  *reinterpret_cast<uint2*>(J.codes + e / 2) = code;
  J.scales[e / 16] = (uint8_t)sc;
}

template <bool kBF16>
__device__ void quant_role(const FusedBatch& b, const FusedGeom& G, int64_t u0, int64_t u1, Smem& sm,
                           uint8_t* stages) {
  using CF = Cfg<kBF16>;
  const int q = threadIdx.x - kST;
  int f = 0;
  for (int j = 0; j < b.n; ++j) {
    const FusedJob& J = b.job[j];
    if (q == 0) {
      const unsigned expected = J.smooth ? (unsigned)G.ngroups : (unsigned)G.P;
      const bool ok = sm.qu.abort == 0 && wait_geq(J.ctr + 1, expected, G.spin_limit);
      if (!ok) {
        sm.qu.abort = 1;
        atomicOr(&sm.status, kStatusTimeout);
      }
      sm.qu.amax_bits = ok ? ld_acquire_u32(J.ctr + 0) : 0u;
    }
    named_barrier(kBarQuant, kQT);
    const bool abort = sm.qu.abort != 0;
    const float amax = __uint_as_float(sm.qu.amax_bits);
    const bool nonfinite = !finite_f(amax);
    const float g = nonfinite ? __int_as_float(0x7fc00000) : __fdiv_rn(amax, kTensorDenom);
    const float k6 = __frcp_rn(__fmul_rn(6.0f, g));
    const float k4 = __frcp_rn(__fmul_rn(4.0f, g));
    if (q < 128) {
      const float E = e4m3_value((uint32_t)q);
      const float S = __fmul_rn(E, g);
      const float inv = __frcp_rn(S);
      const bool ok = (E > 0.0f) && (S > 0.0f) && finite_f(inv);
      sm.qu.tab[q] = make_float2(ok ? inv : 0.0f, ok ? __fmul_rn(E, E) : 0.0f);
    }
    if (blockIdx.x == 0 && q == 0 && !abort) {
      *J.tensor_scale = g;
      if (nonfinite) atomicOr(&sm.status, kStatusNonfinite);
    }
    named_barrier(kBarQuant, kQT);
    for (int64_t u = u0; u < u1;) {
      const Seg sg = seg_at(G, u, u1);
      const int ch_base = sg.k * G.W;
      float mu[16];
      if (J.smooth && !abort) {
        const int bc = q % (G.W / 16);
        const float4* m4 = reinterpret_cast<const float4*>(J.mean + ch_base + 16 * bc);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = __ldcg(m4 + i);
          mu[4 * i] = v.x; mu[4 * i + 1] = v.y; mu[4 * i + 2] = v.z; mu[4 * i + 3] = v.w;
        }
      }
      for (int64_t row0 = sg.r0; row0 < sg.r1; row0 += kTileRows, ++f) {
        const int st = f % CF::kStagesQ;
        const bool full = mbar_wait(&sm.full_q[st], (unsigned)(f / CF::kStagesQ) & 1u, G.spin_limit);
        if (!full && q == 0) atomicOr(&sm.status, kStatusTimeout);
        if (full && !abort) {
          const uint8_t* tile = stages + (size_t)st * CF::kStageBytes;
          if (J.smooth) quant_tile<kBF16, true>(J, G, tile, ch_base, row0, sg.r1, mu, sm.qu.tab, k6, k4, nonfinite);
          else quant_tile<kBF16, false>(J, G, tile, ch_base, row0, sg.r1, mu, sm.qu.tab, k6, k4, nonfinite);
        }
        __syncwarp();
        if ((q & 31) == 0) mbar_arrive(&sm.empty_q[st]);
      }
      u += sg.r1 - sg.r0;
    }
    named_barrier(kBarQuant, kQT);
    if (q == 0) {
      __threadfence_block();
      sm.quant_done = j + 1;
    }
  }
}

// ------------------------------------------------------------------ producers
// One thread per ring keeps it full: a stage is refilled as soon as every
// consumer warp of its role has released it (blocking, hardware-suspended
// mbarrier wait, so the producer issues nothing while it waits).  Stats tiles
// of job j are held back until this CTA's quant warps have finished job j - 2,
// so at most two tensors are in flight per CTA and the quant re-read stays in L2.
template <bool kBF16, bool kStatsRing>
__device__ void producer(const FusedBatch& b, const FusedGeom& G, int64_t u0, int64_t u1, Smem& sm, uint8_t* stages) {
  using CF = Cfg<kBF16>;
  constexpr int NS = kStatsRing ? CF::kStagesS : CF::kStagesQ;
  uint64_t* full = kStatsRing ? sm.full_s : sm.full_q;
  uint64_t* empty = kStatsRing ? sm.empty_s : sm.empty_q;
  const int total = b.n * tiles_per_job(G, u0, u1);
  const unsigned box_bytes = (unsigned)(kTileRows * G.W * CF::kEsize);
  TileCursor c;
  cursor_init(c, G, u0, u1);
  for (int f = 0; f < total; ++f) {
    const int st = f % NS;
    if (f >= NS && !mbar_wait(&empty[st], (unsigned)(f / NS - 1) & 1u, G.spin_limit)) {
      atomicOr(&sm.status, kStatusTimeout);
      return;
    }
    if (kStatsRing && c.j >= 2 && sm.quant_done < c.j - 1) {
      const uint64_t t0 = global_timer_ns();
      while (sm.quant_done < c.j - 1) {
        if (global_timer_ns() - t0 > kWaitNs) {
          atomicOr(&sm.status, kStatusTimeout);
          return;
        }
        __nanosleep(128);
      }
    }
    issue_next(b, G, u0, u1, c, stages, st, CF::kStageBytes, box_bytes, full);
  }
}

}  // namespace

template <bool kBF16>
__global__ void __launch_bounds__(kST + kQT + 64, 1) kv_fused_kernel(const __grid_constant__ FusedBatch b,
                                                                const FusedGeom G) {
  __shared__ Smem sm;
  extern __shared__ __align__(128) uint8_t dsm[];
  using CF = Cfg<kBF16>;
  uint8_t* stages_s = dsm;
  uint8_t* stages_q = dsm + (size_t)CF::kStagesS * CF::kStageBytes;
  const int c = blockIdx.x;
  const int64_t u0 = range_start(G, c), u1 = range_start(G, c + 1);
  if (threadIdx.x == 0) {
    sm.quant_done = 0;
    sm.status = 0u;
    sm.qu.abort = 0;
    for (int i = 0; i < CF::kStagesS; ++i) {
      mbar_init(&sm.full_s[i], 1);
      mbar_init(&sm.empty_s[i], kFusedStatsWarps);
    }
    for (int i = 0; i < CF::kStagesQ; ++i) {
      mbar_init(&sm.full_q[i], 1);
      mbar_init(&sm.empty_q[i], kFusedQuantWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x < (unsigned)b.n)
    asm volatile("prefetch.tensormap [%0];" ::"l"(&b.map[threadIdx.x]) : "memory");
  __syncthreads();

  if (threadIdx.x < kST) stats_role<kBF16>(b, G, u0, u1, sm, stages_s);
  else if (threadIdx.x < kST + kQT) quant_role<kBF16>(b, G, u0, u1, sm, stages_q);
  else if (threadIdx.x == kST + kQT) producer<kBF16, true>(b, G, u0, u1, sm, stages_s);
  else if (threadIdx.x == kST + kQT + 32) producer<kBF16, false>(b, G, u0, u1, sm, stages_q);

  __syncthreads();
  if (threadIdx.x == 0) {
    if (sm.status) atomicOr(G.header + 1, sm.status);
    __threadfence();
    const unsigned done = atomicAdd(G.header + 0, 1u) + 1u;
    sm.exit_last = (done == (unsigned)G.P);
  }
  __syncthreads();
  if (sm.exit_last) {
    // every other CTA has finished with the counters: zero them for the next call
    __threadfence();
    const int per_job = 2 + G.ngroups;
    for (int j = 0; j < b.n; ++j)
      for (int i = threadIdx.x; i < per_job; i += blockDim.x) b.job[j].ctr[i] = 0u;
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned st = atomicAdd(G.header + 1, 0u);
      if (G.dev_status) {
        if (G.first_launch) *G.dev_status = (int)st;
        else atomicOr(G.dev_status, (int)st);
      }
      G.header[1] = 0u;
      G.header[0] = 0u;
      __threadfence();
    }
  }
}

namespace {
template <bool kBF16>
cudaError_t prepare_kernel() {
  return cudaFuncSetAttribute(kv_fused_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<kBF16>::kDynSmem);
}
}  // namespace

cudaError_t launch_kv_fused(const FusedBatch& b, const FusedGeom& g, bool bf16, cudaStream_t s) {
  cudaError_t e = bf16 ? prepare_kernel<true>() : prepare_kernel<false>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.P);
  cfg.blockDim = dim3(kST + kQT + 64);
  cfg.dynamicSmemBytes = bf16 ? Cfg<true>::kDynSmem : Cfg<false>::kDynSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) return cudaLaunchKernelEx(&cfg, kv_fused_kernel<true>, b, g);
  return cudaLaunchKernelEx(&cfg, kv_fused_kernel<false>, b, g);
}

int fused_ctas_per_sm(bool bf16) {
  int n = 0;
  if ((bf16 ? prepare_kernel<true>() : prepare_kernel<false>()) != cudaSuccess) return 0;
  if (bf16)
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kv_fused_kernel<true>, kST + kQT + 64, Cfg<true>::kDynSmem);
  else
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kv_fused_kernel<false>, kST + kQT + 64, Cfg<false>::kDynSmem);
  return n;
}

// 2-D tensor map over x[T][C] with a W x 64-row box (the fused kernel's tile).
cudaError_t make_tile_map(CUtensorMap* map, const void* x, bool bf16, int64_t T, int C, int W) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const int es = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)C * es};
  cuuint32_t box[2] = {(cuuint32_t)W, (cuuint32_t)kTileRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                      const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace nvfp4
