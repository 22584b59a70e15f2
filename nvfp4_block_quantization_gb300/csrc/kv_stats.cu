// kv_stats.cu -- statistics pass of the KV chunk quantizer (sm_103a): per-channel
// token mean and the tensor's absolute maximum after K-smoothing.
//
// Method: "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video
// Generation" (summary page), inference step 7: each chunk's K is smoothed,
// K <- K - mean over the chunk's tokens (per head and channel), then quantized
// with 4/6 adaptive block scales, whose per-tensor scale g = amax / 2688 needs
// the absolute maximum of the smoothed tensor.  V is not smoothed; its amax is
// that of the raw values.
//
// Work split.  A tensor [T][C] is cut into channel groups of W channels; its
// ngroups * T (group, row) units are dealt out in contiguous ranges to P CTAs
// and every CTA walks its range in every job, so it holds one or a few long
// row segments of a group per job.
// One producer thread streams each segment as 2-D TMA tiles of 64 rows x W
// channels through a shared-memory ring; eight consumer warps fold them.  In a
// tile, warp w takes rows [8w, 8w + 8) and lane l owns the 8 channels
// 8 * (l % (W/8)) .. + 7 of every (32 / (W/8))-th of those rows, so a lane
// keeps the running statistics of the same channels over the whole segment in
// registers -- four independent channel-pair chains: (sum, low part) by TwoSum,
// so the partial sums are exact, plus min and max; unsmoothed tensors keep the
// absolute maximum only.
//
// At the end of a segment the CTA combines its lanes in a fixed order and
// publishes the segment's partial for its group; the last CTA to arrive at a
// group combines all of the group's partials (fixed order), computes the mean --
// the binary64 quotient of the compensated sum, rounded once to fp32 -- and the
// group's max |x - mean| (= max(max - mean, mean - min) under monotone
// rounding), and folds that into the job's amax with an atomic max.  The
// quantization kernel, launched after this grid, reads the finished amax.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kv_kernels.cuh"
#include "tma.cuh"

namespace nvfp4 {

namespace {

constexpr int kConsumers = kStatsConsumers;
constexpr int kWarps = kConsumers / 32;
constexpr int kThreads = kConsumers + 64;  // + producer warp + reducer warp
constexpr int kProducer = kConsumers, kReducer = kConsumers + 32;
constexpr int kTileRows = kStatsTileRows;
constexpr int kConsumerBar = 1;  // named barrier of the consumer warps
constexpr unsigned kStatusTimeout = 2u;
static_assert(kWarps * 8 == kTileRows, "each consumer warp folds 8 rows of a tile");

template <bool kBF16>
struct Cfg {
  static constexpr int kEsize = kBF16 ? 2 : 4;
  static constexpr int kStages = kBF16 ? 5 : 3;
  static constexpr int kStageBytes = kTileRows * kMaxGroupW * kEsize;
};

struct StatsSmem {
  uint64_t full[5], empty[5];          // tile ring
  uint64_t seg_full[2], seg_empty[2];  // segment partials handed to the reducer warp
  float wred[kWarps][4][kMaxGroupW];   // per-warp partials: sum, low part, min, max
  float4 seg[2][kMaxGroupW];           // the CTA's partial of a finished segment
  float red[kWarps];
  volatile int abort;  // a wait gave up: stop waiting
};

template <bool kBF16>
constexpr size_t dyn_smem_bytes() {
  return (size_t)Cfg<kBF16>::kStages * Cfg<kBF16>::kStageBytes + sizeof(StatsSmem);
}

__device__ __forceinline__ void consumer_sync() { named_barrier(kConsumerBar, kConsumers); }

// ------------------------------------------------------------------ partition
__device__ __forceinline__ int64_t range_start(const KvGeom& G, int c) { return (int64_t)c * G.U / G.P; }
__device__ __forceinline__ int owner_of(const KvGeom& G, int64_t u) { return (int)(((u + 1) * G.P - 1) / G.U); }
__device__ __forceinline__ unsigned group_arrivals(const KvGeom& G, int k) {
  if (G.U < G.P) return (unsigned)G.T;  // every non-empty CTA owns exactly one unit
  return (unsigned)(owner_of(G, (int64_t)k * G.T + G.T - 1) - owner_of(G, (int64_t)k * G.T) + 1);
}

// ------------------------------------------------------------------ arithmetic
// (s, n) pairs carry sum = s + n (n: the low part lost by s).
__device__ __forceinline__ void comp_add(float& s, float& n, float s2, float n2) {
  float t, e;
  two_sum(s, s2, t, e);
  s = t;
  n = __fadd_rn(n, __fadd_rn(n2, e));
}

// sum += x exactly as sum + low (TwoSum on a channel pair).
__device__ __forceinline__ void two_sum2(float2& sum, float2& low, float2 x) {
  const float2 m1 = make_float2(-1.0f, -1.0f);
  const float2 t = __fadd2_rn(sum, x);
  const float2 bp = __ffma2_rn(sum, m1, t);   // t - sum
  const float2 ap = __ffma2_rn(bp, m1, t);    // t - bp
  const float2 da = __ffma2_rn(ap, m1, sum);  // sum - ap
  const float2 db = __ffma2_rn(bp, m1, x);    // x - bp
  low = __fadd2_rn(low, __fadd2_rn(da, db));
  sum = t;
}

// Max over the consumer threads; valid in every consumer thread.
__device__ __forceinline__ float consumer_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  consumer_sync();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  consumer_sync();
  float r = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) r = max_nan(r, red[w]);
  return r;
}

// Running statistics of the 8 channels a lane owns (4 channel pairs).
struct Acc8 {
  float2 s[4], l[4];
  float mn[8], mx[8];       // fp32 inputs
  uint32_t mnw[4], mxw[4];  // bf16 inputs: bf16 pairs
  float amax;               // unsmoothed tensors
};

__device__ __forceinline__ void acc_reset(Acc8& a) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    a.s[m] = a.l[m] = make_float2(0.f, 0.f);
    a.mnw[m] = 0x7f807f80u;  // +inf pairs
    a.mxw[m] = 0xff80ff80u;  // -inf pairs
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a.mn[i] = __int_as_float(0x7f800000);
    a.mx[i] = -a.mn[i];
  }
}

// Lane geometry in a tile: lpr lanes per row (8 channels each), rpw rows per
// warp pass; the lane's rows are row0 + i * rpw, i < nr, inside its warp's 8.
struct LaneMap {
  int lpr, rpw, cq, row0, nr;
};

__device__ __forceinline__ LaneMap lane_map(int W) {
  LaneMap m;
  m.lpr = W / 8;
  m.rpw = 32 / m.lpr;
  const int lane = threadIdx.x & 31, lr = lane / m.lpr;
  m.cq = lane % m.lpr;
  m.row0 = 8 * (threadIdx.x >> 5) + lr;
  m.nr = lr < 8 ? (8 - lr + m.rpw - 1) / m.rpw : 0;
  return m;
}

// Folds one row (8 channels) into the lane's statistics.
template <bool kBF16, bool kSmooth>
__device__ __forceinline__ void fold_row(const uint4 v0, const uint4 v1, Acc8& a) {
  if (kBF16) {
    const uint32_t w[4] = {v0.x, v0.y, v0.z, v0.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (kSmooth) {
        a.mnw[q] = bf16x2_min_nan(a.mnw[q], w[q]);
        a.mxw[q] = bf16x2_max_nan(a.mxw[q], w[q]);
        two_sum2(a.s[q], a.l[q], make_float2(bf16lo(w[q]), bf16hi(w[q])));
      } else {
        a.mxw[q] = bf16x2_max_nan(a.mxw[q], w[q] & 0x7fff7fffu);
      }
    }
  } else {
    const float f[8] = {__uint_as_float(v0.x), __uint_as_float(v0.y), __uint_as_float(v0.z), __uint_as_float(v0.w),
                        __uint_as_float(v1.x), __uint_as_float(v1.y), __uint_as_float(v1.z), __uint_as_float(v1.w)};
    if (kSmooth) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a.mn[2 * q] = min_nan(a.mn[2 * q], f[2 * q]);
        a.mx[2 * q] = max_nan(a.mx[2 * q], f[2 * q]);
        a.mn[2 * q + 1] = min_nan(a.mn[2 * q + 1], f[2 * q + 1]);
        a.mx[2 * q + 1] = max_nan(a.mx[2 * q + 1], f[2 * q + 1]);
        two_sum2(a.s[q], a.l[q], make_float2(f[2 * q], f[2 * q + 1]));
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) a.amax = max_nan(a.amax, fabsf(f[q]));
    }
  }
}

// Folds this lane's rows of one landed tile with `nrows` valid rows.  A full
// tile with 128-channel groups (4 rows per lane) loads all of its rows first.
template <bool kBF16, bool kSmooth>
__device__ __forceinline__ void fold_tile(const uint8_t* tile, int W, const LaneMap& m, int nrows, Acc8& a) {
  constexpr int es = kBF16 ? 2 : 4;
  const uint8_t* base = tile + ((size_t)m.row0 * W + 8 * m.cq) * es;
  const size_t rstep = (size_t)m.rpw * W * es;
  if (m.nr == 4 && nrows == kTileRows) {
    uint4 v[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i][0] = *reinterpret_cast<const uint4*>(base + i * rstep);
      if (!kBF16) v[i][1] = *reinterpret_cast<const uint4*>(base + i * rstep + 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) fold_row<kBF16, kSmooth>(v[i][0], v[i][1], a);
    return;
  }
  for (int i = 0; i < m.nr; ++i) {
    if (m.row0 + i * m.rpw >= nrows) break;
    const uint4 v0 = *reinterpret_cast<const uint4*>(base + i * rstep);
    const uint4 v1 = kBF16 ? v0 : *reinterpret_cast<const uint4*>(base + i * rstep + 16);
    fold_row<kBF16, kSmooth>(v0, v1, a);
  }
}

// The last CTA to arrive at group k of job J (its reducer warp): combines every
// CTA's partial of the group in CTA order, writes the mean -- the binary64
// quotient of the compensated sum, rounded once to fp32 -- and folds the group's
// max |x - mean| into the job's amax.  Lane l handles channels l, l + 32, ...
__device__ __noinline__ void group_reduce(const KvJob& J, const KvGeom& G, int k) {
  const int lane = threadIdx.x & 31;
  const int cf = owner_of(G, (int64_t)k * G.T), cl = owner_of(G, (int64_t)k * G.T + G.T - 1);
  const int n = cl - cf + 1;
  float cam = 0.0f;
  for (int c0 = 0; c0 < G.W; c0 += 32) {  // warp-uniform: the shuffles below need every lane
    const int ch = c0 + lane;
    const bool act = ch < G.W;
    float s = 0.0f, l = 0.0f, mn = __int_as_float(0x7f800000), mx = -mn;
    for (int p0 = 0; p0 < n; p0 += 32) {
      // range starts of CTAs cf + p0 .. + 32, one per lane
      const int64_t rs_l = range_start(G, cf + p0 + lane);
      const int64_t re_l = range_start(G, cf + p0 + lane + 1);
      const int m = min(32, n - p0);
      for (int q0 = 0; q0 < m; q0 += 8) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int q = q0 + i;
          const int64_t a = __shfl_sync(0xffffffffu, rs_l, q & 31), e = __shfl_sync(0xffffffffu, re_l, q & 31);
          v[i] = make_float4(0.0f, 0.0f, mn, mx);  // neutral
          if (act && q < m && a != e) {  // an empty CTA (only when units < CTAs) has no partial
            const int seg = k - (int)(a / G.T);
            v[i] = __ldcg(J.part + ((int64_t)(cf + p0 + q) * G.smax + seg) * G.W + ch);
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          comp_add(s, l, v[i].x, v[i].y);
          mn = min_nan(mn, v[i].z);
          mx = max_nan(mx, v[i].w);
        }
      }
    }
    if (act) {
      const int c = k * G.W + ch;
      const float mu = J.mean_in ? J.mean_in[c] : (float)(((double)s + (double)l) / (double)G.T);
      J.mean[c] = mu;
      if (J.mean_out) J.mean_out[c] = mu;
      cam = max_nan(cam, max_nan(__fsub_rn(mx, mu), __fsub_rn(mu, mn)));
    }
  }
  for (int o = 16; o > 0; o >>= 1) cam = max_nan(cam, __shfl_xor_sync(0xffffffffu, cam, o));
  if (lane == 0) {
    atomicMax(J.ctr + 0, __float_as_uint(cam) & 0x7fffffffu);
    J.ctr[1 + k] = 0u;  // every partial of the group has arrived: ready for the next call
  }
}

// End of a segment (consumer threads): combine the lanes per channel in a fixed
// order and hand the CTA's partial to the reducer warp through slot `slot`
// (after the reducer has released the slot's previous use, when `reuse`).
template <bool kBF16>
__device__ __noinline__ void flush_segment(int W, const Acc8& a, int slot, unsigned reuse_parity, bool reuse,
                                           StatsSmem& sm) {
  const LaneMap m = lane_map(W);
  const int warp = threadIdx.x >> 5;
  float S[8], L[8], mn[8], mx[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    S[2 * q] = a.s[q].x; S[2 * q + 1] = a.s[q].y;
    L[2 * q] = a.l[q].x; L[2 * q + 1] = a.l[q].y;
    if (kBF16) {
      mn[2 * q] = bf16lo(a.mnw[q]); mn[2 * q + 1] = bf16hi(a.mnw[q]);
      mx[2 * q] = bf16lo(a.mxw[q]); mx[2 * q + 1] = bf16hi(a.mxw[q]);
    } else {
      mn[2 * q] = a.mn[2 * q]; mn[2 * q + 1] = a.mn[2 * q + 1];
      mx[2 * q] = a.mx[2 * q]; mx[2 * q + 1] = a.mx[2 * q + 1];
    }
  }
  // lanes of a warp that own the same channels (other rows) combine first
  for (int o = m.lpr; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float s2 = __shfl_xor_sync(0xffffffffu, S[i], o), l2 = __shfl_xor_sync(0xffffffffu, L[i], o);
      const float a2 = __shfl_xor_sync(0xffffffffu, mn[i], o), b2 = __shfl_xor_sync(0xffffffffu, mx[i], o);
      comp_add(S[i], L[i], s2, l2);
      mn[i] = min_nan(mn[i], a2);
      mx[i] = max_nan(mx[i], b2);
    }
  }
  consumer_sync();  // the previous segment's combine has read wred
  if ((threadIdx.x & 31) < m.lpr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sm.wred[warp][0][8 * m.cq + i] = S[i];
      sm.wred[warp][1][8 * m.cq + i] = L[i];
      sm.wred[warp][2][8 * m.cq + i] = mn[i];
      sm.wred[warp][3][8 * m.cq + i] = mx[i];
    }
  }
  consumer_sync();
  if (threadIdx.x < W) {  // every warp holds a partial of all W channels
    const int t = threadIdx.x;
    float s = 0.0f, l = 0.0f, lo = __int_as_float(0x7f800000), hi = -lo;
    for (int w = 0; w < kWarps; ++w) {
      comp_add(s, l, sm.wred[w][0][t], sm.wred[w][1][t]);
      lo = min_nan(lo, sm.wred[w][2][t]);
      hi = max_nan(hi, sm.wred[w][3][t]);
    }
    if (reuse && !sm.abort && !mbar_wait(&sm.seg_empty[slot], reuse_parity)) sm.abort = 1;
    sm.seg[slot][t] = make_float4(s, l, lo, hi);
    mbar_arrive(&sm.seg_full[slot]);
  }
}

// Walks the segments of [u0, u1): calls f(k, seg, r0, r1) per segment.
template <typename F>
__device__ __forceinline__ void for_each_segment(const KvGeom& G, int64_t u0, int64_t u1, F f) {
  const int k0 = (int)(u0 / G.T);
  for (int64_t u = u0; u < u1;) {
    const int k = (int)(u / G.T);
    const int64_t r0 = u - (int64_t)k * G.T, r1 = min(G.T, r0 + (u1 - u));
    f(k, k - k0, r0, r1);
    u += r1 - r0;
  }
}

// Walks the tiles of [u0, u1): calls f(k, seg, row0, rows, last_of_segment) per tile.
template <typename F>
__device__ __forceinline__ void for_each_tile(const KvGeom& G, int64_t u0, int64_t u1, F f) {
  for_each_segment(G, u0, u1, [&](int k, int seg, int64_t r0, int64_t r1) {
    for (int64_t row = r0; row < r1; row += kTileRows)
      f(k, seg, row, (int)min((int64_t)kTileRows, r1 - row), row + kTileRows >= r1);
  });
}

}  // namespace

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, kStatsCtasPerSm) kv_stats_kernel(const __grid_constant__ KvBatch b,
                                                                           const KvGeom G) {
  using CF = Cfg<kBF16>;
  extern __shared__ __align__(128) uint8_t dsm[];
  StatsSmem& sm = *reinterpret_cast<StatsSmem*>(dsm + (size_t)CF::kStages * CF::kStageBytes);
  const int cta = blockIdx.x;
  const int64_t u0 = range_start(G, cta), u1 = range_start(G, cta + 1);
  if (u0 >= u1) return;  // only when units < CTAs
  if (threadIdx.x == 0) {
    for (int i = 0; i < CF::kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.seg_full[i], G.W);
      mbar_init(&sm.seg_empty[i], 1);
    }
    sm.abort = 0;
    mbar_fence_init();
  }
  if (threadIdx.x < b.n) prefetch_tensormap(&b.map[threadIdx.x]);
  __syncthreads();

  // The CTA walks the same unit range of every job, in batch order (the host
  // puts smoothed tensors first, so their segment reductions overlap the
  // streaming of the others); one tile counter runs across jobs and one
  // segment counter across the smoothed jobs' segments.
  if (threadIdx.x >= kReducer) {
    // reducer warp: publishes each finished segment's partial; the group's last arrival reduces it
    const int lane = threadIdx.x & 31;
    int ns = 0;
    for (int job = 0; job < b.n; ++job) {
      const KvJob& J = b.job[job];
      if (!J.smooth) continue;
      for_each_segment(G, u0, u1, [&](int k, int seg, int64_t, int64_t) {
        const int slot = ns & 1;
        if (!sm.abort && !mbar_wait(&sm.seg_full[slot], (unsigned)(ns >> 1) & 1u)) {
          sm.abort = 1;
          atomicOr(G.header + 1, kStatusTimeout);
        }
        float4* dst = J.part + ((int64_t)cta * G.smax + seg) * G.W;
        for (int ch = lane; ch < G.W; ch += 32) dst[ch] = sm.seg[slot][ch];
        __threadfence();
        __syncwarp();
        bool last = false;
        if (lane == 0) {
          mbar_arrive(&sm.seg_empty[slot]);
          last = atomicAdd(J.ctr + 1 + k, 1u) + 1u == group_arrivals(G, k);
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
          __threadfence();
          group_reduce(J, G, k);
        }
        ++ns;
      });
    }
    return;
  }
  if (threadIdx.x >= kProducer) {
    // producer: one thread streams the tiles through the ring
    if (threadIdx.x != kProducer) return;
    const unsigned box_bytes = (unsigned)(kTileRows * G.W * CF::kEsize);
    int f = 0;
    for (int job = 0; job < b.n; ++job) {
      for_each_tile(G, u0, u1, [&](int k, int, int64_t row, int, bool) {
        const int st = f % CF::kStages;
        if (f >= CF::kStages && !sm.abort && !mbar_wait(&sm.empty[st], (unsigned)(f / CF::kStages - 1) & 1u)) {
          sm.abort = 1;
          atomicOr(G.header + 1, kStatusTimeout);
        }
        if (!sm.abort)
          tma_load_2d(dsm + (size_t)st * CF::kStageBytes, &b.map[job], k * G.W, (int)row, &sm.full[st], box_bytes);
        ++f;
      });
    }
    return;
  }

  // consumers
  const LaneMap m = lane_map(G.W);
  int f = 0, ns = 0;
  for (int job = 0; job < b.n; ++job) {
    const KvJob& J = b.job[job];
    const bool smooth = J.smooth != 0;
    Acc8 a;
    a.amax = 0.0f;
    acc_reset(a);
    for_each_tile(G, u0, u1, [&](int, int, int64_t, int rows, bool seg_end) {
      const int st = f % CF::kStages;
      if (!sm.abort && !mbar_wait(&sm.full[st], (unsigned)(f / CF::kStages) & 1u)) {
        sm.abort = 1;
        atomicOr(G.header + 1, kStatusTimeout);
      }
      const uint8_t* tile = dsm + (size_t)st * CF::kStageBytes;
      if (smooth) fold_tile<kBF16, true>(tile, G.W, m, rows, a);
      else fold_tile<kBF16, false>(tile, G.W, m, rows, a);
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&sm.empty[st]);
      ++f;
      if (smooth && seg_end) {
        flush_segment<kBF16>(G.W, a, ns & 1, (unsigned)((ns >> 1) - 1) & 1u, ns >= 2, sm);
        acc_reset(a);
        ++ns;
      }
    });
    if (!smooth) {
      float v = a.amax;
      if (kBF16) {
        const uint32_t w = bf16x2_max_nan(bf16x2_max_nan(a.mxw[0], a.mxw[1]), bf16x2_max_nan(a.mxw[2], a.mxw[3]));
        v = max_nan(v, max_nan(bf16lo(w), bf16hi(w)));
      }
      const float mx = consumer_max(v, sm.red);
      if (threadIdx.x == 0) atomicMax(J.ctr + 0, __float_as_uint(mx) & 0x7fffffffu);
    }
  }
  // the quantization kernel may start its prologue now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

namespace {
template <bool kBF16>
cudaError_t prepare() {
  return cudaFuncSetAttribute(kv_stats_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)dyn_smem_bytes<kBF16>());
}
}  // namespace

cudaError_t launch_kv_stats(const KvBatch& b, const KvGeom& g, bool bf16, cudaStream_t s) {
  cudaError_t e = bf16 ? prepare<true>() : prepare<false>();
  if (e != cudaSuccess) return e;
  const dim3 grid(g.P);
  if (bf16) kv_stats_kernel<true><<<grid, kThreads, dyn_smem_bytes<true>(), s>>>(b, g);
  else kv_stats_kernel<false><<<grid, kThreads, dyn_smem_bytes<false>(), s>>>(b, g);
  return cudaGetLastError();
}

// 2-D tensor map over x[T][C] with a W x 64-row box (the statistics tile).
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
