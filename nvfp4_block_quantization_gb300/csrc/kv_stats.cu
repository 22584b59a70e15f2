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
// Work split.  The grid is cooperative, one CTA per SM.  The rows of every job
// are cut into stages of R rows and CTA c takes stages c, c + P, c + 2 P, ...
// (neighbouring CTAs read neighbouring stages at the same time).  A producer
// thread streams them into a shared-memory ring with 1-D bulk copies
// (cp.async.bulk), stage by stage; consumer thread t owns the 8-channel chunk
// t % tpr of every rpp-th row of a stage from t / tpr (a slab of 8 tpr
// channels; wider tensors take several slabs, and then each row of a stage is
// its own copy) and keeps, per channel,
// (sum, low part) by TwoSum -- so its partial sum is exact -- plus min and max
// (unsmoothed tensors: the absolute maximum only).
//
// A smoothed job's per-thread partials go to the workspace (one slice per job,
// [P][rpp][C] {sum, low, min, max}) and the CTA arrives on the job's counter;
// it then waits (bounded; all CTAs stream the same job at about the same time)
// until every CTA has arrived, reduces its slice of channels [c C / P,
// (c + 1) C / P) -- each channel's P * rpp partials combined in a fixed order,
// the mean the binary64 quotient of the compensated sum rounded once to fp32 --
// and folds max |x - mean| = max(max - mean, mean - min) (monotone rounding)
// into the job's amax.  An unsmoothed job's absolute maximum is folded into its
// amax directly.  Either way the CTA then counts itself on the job's ready
// counter (release).  The host orders unsmoothed jobs first.
//
// The grid lets its dependent launch start at once: the quantization kernel's
// CTAs wait for their own job's ready count (acquire), so one job's
// quantization overlaps the statistics of the next.
#include "bulk.cuh"
#include "common.cuh"
#include "kv_kernels.cuh"

namespace nvfp4 {

namespace {

constexpr int kThreads = kStatsConsumers + 32;  // consumer warps + one producer warp
constexpr int kWarps = kThreads / 32;
constexpr unsigned kStatusTimeout = 2u;

// Atomic add with release semantics at GPU scope: the calling thread's earlier
// writes and atomics, and those it has observed through a CTA barrier, are
// visible before the counter moves.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

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

struct StatsSmem {
  uint64_t full[kStatsStages], empty[kStatsStages];
  float4 runs[kThreads];  // slice reduction: one run per thread
  float red[kWarps];
  int ok;
  volatile int abort;  // a ring wait gave up: stop waiting
};

// Max over the CTA's threads; valid in every thread.
__device__ __forceinline__ float block_max(float v, StatsSmem& sm) {
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = max_nan(r, sm.red[w]);
  return r;
}

// Max over the first `n` threads (whole warps, synchronised by named barrier 1).
__device__ __forceinline__ float consumer_max(float v, StatsSmem& sm, int n) {
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  named_barrier(1, n);
  if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5] = v;
  named_barrier(1, n);
  float r = 0.0f;
  for (int w = 0; w < n / 32; ++w) r = max_nan(r, sm.red[w]);
  named_barrier(1, n);
  return r;
}

// Running statistics of the 8 channels a thread owns (4 channel pairs).
struct Acc8 {
  float2 s[4], l[4];
  float mn[8], mx[8];       // fp32 inputs
  uint32_t mnw[4], mxw[4];  // bf16 inputs: bf16 pairs
  float amax;               // unsmoothed fp32 inputs
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
  a.amax = 0.0f;
}

// One row of 8 channels (bf16: v0; fp32: v0, v1).
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

// 16-byte shared-memory load at a 32-bit shared address.
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

// Folds this thread's rows of one landed stage (`rows` valid rows of slab_bytes
// each, starting at shared address stage_s).
template <bool kBF16, bool kSmooth>
__device__ __forceinline__ void fold_stage(uint32_t stage_s, int slab_bytes, int rows, int rl, int rpp, int chunk,
                                           Acc8& a) {
  constexpr int es = kBF16 ? 2 : 4;
  uint32_t p = stage_s + (uint32_t)(rl * slab_bytes + 8 * chunk * es);
  const uint32_t step = (uint32_t)(rpp * slab_bytes);
  int j = rl;
  for (; j + 3 * rpp < rows; j += 4 * rpp, p += 4 * step) {  // four rows at a time
    uint4 v[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i][0] = lds_v4(p + i * step);
      v[i][1] = kBF16 ? v[i][0] : lds_v4(p + i * step + 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) fold_row<kBF16, kSmooth>(v[i][0], v[i][1], a);
  }
  for (; j < rows; j += rpp, p += step) {
    const uint4 v0 = lds_v4(p);
    const uint4 v1 = kBF16 ? v0 : lds_v4(p + 16);
    fold_row<kBF16, kSmooth>(v0, v1, a);
  }
}

// Combines, for this CTA's channel slice of smoothed job J, every CTA's
// partials (fixed order), writes the means and folds the slice's
// max |x - mean| into the job's amax.  The blockDim / nch threads of a channel
// each fold a contiguous run of its partials (loads 8 at a time); thread j < nch
// then folds channel j's runs in order.
__device__ void reduce_slice(const KvJob& J, const KvGeom& G, StatsSmem& sm, int nt) {
  const int c = blockIdx.x;
  const int ch0 = (int)((int64_t)c * G.C / G.P), ch1 = (int)((int64_t)(c + 1) * G.C / G.P);
  const int np = G.P * G.rpp;  // partials per channel
  float cam = 0.0f;
  for (int cb = ch0; cb < ch1; cb += nt) {
    const int nch = min(nt, ch1 - cb);
    const int runs = nt / nch;  // runs per channel
    const int j = threadIdx.x % nch, q = threadIdx.x / nch;
    float s = 0.0f, l = 0.0f, mn = __int_as_float(0x7f800000), mx = -mn;
    if (q < runs) {
      const int pa = (int)((int64_t)q * np / runs), pb = (int)((int64_t)(q + 1) * np / runs);
      const float4* src = J.part + cb + j;
      for (int p0 = pa; p0 < pb; p0 += 8) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          v[i] = p0 + i < pb ? __ldcg(src + (size_t)(p0 + i) * G.C) : make_float4(0.0f, 0.0f, mn, mx);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          comp_add(s, l, v[i].x, v[i].y);
          mn = min_nan(mn, v[i].z);
          mx = max_nan(mx, v[i].w);
        }
      }
    }
    named_barrier(1, nt);  // the previous block's runs have been read
    sm.runs[threadIdx.x] = make_float4(s, l, mn, mx);
    named_barrier(1, nt);
    if (threadIdx.x < nch) {
      s = 0.0f;
      l = 0.0f;
      for (int r = 0; r < runs; ++r) {
        const float4 v = sm.runs[r * nch + threadIdx.x];
        comp_add(s, l, v.x, v.y);
        mn = min_nan(mn, v.z);
        mx = max_nan(mx, v.w);
      }
      const int ch = cb + threadIdx.x;
      const float mu = J.mean_in ? J.mean_in[ch] : (float)(((double)s + (double)l) * G.inv_T);
      J.mean[ch] = mu;
      if (J.mean_out) J.mean_out[ch] = mu;
      cam = max_nan(cam, max_nan(__fsub_rn(mx, mu), __fsub_rn(mu, mn)));
    }
  }
  // consumer_max's barriers order every thread's mean stores before thread 0's release
  const float m = consumer_max(cam, sm, nt);
  if (threadIdx.x == 0) {
    atomicMax(J.ctr + 0, __float_as_uint(m) & 0x7fffffffu);
    red_release_add(J.ctr + 2, 1u);  // this CTA's share of the job is final
  }
}

}  // namespace

template <bool kBF16>
// at most 80 registers, so that a quantization CTA fits on the SM beside this one
__global__ void __maxnreg__(80) kv_stats_kernel(const __grid_constant__ KvBatch b, const KvGeom G) {
  extern __shared__ __align__(128) uint8_t ring[];
  StatsSmem& sm = *reinterpret_cast<StatsSmem*>(ring + (size_t)kStatsStages * kStatsStageBytes);
  constexpr int es = kBF16 ? 2 : 4;
  const int c = blockIdx.x;
  const size_t rs = (size_t)G.C * es;                 // row stride in bytes
  const int slab_ch = 8 * G.tpr;                      // channels per slab
  const int nslab = (G.C + slab_ch - 1) / slab_ch;
  const int consumers = (G.tpr * G.rpp + 31) / 32 * 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStatsStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], consumers / 32);
    }
    sm.abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // the quantization grid may launch now: its CTAs wait for each job's ready count,
  // not for this grid to end
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x >= consumers) {
    // producer: one thread streams the CTA's rows of every job and slab, stage by stage
    if (threadIdx.x == consumers) {
      const int T = (int)G.T, row_step = G.P * G.rows_per_stage;
      int st = 0, used = 0;  // ring slot; stages issued so far
      unsigned ph = 0;        // phase of the slot's current round
      for (int job = 0; job < b.n; ++job) {
        const uint8_t* x = static_cast<const uint8_t*>(b.job[job].x);
        for (int sl = 0; sl < nslab; ++sl) {
          const int s0 = sl * slab_ch, sb = min(slab_ch, G.C - s0) * es;  // slab bytes of this slab
          for (int row = c * G.rows_per_stage; row < T; row += row_step) {
            const int rows = min(G.rows_per_stage, T - row);
            if (used >= kStatsStages && !sm.abort && !mbar_wait(&sm.empty[st], ph ^ 1u)) {
              sm.abort = 1;
              atomicOr(G.header + 1, kStatusTimeout);
            }
            const int cur = st;
            if (++st == kStatsStages) {
              st = 0;
              ph ^= 1u;
            }
            ++used;
            if (sm.abort) continue;
            uint8_t* dst = ring + (size_t)cur * kStatsStageBytes;
            mbar_expect_tx(&sm.full[cur], (unsigned)(rows * sb));
            if (nslab == 1) {  // whole rows: the stage is one contiguous range
              bulk_load(dst, x + (size_t)row * rs, (unsigned)(rows * sb), &sm.full[cur]);
            } else {
              for (int i = 0; i < rows; ++i)
                bulk_load(dst + (size_t)i * sb, x + (size_t)(row + i) * rs + (size_t)s0 * es, (unsigned)sb,
                          &sm.full[cur]);
            }
          }
        }
      }
    }
  } else {
    // consumers
    const int chunk = threadIdx.x % G.tpr, rl = threadIdx.x / G.tpr;
    const bool lane_on = rl < G.rpp;  // threads beyond tpr * rpp idle
    const int T = (int)G.T, row_step = G.P * G.rows_per_stage;
    int st = 0;
    unsigned ph = 0;
    for (int job = 0; job < b.n; ++job) {
      const KvJob& J = b.job[job];
      const bool smooth = J.smooth != 0;
      float amax = 0.0f;
      for (int sl = 0; sl < nslab; ++sl) {
        const int s0 = sl * slab_ch, sb = min(slab_ch, G.C - s0) * es;
        const int ch = s0 + 8 * chunk;
        const bool on = lane_on && ch < G.C;
        Acc8 a;
        acc_reset(a);
        for (int row = c * G.rows_per_stage; row < T; row += row_step) {
          const int rows = min(G.rows_per_stage, T - row);
          if (!sm.abort && !mbar_wait(&sm.full[st], ph)) {
            sm.abort = 1;
            atomicOr(G.header + 1, kStatusTimeout);
          }
          const uint32_t stage = smem_u32(ring) + (uint32_t)(st * kStatsStageBytes);
          if (on) {
            if (smooth) fold_stage<kBF16, true>(stage, sb, rows, rl, G.rpp, chunk, a);
            else fold_stage<kBF16, false>(stage, sb, rows, rl, G.rpp, chunk, a);
          }
          __syncwarp();
          if ((threadIdx.x & 31) == 0) mbar_arrive(&sm.empty[st]);
          if (++st == kStatsStages) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (smooth) {
          if (on) {
            float4* dst = J.part + ((size_t)c * G.rpp + rl) * G.C + ch;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float mn0, mn1, mx0, mx1;
              if (kBF16) {
                mn0 = bf16lo(a.mnw[q]); mn1 = bf16hi(a.mnw[q]); mx0 = bf16lo(a.mxw[q]); mx1 = bf16hi(a.mxw[q]);
              } else {
                mn0 = a.mn[2 * q]; mn1 = a.mn[2 * q + 1]; mx0 = a.mx[2 * q]; mx1 = a.mx[2 * q + 1];
              }
              dst[2 * q] = make_float4(a.s[q].x, a.l[q].x, mn0, mx0);
              dst[2 * q + 1] = make_float4(a.s[q].y, a.l[q].y, mn1, mx1);
            }
          }
        } else {
          float v = a.amax;
          if (kBF16) {
            const uint32_t w = bf16x2_max_nan(bf16x2_max_nan(a.mxw[0], a.mxw[1]), bf16x2_max_nan(a.mxw[2], a.mxw[3]));
            v = max_nan(v, max_nan(bf16lo(w), bf16hi(w)));
          }
          amax = max_nan(amax, v);
        }
      }
      if (smooth) {
        named_barrier(1, consumers);  // every consumer's partials are written
        if (threadIdx.x == 0) {
          red_release_add(J.ctr + 1, 1u);  // this CTA's partials are published
          // every CTA streams the same job at about the same time: a short wait
          const uint64_t t0 = bulk_timer_ns();
          int ok = 1;
          for (unsigned it = 0; ld_acquire_u32(J.ctr + 1) < (unsigned)G.P; ++it) {
            if (bulk_timer_ns() - t0 > kBulkWaitNs) {
              ok = 0;
              atomicOr(G.header + 1, kStatusTimeout);
              break;
            }
            __nanosleep(it < 16 ? 64 : 256);
          }
          sm.ok = ok;
        }
        named_barrier(1, consumers);
        if (sm.ok) reduce_slice(J, G, sm, consumers);
      } else {
        const float m = consumer_max(amax, sm, consumers);
        if (threadIdx.x == 0) {
          atomicMax(J.ctr + 0, __float_as_uint(m) & 0x7fffffffu);
          red_release_add(J.ctr + 2, 1u);  // this CTA's share of the job is final
        }
      }
    }
  }
}

cudaError_t launch_kv_stats(const KvBatch& b, const KvGeom& g, bool bf16, cudaStream_t s) {
  const size_t smem = (size_t)kStatsStages * kStatsStageBytes + sizeof(StatsSmem);
  static std::atomic<unsigned long long> set_bf16{0}, set_f32{0};  // the limit is raised once per device
  cudaError_t e = bf16 ? smem_limit_once(kv_stats_kernel<true>, (int)smem, set_bf16)
                       : smem_limit_once(kv_stats_kernel<false>, (int)smem, set_f32);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.P);
  cfg.blockDim = dim3((g.tpr * g.rpp + 31) / 32 * 32 + 32);  // consumer warps + the producer warp
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // CTAs wait for each other's partials: all must be resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) return cudaLaunchKernelEx(&cfg, kv_stats_kernel<true>, b, g);
  return cudaLaunchKernelEx(&cfg, kv_stats_kernel<false>, b, g);
}

}  // namespace nvfp4
