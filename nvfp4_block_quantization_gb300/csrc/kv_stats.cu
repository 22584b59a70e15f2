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
// (grid.y = job), so a CTA holds a few long row segments of one or two groups.
// Thread (ls, ro) of a CTA owns the 8 channels 8 * ls .. + 7 of a segment and
// every (256 / (W/8))-th row from ro: rows are read with 16-byte non-caching
// loads, 8 rows in flight per thread.  Smoothed tensors keep per-channel
// (sum, low part) by TwoSum, so the partial sums are exact, plus min and max;
// unsmoothed ones keep the absolute maximum only.
//
// At the end of a segment the CTA combines its threads in a fixed order and
// publishes the segment's partial for its group; the last CTA to arrive at a
// group combines all the group's partials (fixed order), computes the mean --
// the binary64 quotient of the compensated sum, rounded once to fp32 -- and the
// group's max |x - mean| (= max(max - mean, mean - min) under monotone
// rounding), and folds that into the job's amax with an atomic max.  The
// quantization kernel, launched after this one, reads the finished amax.
#include "common.cuh"
#include "kv_kernels.cuh"

namespace nvfp4 {

namespace {

constexpr int kThreads = kStatsThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsInFlight = 8;

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

__device__ __forceinline__ float block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) r = max_nan(r, red[w]);
  return r;
}

struct StatsSmem {
  float wred[kWarps][4][kMaxGroupW];  // per-warp partials: sum, low part, min, max; reused as scratch
  float red[kWarps];
  int last;
};

// Running statistics of the 8 channels a thread owns.
struct Acc8 {
  float2 s[4], l[4];
  float mn[8], mx[8];
  uint32_t mnw[4], mxw[4];  // bf16 inputs: min / max as bf16 pairs
  float amax;               // unsmoothed tensors
};

template <bool kBF16>
__device__ __forceinline__ void acc_init(Acc8& a) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    a.s[m] = make_float2(0.f, 0.f);
    a.l[m] = make_float2(0.f, 0.f);
    a.mnw[m] = 0x7f807f80u;  // +inf pairs
    a.mxw[m] = 0xff80ff80u;  // -inf pairs
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a.mn[i] = __int_as_float(0x7f800000);
    a.mx[i] = -a.mn[i];
  }
}

// Folds the rows [r0 + ro + i * rpp] < r1 of channels ch0 .. ch0 + 7.
template <bool kBF16, bool kSmooth>
__device__ __forceinline__ void fold_rows(const uint8_t* x, int64_t C, int ch0, int64_t r0, int64_t r1, int rpp, Acc8& a) {
  constexpr int es = kBF16 ? 2 : 4;
  constexpr int kIn = kBF16 ? kRowsInFlight : kRowsInFlight / 2;
  for (int64_t r = r0; r < r1; r += (int64_t)kIn * rpp) {
    uint4 v[kIn][kBF16 ? 1 : 2];
#pragma unroll
    for (int i = 0; i < kIn; ++i) {
      const int64_t rr = r + (int64_t)i * rpp;
      if (rr < r1) {
        const uint8_t* p = x + ((size_t)rr * C + ch0) * es;
        v[i][0] = ld_nc_v4(p);
        if (!kBF16) v[i][kBF16 ? 0 : 1] = ld_nc_v4(p + 16);  // fp32: 8 channels are 32 bytes
      }
    }
#pragma unroll
    for (int i = 0; i < kIn; ++i) {
      if (r + (int64_t)i * rpp >= r1) break;
      if (kBF16) {
        const uint32_t w[4] = {v[i][0].x, v[i][0].y, v[i][0].z, v[i][0].w};
        if (kSmooth) {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            a.mnw[m] = bf16x2_min_nan(a.mnw[m], w[m]);
            a.mxw[m] = bf16x2_max_nan(a.mxw[m], w[m]);
            two_sum2(a.s[m], a.l[m], make_float2(bf16lo(w[m]), bf16hi(w[m])));
          }
        } else {
#pragma unroll
          for (int m = 0; m < 4; ++m) a.mxw[m] = bf16x2_max_nan(a.mxw[m], w[m] & 0x7fff7fffu);
        }
      } else {
        const float f[8] = {__uint_as_float(v[i][0].x), __uint_as_float(v[i][0].y), __uint_as_float(v[i][0].z),
                            __uint_as_float(v[i][0].w), __uint_as_float(v[i][kBF16 ? 0 : 1].x),
                            __uint_as_float(v[i][kBF16 ? 0 : 1].y), __uint_as_float(v[i][kBF16 ? 0 : 1].z),
                            __uint_as_float(v[i][kBF16 ? 0 : 1].w)};
        if (kSmooth) {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            a.mn[2 * m] = min_nan(a.mn[2 * m], f[2 * m]);
            a.mn[2 * m + 1] = min_nan(a.mn[2 * m + 1], f[2 * m + 1]);
            a.mx[2 * m] = max_nan(a.mx[2 * m], f[2 * m]);
            a.mx[2 * m + 1] = max_nan(a.mx[2 * m + 1], f[2 * m + 1]);
            two_sum2(a.s[m], a.l[m], make_float2(f[2 * m], f[2 * m + 1]));
          }
        } else {
#pragma unroll
          for (int m = 0; m < 8; ++m) a.amax = max_nan(a.amax, fabsf(f[m]));
        }
      }
    }
  }
}

// The last CTA to arrive at group k of job J: combines every CTA's partial of
// the group, writes the mean and folds the group's max |x - mean| into the amax.
// The kThreads / W threads of a channel each fold a contiguous run of the
// partials (loads issued 8 at a time); thread tid < W then folds the runs in
// order, so the result does not depend on timing.
__device__ __noinline__ void group_reduce(const KvJob& J, const KvGeom& G, int k, StatsSmem& sm) {
  const int tid = threadIdx.x;
  const int chl = tid % G.W, q = tid / G.W, tpc = kThreads / G.W;
  const int cf = owner_of(G, (int64_t)k * G.T), cl = owner_of(G, (int64_t)k * G.T + G.T - 1);
  const int n = cl - cf + 1;
  // scratch: CTA range starts [n + 1] int64, then the runs [kThreads] float4
  int64_t* rs = reinterpret_cast<int64_t*>(&sm.wred[0][0][0]);
  float4* runs = reinterpret_cast<float4*>(rs + ((n + 2) & ~1));
  for (int i = tid; i <= n; i += kThreads) rs[i] = range_start(G, cf + i);
  __syncthreads();
  const int pa = q * n / tpc, pb = (q + 1) * n / tpc;
  float s = 0.0f, l = 0.0f, mn = __int_as_float(0x7f800000), mx = -mn;
  for (int p0 = pa; p0 < pb; p0 += 8) {
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = make_float4(0.0f, 0.0f, mn, mx);  // neutral
      const int p = p0 + i;
      if (p < pb && rs[p] != rs[p + 1]) {  // an empty CTA (only when units < CTAs) has no partial
        const int seg = k - (int)(rs[p] / G.T);
        v[i] = __ldcg(J.part + ((int64_t)(cf + p) * G.smax + seg) * G.W + chl);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      comp_add(s, l, v[i].x, v[i].y);
      mn = min_nan(mn, v[i].z);
      mx = max_nan(mx, v[i].w);
    }
  }
  runs[tid] = make_float4(s, l, mn, mx);
  __syncthreads();
  float cam = 0.0f;
  if (tid < G.W) {
    s = 0.0f;
    l = 0.0f;
    for (int r = 0; r < tpc; ++r) {
      const float4 v = runs[r * G.W + tid];
      comp_add(s, l, v.x, v.y);
      mn = min_nan(mn, v.z);
      mx = max_nan(mx, v.w);
    }
    const int ch = k * G.W + tid;
    const float mu = J.mean_in ? J.mean_in[ch] : (float)(((double)s + (double)l) / (double)G.T);
    J.mean[ch] = mu;
    if (J.mean_out) J.mean_out[ch] = mu;
    cam = max_nan(__fsub_rn(mx, mu), __fsub_rn(mu, mn));
  }
  const float gmax = block_max(cam, sm.red);
  if (tid == 0) {
    atomicMax(J.ctr + 0, __float_as_uint(gmax) & 0x7fffffffu);
    J.ctr[1 + k] = 0u;  // every partial of the group has arrived: ready for the next call
  }
}

// End of a segment: combine the CTA's threads per channel (fixed order), publish
// the partial, arrive; the last arrival reduces the group.
template <bool kBF16>
__device__ void flush_segment(const KvJob& J, const KvGeom& G, int k, int seg, Acc8& a, int ls, StatsSmem& sm) {
  const int tpr = G.W / 8, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float S[8], L[8], mn[8], mx[8];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    S[2 * m] = a.s[m].x; S[2 * m + 1] = a.s[m].y;
    L[2 * m] = a.l[m].x; L[2 * m + 1] = a.l[m].y;
    if (kBF16) {
      mn[2 * m] = bf16lo(a.mnw[m]); mn[2 * m + 1] = bf16hi(a.mnw[m]);
      mx[2 * m] = bf16lo(a.mxw[m]); mx[2 * m + 1] = bf16hi(a.mxw[m]);
    } else {
      mn[2 * m] = a.mn[2 * m]; mn[2 * m + 1] = a.mn[2 * m + 1];
      mx[2 * m] = a.mx[2 * m]; mx[2 * m + 1] = a.mx[2 * m + 1];
    }
  }
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
  __syncthreads();  // the scratch may still be in use by the previous segment's reduce
  if (lane < tpr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sm.wred[warp][0][8 * ls + i] = S[i];
      sm.wred[warp][1][8 * ls + i] = L[i];
      sm.wred[warp][2][8 * ls + i] = mn[i];
      sm.wred[warp][3][8 * ls + i] = mx[i];
    }
  }
  __syncthreads();
  if (threadIdx.x < G.W) {  // every warp holds a partial of all W channels
    const int t = threadIdx.x;
    float s = 0.0f, l = 0.0f, lo = __int_as_float(0x7f800000), hi = -lo;
    for (int w = 0; w < kWarps; ++w) {
      comp_add(s, l, sm.wred[w][0][t], sm.wred[w][1][t]);
      lo = min_nan(lo, sm.wred[w][2][t]);
      hi = max_nan(hi, sm.wred[w][3][t]);
    }
    J.part[((int64_t)blockIdx.x * G.smax + seg) * G.W + t] = make_float4(s, l, lo, hi);
    __threadfence();
  }
  __syncthreads();
  if (threadIdx.x == 0) sm.last = (atomicAdd(J.ctr + 1 + k, 1u) + 1u == group_arrivals(G, k));
  __syncthreads();
  if (sm.last) {
    __threadfence();
    group_reduce(J, G, k, sm);
  }
}

}  // namespace

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, kStatsCtasPerSm) kv_stats_kernel(const __grid_constant__ KvBatch b,
                                                                           const KvGeom G) {
  __shared__ StatsSmem sm;
  const KvJob& J = b.job[blockIdx.y];
  const int64_t u0 = range_start(G, blockIdx.x), u1 = range_start(G, blockIdx.x + 1);
  if (u0 >= u1) return;  // only when units < CTAs
  const uint8_t* x = static_cast<const uint8_t*>(J.x);
  const int tpr = G.W / 8, rpp = kThreads / tpr;
  const int ls = threadIdx.x % tpr, ro = threadIdx.x / tpr;
  const int k0 = (int)(u0 / G.T);
  Acc8 a;
  a.amax = 0.0f;
  acc_init<kBF16>(a);
  for (int64_t u = u0; u < u1;) {
    const int k = (int)(u / G.T);
    const int64_t r0 = u - (int64_t)k * G.T, r1 = min(G.T, r0 + (u1 - u));
    const int ch0 = k * G.W + 8 * ls;
    if (J.smooth) {
      fold_rows<kBF16, true>(x, G.C, ch0, r0 + ro, r1, rpp, a);
      flush_segment<kBF16>(J, G, k, k - k0, a, ls, sm);
      acc_init<kBF16>(a);
    } else {
      fold_rows<kBF16, false>(x, G.C, ch0, r0 + ro, r1, rpp, a);
    }
    u += r1 - r0;
  }
  if (!J.smooth) {
    float v = a.amax;
    if (kBF16) {
      const uint32_t w = bf16x2_max_nan(bf16x2_max_nan(a.mxw[0], a.mxw[1]), bf16x2_max_nan(a.mxw[2], a.mxw[3]));
      v = max_nan(v, max_nan(bf16lo(w), bf16hi(w)));
    }
    const float m = block_max(v, sm.red);
    if (threadIdx.x == 0) atomicMax(J.ctr + 0, __float_as_uint(m) & 0x7fffffffu);
  }
  // the quantization kernel may start its prologue now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

cudaError_t launch_kv_stats(const KvBatch& b, const KvGeom& g, bool bf16, cudaStream_t s) {
  const dim3 grid(g.P, b.n);
  if (bf16) kv_stats_kernel<true><<<grid, kThreads, 0, s>>>(b, g);
  else kv_stats_kernel<false><<<grid, kThreads, 0, s>>>(b, g);
  return cudaGetLastError();
}

}  // namespace nvfp4
