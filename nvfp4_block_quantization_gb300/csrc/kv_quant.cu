// kv_quant.cu -- Four-Over-Six NVFP4 quantization pass of the KV chunk
// quantizer (sm_103a).
//
// Method: "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video
// Generation" (summary page), inference step 7 (smoothed K and V go into the
// NVFP4 KV cache with 4/6 adaptive block scales) and the "full-stack NVFP4"
// paragraph: per 16-element block, two FP8 (E4M3) block-scale candidates map
// the block's absolute maximum to 6 and to 4; the block is quantized to E2M1
// under both and the candidate with the lower squared error is kept, ties to 6.
//
// Launch: a 1-D grid of CTAs of cw * rpp threads; CTA (job, y, x) owns block
// columns x * cw + c (16 channels each) of the rows y * rpp + r + i * gy * rpp, so
// a column's 16 channel means stay in registers for the whole loop; the next
// row's block is loaded before the current one is quantized.  All jobs but the
// last come first with gy_early row slots each (they run beside the statistics
// grid); the last job follows with gy_last slots (two CTAs per SM once the
// statistics grid has finished).  A warp reads 32 consecutive blocks of a row
// (coalesced) and writes their codes and scale bytes contiguously.
//
// The grid is a programmatic dependent of the statistics grid and may run beside
// it: each CTA fetches its first rows, waits (bounded) until every statistics
// CTA has counted itself ready for this CTA's job, reads the job's amax, and
// builds the per-tensor table: g = fl(amax / 2688) (or / 1792 with headroom) and, per E4M3 code E,
// fl(1 / fl(E * g)) and E * E.  Once every CTA has read the counters it needs
// (before its rows), the last of them resets the jobs' counters in the
// workspace and publishes the status word.
#include "common.cuh"
#include "four_over_six.cuh"
#include "kv_kernels.cuh"

namespace nvfp4 {

namespace {

constexpr unsigned kStatusNonfinite = 1u;

struct QuantConst {
  float2 tab[128];  // {fl(1 / fl(E * g)) or 0 when unusable, E * E} per E4M3 code
  int ok;  // this job's statistics are final
};

constexpr unsigned kStatusTimeout = 2u;
constexpr uint64_t kReadyWaitNs = 2000000000ull;

__device__ __forceinline__ uint64_t timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// One block's 16 inputs minus the channel means: z = fl(x - mu) (mu = 0 for
// unsmoothed tensors gives z = x exactly).
template <bool kBF16>
struct RawBlock {
  uint4 v[kBF16 ? 2 : 4];
};

template <bool kBF16>
__device__ __forceinline__ void load_block(const uint8_t* p, RawBlock<kBF16>& r) {
#pragma unroll
  for (int i = 0; i < (kBF16 ? 2 : 4); ++i) r.v[i] = ld_nc_v4(p + 16 * i);
}

__device__ __forceinline__ void st_cs_v2(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_cs_u8(void* p, uint32_t v) {
  asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <bool kBF16>
__device__ __forceinline__ void smooth_block(const RawBlock<kBF16>& r, const float mu[16], float z[16]) {
  if (kBF16) {
    const uint32_t w[8] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w, r.v[1].x, r.v[1].y, r.v[1].z, r.v[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) bf16x2_minus(w[i], mu[2 * i], mu[2 * i + 1], z[2 * i], z[2 * i + 1]);
  } else {
#pragma unroll
    for (int q = 0; q < (kBF16 ? 2 : 4); ++q) {
      z[4 * q] = __fsub_rn(__uint_as_float(r.v[q].x), mu[4 * q]);
      z[4 * q + 1] = __fsub_rn(__uint_as_float(r.v[q].y), mu[4 * q + 1]);
      z[4 * q + 2] = __fsub_rn(__uint_as_float(r.v[q].z), mu[4 * q + 2]);
      z[4 * q + 3] = __fsub_rn(__uint_as_float(r.v[q].w), mu[4 * q + 3]);
    }
  }
}

// Smooths, quantizes and stores one loaded block.
template <bool kBF16>
__device__ __forceinline__ void quant_store(const RawBlock<kBF16>& r, const float mu[16], const float2* tab, float k6,
                                            float k4, bool nonfinite, uint2* pc, uint8_t* ps) {
  float z[16];
  smooth_block<kBF16>(r, mu, z);
  uint2 code;
  uint32_t sc;
  quant_block(z, tab, k6, k4, nonfinite, code, sc);
  st_cs_v2(pc, code);
  st_cs_u8(ps, sc);
}

}  // namespace

template <bool kBF16>
__global__ void __launch_bounds__(256, 2) kv_quant_kernel(const __grid_constant__ KvBatch b, const KvGeom G,
                                                          const KvQuantShape S) {
  __shared__ QuantConst qc;
  constexpr int es = kBF16 ? 2 : 4;
  // this CTA's job, row slot y of gy, and column group x
  const int n_early = S.gx * S.gy_early * (b.n - 1);
  int job, y, x, gy;
  if ((int)blockIdx.x < n_early) {
    job = blockIdx.x / (S.gx * S.gy_early);
    const int rem = blockIdx.x - job * (S.gx * S.gy_early);
    y = rem / S.gx;
    x = rem - y * S.gx;
    gy = S.gy_early;
  } else {
    job = b.n - 1;
    const int rem = blockIdx.x - n_early;
    y = rem / S.gx;
    x = rem - y * S.gx;
    gy = S.gy_last;
  }
  const KvJob& J = b.job[job];
  const int nbr = G.C / 16;  // blocks per row
  const int c = threadIdx.x % S.cw, rl = threadIdx.x / S.cw;
  const int cb = x * S.cw + c;
  const bool active = cb < nbr;
  // rows r, r + step, r + 2 step, ... in pairs (r, r + step)
  const int64_t step = (int64_t)gy * S.rpp;
  const size_t row_bytes = (size_t)G.C * es;
  int64_t r = (int64_t)y * S.rpp + rl;
  const uint8_t* px = static_cast<const uint8_t*>(J.x) + (size_t)16 * cb * es + (size_t)r * row_bytes;
  const size_t px_step = (size_t)step * row_bytes;

  // the inputs do not depend on the statistics grid: fetch the first pair now
  RawBlock<kBF16> a0 = {}, a1 = {};
  if (active && r < G.T) load_block<kBF16>(px, a0);
  if (active && r + step < G.T) load_block<kBF16>(px + px_step, a1);

  // wait (bounded) until every statistics CTA has finished this job: its amax and means are read below
  if (threadIdx.x == 0) {
    const uint64_t t0 = timer_ns();
    int ok = 1;
    for (unsigned it = 0; ld_acquire_u32(J.ctr + 2) < (unsigned)G.P; ++it) {
      if (timer_ns() - t0 > kReadyWaitNs) {
        ok = 0;
        atomicOr(G.header + 1, kStatusTimeout);
        break;
      }
      __nanosleep(64);
    }
    qc.ok = ok;
  }
  __syncthreads();
  const unsigned amax_bits = qc.ok ? *reinterpret_cast<volatile const unsigned*>(J.ctr) : 0x7fc00000u;
  const float amax = __uint_as_float(amax_bits);
  const bool nonfinite = !finite_f(amax);
  const float g = nonfinite ? __int_as_float(0x7fc00000) : __fdiv_rn(amax, G.denom);
  for (int e = threadIdx.x; e < 128; e += blockDim.x) {
    const float E = e4m3_value((uint32_t)e);
    const float Sc = __fmul_rn(E, g);
    const float inv = __frcp_rn(Sc);
    const bool ok = (E > 0.0f) && (Sc > 0.0f) && finite_f(inv);
    qc.tab[e] = make_float2(ok ? inv : 0.0f, ok ? __fmul_rn(E, E) : 0.0f);
  }
  if (threadIdx.x == 0 && x == 0 && y == 0) {
    *J.tensor_scale = g;
    if (nonfinite) atomicOr(G.header + 1, kStatusNonfinite);
  }
  const float k6 = __frcp_rn(__fmul_rn(6.0f, g)), k4 = __frcp_rn(__fmul_rn(4.0f, g));
  __syncthreads();
  // Every thread of this CTA has read the counters it needs, so the CTA counts
  // itself done with the workspace now (not after its rows): the last CTA to
  // arrive returns the workspace to its idle state while the others still work.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(G.header + 0, 1u) + 1u == gridDim.x) {
      __threadfence();
      for (int j = 0; j < b.n; ++j) {
        b.job[j].ctr[0] = 0u;
        b.job[j].ctr[1] = 0u;
        b.job[j].ctr[2] = 0u;
      }
      const unsigned st = atomicAdd(G.header + 1, 0u);
      if (G.dev_status) {
        if (G.first_launch) *G.dev_status = (int)st;
        else atomicOr(G.dev_status, (int)st);
      }
      G.header[1] = 0u;
      G.header[0] = 0u;
    }
  }

  if (active) {
    float mu[16];
    if (J.smooth) {
      const float4* m4 = reinterpret_cast<const float4*>(J.mean + 16 * cb);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = __ldcg(m4 + i);
        mu[4 * i] = v.x; mu[4 * i + 1] = v.y; mu[4 * i + 2] = v.z; mu[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) mu[i] = 0.0f;
    }
    uint2* pc = reinterpret_cast<uint2*>(J.codes) + (size_t)r * nbr + cb;
    uint8_t* ps = J.scales + (size_t)r * nbr + cb;
    const size_t pq_step = (size_t)step * nbr;
    // rows k = 0 .. n-1 of this thread (row r + k * step), two per half-iteration: the
    // pair in (a0, a1) is quantized while the next pair loads into (b0, b1), then
    // the roles swap, so no buffer is copied
    const int n = r < G.T ? (int)((G.T - r + step - 1) / step) : 0;
    RawBlock<kBF16> b0, b1;
    for (int k = 0; k < n; k += 4) {
      if (k + 2 < n) load_block<kBF16>(px + 2 * px_step, b0);
      if (k + 3 < n) load_block<kBF16>(px + 3 * px_step, b1);
      quant_store<kBF16>(a0, mu, qc.tab, k6, k4, nonfinite, pc, ps);
      if (k + 1 < n) quant_store<kBF16>(a1, mu, qc.tab, k6, k4, nonfinite, pc + pq_step, ps + pq_step);
      if (k + 2 >= n) break;
      if (k + 4 < n) load_block<kBF16>(px + 4 * px_step, a0);
      if (k + 5 < n) load_block<kBF16>(px + 5 * px_step, a1);
      quant_store<kBF16>(b0, mu, qc.tab, k6, k4, nonfinite, pc + 2 * pq_step, ps + 2 * pq_step);
      if (k + 3 < n) quant_store<kBF16>(b1, mu, qc.tab, k6, k4, nonfinite, pc + 3 * pq_step, ps + 3 * pq_step);
      px += 4 * px_step;
      pc += 4 * pq_step;
      ps += 4 * pq_step;
    }
  }

}

KvQuantShape kv_quant_shape(int64_t T, int C, int n_jobs, int sms) {
  KvQuantShape q;
  const int nbr = C / 16;
  q.cw = nbr < 256 ? nbr : 256;
  q.rpp = 256 / q.cw;
  q.gx = (nbr + q.cw - 1) / q.cw;
  const int64_t max_gy = (T + q.rpp - 1) / q.rpp;
  auto clamp_gy = [&](int64_t want_ctas) {
    int64_t gy = (want_ctas + q.gx - 1) / q.gx;
    if (gy > max_gy) gy = max_gy;
    if (gy < 1) gy = 1;
    if (gy > 65535) gy = 65535;
    return (int)gy;
  };
  const int64_t s = sms > 0 ? sms : 1;
  // jobs but the last share two CTAs per SM (one of which fits beside the statistics
  // grid); the last job, which starts when the statistics grid has finished, gets two
  // CTAs per SM of its own
  q.gy_early = n_jobs > 1 ? clamp_gy((2 * s + n_jobs - 1) / n_jobs) : 1;
  q.gy_last = clamp_gy(2 * s);
  q.ctas = q.gx * q.gy_early * (n_jobs - 1) + q.gx * q.gy_last;
  return q;
}

cudaError_t launch_kv_quant(const KvBatch& b, const KvGeom& g, const KvQuantShape& q, bool bf16, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(q.ctas);
  cfg.blockDim = dim3(q.cw * q.rpp);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) return cudaLaunchKernelEx(&cfg, kv_quant_kernel<true>, b, g, q);
  return cudaLaunchKernelEx(&cfg, kv_quant_kernel<false>, b, g, q);
}

}  // namespace nvfp4
