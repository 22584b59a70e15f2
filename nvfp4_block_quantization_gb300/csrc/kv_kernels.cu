// kv_kernels.cu -- NVFP4 KV-chunk quantizer and dequantizer kernels (sm_103a).
//
// Method: "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video
// Generation" (summary page), inference step 7: each chunk's K is smoothed by
// subtracting its per-(head, channel) token mean and then quantized into the
// NVFP4 KV cache with Four-Over-Six ("4/6") adaptive block scales ("full-stack
// NVFP4" paragraph: keep whichever of two FP8 block-scale candidates has the
// lower MSE).
//
// Three stream-ordered kernels per call (or per batch of same-shape tensors):
//   kv_stats     one pass over x: per-(chunk of tokens, channel) partial sums
//                (TwoSum-compensated fp32), min and max for smoothed tensors;
//                per-CTA absolute maximum for unsmoothed ones.
//   kv_finalize  per channel: sum of the partials in binary64, mean rounded
//                once to fp32, channel amax = max(max - mean, mean - min)
//                (exactly max |fl(x - mean)| since rounding is monotone).
//   kv_quant     per 16-element block: smoothing, block amax, both candidate
//                scales, both quantizations and errors, the choice, packing.
#include "common.cuh"
#include "kv_kernels.cuh"

namespace nvfp4 {

// ---------------------------------------------------------------- loads
template <bool kBF16>
__device__ __forceinline__ void load8(const void* base, int64_t elem, float v[8]) {
  if (kBF16) {
    uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem));
    v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
    v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
    float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

template <int kThreads>
__device__ __forceinline__ float block_max_nan(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = (lane < (int)(blockDim.x >> 5)) ? red[lane] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  float r = red[0];
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------- stats
template <bool kBF16>
__global__ void __launch_bounds__(512) kv_stats_kernel(KvBatch b, KvGeom geo, int* dev_status) {
  __shared__ float red[32];
  const KvJob& J = b.job[blockIdx.z];
  const int chunk = blockIdx.x, ctile = blockIdx.y;
  const int c0 = ctile * kCTile + threadIdx.x * 8;
  const bool active = c0 < geo.C;
  const int64_t t0 = (int64_t)chunk * geo.rows_per_chunk;
  const int64_t t1 = min(geo.T, t0 + geo.rows_per_chunk);
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0 && dev_status) *dev_status = 0;

  if (J.smooth) {
    if (!active) return;
    float s[8], e[8], mn[8], mx[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) { s[j] = 0.0f; e[j] = 0.0f; mn[j] = __int_as_float(0x7f800000); mx[j] = -mn[j]; }
#pragma unroll 4
    for (int64_t t = t0; t < t1; ++t) {
      float v[8];
      load8<kBF16>(J.x, t * geo.C + c0, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float ns, err;
        two_sum(s[j], v[j], ns, err);
        s[j] = ns;
        e[j] = __fadd_rn(e[j], err);
        mn[j] = min_nan(mn[j], v[j]);
        mx[j] = max_nan(mx[j], v[j]);
      }
    }
    float4* part = J.part + (int64_t)chunk * geo.C + c0;
#pragma unroll
    for (int j = 0; j < 8; ++j) part[j] = make_float4(s[j], e[j], mn[j], mx[j]);
  } else {
    float m = 0.0f;
    if (active) {
#pragma unroll 4
      for (int64_t t = t0; t < t1; ++t) {
        float v[8];
        load8<kBF16>(J.x, t * geo.C + c0, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) m = max_nan(m, fabsf(v[j]));
      }
    }
    m = block_max_nan<512>(m, red);
    if (threadIdx.x == 0) J.amax_part[chunk * geo.nctiles + ctile] = m;
  }
}

// ---------------------------------------------------------------- finalize
__global__ void __launch_bounds__(256) kv_finalize_kernel(KvBatch b, KvGeom geo) {
  __shared__ float red[32];
  const KvJob& J = b.job[blockIdx.y];
  if (!J.smooth) return;
  const int c = blockIdx.x * 256 + threadIdx.x;
  float cam = 0.0f;
  if (c < geo.C) {
    double S = 0.0;
    float mn = __int_as_float(0x7f800000), mx = -mn;
    for (int k = 0; k < geo.nchunks; ++k) {
      float4 p = J.part[(int64_t)k * geo.C + c];
      S += (double)p.x;
      S += (double)p.y;
      mn = min_nan(mn, p.z);
      mx = max_nan(mx, p.w);
    }
    float mu = J.mean_in ? J.mean_in[c] : (float)(S / (double)geo.T);
    J.mean[c] = mu;
    if (J.mean_out) J.mean_out[c] = mu;
    cam = max_nan(__fsub_rn(mx, mu), __fsub_rn(mu, mn));
  }
  cam = block_max_nan<256>(cam, red);
  if (threadIdx.x == 0) J.amax_part[blockIdx.x] = cam;
}

// ---------------------------------------------------------------- quant
// Quantize the 16 values of one block under one candidate (inverse scale
// `inv`): codes packed into w[0..1], returns the fused sum of squared errors.
__device__ __forceinline__ float quant_candidate(const float z[16], float inv, uint32_t w[2]) {
  float acc = 0.0f;
  w[0] = 0u;
  w[1] = 0u;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    float y0 = __fmul_rn(z[2 * p], inv);
    float y1 = __fmul_rn(z[2 * p + 1], inv);
    uint32_t byte = e2m1x2(y0, y1);
    uint32_t q = e2m1x2_to_f16x2(byte);
    float d0 = __fsub_rn(y0, f16lo(q));
    acc = __fmaf_rn(d0, d0, acc);
    float d1 = __fsub_rn(y1, f16hi(q));
    acc = __fmaf_rn(d1, d1, acc);
    w[p >> 2] |= byte << (8 * (p & 3));
  }
  return acc;
}

template <bool kBF16>
__global__ void __launch_bounds__(256) kv_quant_kernel(KvBatch b, KvGeom geo, int* dev_status) {
  __shared__ QuantTable tab;
  __shared__ float red[32];
  const KvJob& J = b.job[blockIdx.y];

  float m = 0.0f;
  for (int i = threadIdx.x; i < J.namax; i += blockDim.x) m = max_nan(m, J.amax_part[i]);
  const float amax = block_max_nan<256>(m, red);
  const bool nonfinite = !finite_f(amax);
  const float g = nonfinite ? __int_as_float(0x7fc00000) : __fdiv_rn(amax, kTensorDenom);
  const float k6 = __frcp_rn(__fmul_rn(6.0f, g));
  const float k4 = __frcp_rn(__fmul_rn(4.0f, g));
  build_table(&tab, g);
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *J.tensor_scale = g;
    if (nonfinite && dev_status) atomicOr(dev_status, NVFP4_DEV_NONFINITE_FLAG);
  }

  const int64_t nb = geo.T * (int64_t)(geo.C / 16);
  const int bpr = geo.C / 16;
  for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nb; blk += (int64_t)gridDim.x * blockDim.x) {
    uint2 cw = make_uint2(0u, 0u);
    uint32_t sc = 0u;
    if (nonfinite) {
      sc = 0x7Fu;
    } else {
      float z[16];
      load8<kBF16>(J.x, blk * 16, z);
      load8<kBF16>(J.x, blk * 16 + 8, z + 8);
      if (J.smooth) {
        const int cb = (int)(blk % bpr);
        const float4* mu4 = reinterpret_cast<const float4*>(J.mean + cb * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float4 mu = mu4[q];
          z[4 * q + 0] = __fsub_rn(z[4 * q + 0], mu.x);
          z[4 * q + 1] = __fsub_rn(z[4 * q + 1], mu.y);
          z[4 * q + 2] = __fsub_rn(z[4 * q + 2], mu.z);
          z[4 * q + 3] = __fsub_rn(z[4 * q + 3], mu.w);
        }
      }
      float ab = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(z[i]));
      if (g > 0.0f && ab > 0.0f) {
        const uint32_t ee = e4m3x2(__fmul_rn(ab, k6), __fmul_rn(ab, k4));
        const uint32_t e6 = ee & 0xFFu, e4 = ee >> 8;
        const float inv6 = tab.inv[e6], inv4 = tab.inv[e4];
        uint32_t w6[2], w4[2];
        const float sum6 = quant_candidate(z, inv6, w6);
        const float sum4 = quant_candidate(z, inv4, w4);
        const float err6 = __fmul_rn(tab.e2[e6], sum6);
        const float err4 = __fmul_rn(tab.e2[e4], sum4);
        const bool ok6 = inv6 > 0.0f, ok4 = inv4 > 0.0f;
        if (ok4 && (!ok6 || err4 < err6)) {
          cw = make_uint2(w4[0], w4[1]);
          sc = e4;
        } else if (ok6) {
          cw = make_uint2(w6[0], w6[1]);
          sc = e6;
        }
      }
    }
    reinterpret_cast<uint2*>(J.codes)[blk] = cw;
    J.scales[blk] = (uint8_t)sc;
  }
}

// Empty chunk: nothing to quantize; the tensor scale and the mean are 0.
__global__ void kv_empty_kernel(KvBatch b, int C, int* dev_status) {
  const KvJob& J = b.job[blockIdx.x];
  for (int c = threadIdx.x; c < C; c += blockDim.x)
    if (J.mean_out) J.mean_out[c] = J.mean_in ? J.mean_in[c] : 0.0f;
  if (threadIdx.x == 0) {
    *J.tensor_scale = 0.0f;
    if (blockIdx.x == 0 && dev_status) *dev_status = 0;
  }
}

// ---------------------------------------------------------------- dequant
__global__ void __launch_bounds__(256) kv_dequant_kernel(const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ scales,
                                                         const float* __restrict__ tensor_scale,
                                                         const float* __restrict__ mean, int64_t tpg, int64_t T,
                                                         int C, __nv_bfloat16* __restrict__ out) {
  const int64_t nb = T * (int64_t)(C / 16);
  const int bpr = C / 16;
  for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nb; blk += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = blk / bpr;
    const int cb = (int)(blk - t * bpr);
    const int64_t grp = t / tpg;
    const float S = __fmul_rn(e4m3_value(scales[blk]), __ldg(tensor_scale + grp));
    const uint2 cw = __ldg(reinterpret_cast<const uint2*>(codes) + blk);
    const float* mu = mean ? mean + grp * C + cb * 16 : nullptr;
    uint32_t o[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const uint32_t byte = ((p < 4 ? cw.x : cw.y) >> (8 * (p & 3))) & 0xFFu;
      const uint32_t q = e2m1x2_to_f16x2(byte);
      float v0 = __fmul_rn(f16lo(q), S);
      float v1 = __fmul_rn(f16hi(q), S);
      if (mu) {
        v0 = __fadd_rn(v0, __ldg(mu + 2 * p));
        v1 = __fadd_rn(v1, __ldg(mu + 2 * p + 1));
      }
      __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
      o[p] = *reinterpret_cast<uint32_t*>(&h);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + blk * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_kv_quant(const KvBatch& b, const KvGeom& geo, bool bf16, int* status_reset, int* status_or,
                            int quant_ctas, cudaStream_t s) {
  if (geo.T == 0) {
    kv_empty_kernel<<<b.n, 256, 0, s>>>(b, geo.C, status_reset);
    return cudaGetLastError();
  }
  dim3 sg(geo.nchunks, geo.nctiles, b.n);
  if (bf16) kv_stats_kernel<true><<<sg, geo.ctile_threads, 0, s>>>(b, geo, status_reset);
  else kv_stats_kernel<false><<<sg, geo.ctile_threads, 0, s>>>(b, geo, status_reset);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kv_finalize_kernel<<<dim3(geo.nfin, b.n), 256, 0, s>>>(b, geo);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 qg(quant_ctas, b.n);
  if (bf16) kv_quant_kernel<true><<<qg, 256, 0, s>>>(b, geo, status_or);
  else kv_quant_kernel<false><<<qg, 256, 0, s>>>(b, geo, status_or);
  return cudaGetLastError();
}

cudaError_t launch_kv_dequant(const uint8_t* codes, const uint8_t* scales, const float* g, const float* mean,
                              int64_t tpg, int64_t T, int C, void* out, int ctas, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  kv_dequant_kernel<<<ctas, 256, 0, s>>>(codes, scales, g, mean, tpg, T, C, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace nvfp4
