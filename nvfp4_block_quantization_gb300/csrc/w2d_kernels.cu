// w2d_kernels.cu -- NVFP4 weight quantizer with 16x16 2-D blocks (sm_103a).
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page), training pipeline step 4: weights carry 2-D block scales.
// Each 16x16 tile gets one E4M3 scale chosen by Four-Over-Six; the tile's error
// accumulates its 256 squared errors in row-major order.
//
//   w2d_amax   per-CTA absolute maximum (NaN-propagating) over the matrix.
//   w2d_quant  one thread per tile: tile amax, both candidates' errors, the
//              choice, then the chosen codes (the tile is re-read from L1/L2).
#include "common.cuh"
#include "kv_kernels.cuh"

namespace nvfp4 {

template <bool kBF16>
__device__ __forceinline__ void load_row16(const void* base, int64_t elem, float v[16]) {
  if (kBF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem);
    uint4 a = __ldg(p), b = __ldg(p + 1);
    uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) { v[2 * j] = bf16lo(w[j]); v[2 * j + 1] = bf16hi(w[j]); }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float4 a = __ldg(p + j);
      v[4 * j] = a.x; v[4 * j + 1] = a.y; v[4 * j + 2] = a.z; v[4 * j + 3] = a.w;
    }
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(256) w2d_amax_kernel(const void* w, int64_t n16, float* amax_part, int* dev_status) {
  __shared__ float red[32];
  if (blockIdx.x == 0 && threadIdx.x == 0 && dev_status) *dev_status = 0;
  float m = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x) {
    float v[16];
    load_row16<kBF16>(w, i * 16, v);
#pragma unroll
    for (int j = 0; j < 16; ++j) m = max_nan(m, fabsf(v[j]));
  }
  for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) amax_part[blockIdx.x] = m;
  }
}

// Sum of fused squared errors of one 16-element tile row under `inv`.
__device__ __forceinline__ float row_err(const float v[16], float inv, float acc) {
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    float y0 = __fmul_rn(v[2 * p], inv);
    float y1 = __fmul_rn(v[2 * p + 1], inv);
    uint32_t q = e2m1x2_to_f16x2(e2m1x2(y0, y1));
    float d0 = __fsub_rn(y0, f16lo(q));
    acc = __fmaf_rn(d0, d0, acc);
    float d1 = __fsub_rn(y1, f16hi(q));
    acc = __fmaf_rn(d1, d1, acc);
  }
  return acc;
}

template <bool kBF16>
__global__ void __launch_bounds__(256) w2d_quant_kernel(const void* w, int64_t M, int64_t N,
                                                        const float* amax_part, int namax, uint8_t* codes,
                                                        uint8_t* scales, float* tensor_scale, int* dev_status) {
  __shared__ QuantTable tab;
  __shared__ float red[32];
  float m = 0.0f;
  for (int i = threadIdx.x; i < namax; i += blockDim.x) m = max_nan(m, amax_part[i]);
  for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float amax = red[0];
  const bool nonfinite = !finite_f(amax);
  const float g = nonfinite ? __int_as_float(0x7fc00000) : __fdiv_rn(amax, kTensorDenom);
  const float k6 = __frcp_rn(__fmul_rn(6.0f, g));
  const float k4 = __frcp_rn(__fmul_rn(4.0f, g));
  build_table(&tab, g);
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *tensor_scale = g;
    if (nonfinite && dev_status) atomicOr(dev_status, NVFP4_DEV_NONFINITE_FLAG);
  }

  const int64_t TN = N / 16;
  const int64_t ntiles = (M / 16) * TN;
  for (int64_t tl = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; tl < ntiles; tl += (int64_t)gridDim.x * blockDim.x) {
    const int64_t ti = tl / TN, tj = tl - ti * TN;
    const int64_t base = ti * 16 * N + tj * 16;
    uint32_t sc = 0u;
    float inv = 0.0f;
    if (nonfinite) {
      sc = 0x7Fu;
    } else {
      float ab = 0.0f;
      for (int r = 0; r < 16; ++r) {
        float v[16];
        load_row16<kBF16>(w, base + r * N, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) ab = fmaxf(ab, fabsf(v[j]));
      }
      if (g > 0.0f && ab > 0.0f) {
        const uint32_t ee = e4m3x2(__fmul_rn(ab, k6), __fmul_rn(ab, k4));
        const uint32_t e6 = ee & 0xFFu, e4 = ee >> 8;
        const float inv6 = tab.inv[e6], inv4 = tab.inv[e4];
        float acc6 = 0.0f, acc4 = 0.0f;
        for (int r = 0; r < 16; ++r) {
          float v[16];
          load_row16<kBF16>(w, base + r * N, v);
          acc6 = row_err(v, inv6, acc6);
          acc4 = row_err(v, inv4, acc4);
        }
        const float err6 = __fmul_rn(tab.e2[e6], acc6);
        const float err4 = __fmul_rn(tab.e2[e4], acc4);
        const bool ok6 = inv6 > 0.0f, ok4 = inv4 > 0.0f;
        if (ok4 && (!ok6 || err4 < err6)) {
          sc = e4;
          inv = inv4;
        } else if (ok6) {
          sc = e6;
          inv = inv6;
        }
      }
    }
    for (int r = 0; r < 16; ++r) {
      uint32_t wd[2] = {0u, 0u};
      if (inv > 0.0f) {
        float v[16];
        load_row16<kBF16>(w, base + r * N, v);
#pragma unroll
        for (int p = 0; p < 8; ++p)
          wd[p >> 2] |= e2m1x2(__fmul_rn(v[2 * p], inv), __fmul_rn(v[2 * p + 1], inv)) << (8 * (p & 3));
      }
      reinterpret_cast<uint2*>(codes + (base + r * N) / 2)[0] = make_uint2(wd[0], wd[1]);
    }
    scales[tl] = (uint8_t)sc;
  }
}

__global__ void __launch_bounds__(256) w2d_dequant_kernel(const uint8_t* __restrict__ codes,
                                                          const uint8_t* __restrict__ scales,
                                                          const float* __restrict__ tensor_scale, int64_t M,
                                                          int64_t N, __nv_bfloat16* __restrict__ out) {
  const int64_t n16 = M * N / 16;
  const int64_t TN = N / 16;
  const float g = __ldg(tensor_scale);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = (i * 16) / N, c = (i * 16) - r * N;
    const float S = __fmul_rn(e4m3_value(scales[(r / 16) * TN + c / 16]), g);
    const uint2 cw = __ldg(reinterpret_cast<const uint2*>(codes) + i);
    uint32_t o[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const uint32_t byte = ((p < 4 ? cw.x : cw.y) >> (8 * (p & 3))) & 0xFFu;
      const uint32_t q = e2m1x2_to_f16x2(byte);
      __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(f16lo(q), S), __fmul_rn(f16hi(q), S));
      o[p] = *reinterpret_cast<uint32_t*>(&h);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + i * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

cudaError_t launch_w2d_quant(const void* w, bool bf16, const W2dGeom& geo, uint8_t* codes, uint8_t* scales,
                             float* tensor_scale, int* dev_status, float* amax_part, int quant_ctas,
                             cudaStream_t s) {
  const int64_t n16 = geo.M * geo.N / 16;
  if (bf16) w2d_amax_kernel<true><<<geo.amax_ctas, 256, 0, s>>>(w, n16, amax_part, dev_status);
  else w2d_amax_kernel<false><<<geo.amax_ctas, 256, 0, s>>>(w, n16, amax_part, dev_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (bf16)
    w2d_quant_kernel<true><<<quant_ctas, 256, 0, s>>>(w, geo.M, geo.N, amax_part, geo.amax_ctas, codes, scales,
                                                      tensor_scale, dev_status);
  else
    w2d_quant_kernel<false><<<quant_ctas, 256, 0, s>>>(w, geo.M, geo.N, amax_part, geo.amax_ctas, codes, scales,
                                                       tensor_scale, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_w2d_dequant(const uint8_t* codes, const uint8_t* scales, const float* g, int64_t M, int64_t N,
                               void* out, int ctas, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  w2d_dequant_kernel<<<ctas, 256, 0, s>>>(codes, scales, g, M, N, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace nvfp4
