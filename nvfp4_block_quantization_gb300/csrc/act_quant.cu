// act_quant.cu -- the W4A4 path's activation quantizer (sm_103a): optionally
// the random Hadamard transform of every 16-element block, then 1-D
// Four-Over-Six NVFP4, with the block scales written straight into the tensor
// cores' scale layout.
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page), training step 4: NVFP4 GEMMs with 1-D block scales for
// activations and random Hadamard transforms against outliers; inference
// step 6: W4A4.
//
// The result is, bit for bit, the composition of the separate calls: the
// transform (nvfp4_rht16, fp32 out), the 1-D quantizer on that fp32 tensor
// (nvfp4_kv_smooth_quant with H = 1, no smoothing), and the scale
// rearrangement (nvfp4_scales_to_mma).  Fused, the transformed values never
// leave registers:
//   act_amax   one thread per block: load 32 bytes, transform, fold |y| into a
//              NaN-propagating maximum; one partial per CTA;
//   act_quant  reduce the partials to the tensor scale, build the candidate
//              table, then one thread per block: load (the second read mostly
//              hits L2), transform again, Four-Over-Six, store 8 code bytes and
//              the scale byte at its place in the tensor-core layout; the
//              layout's padding is zeroed by the same grid.
#include "nvfp4.h"
#include "common.cuh"
#include "four_over_six.cuh"
#include "rht16.cuh"

namespace nvfp4 {
namespace {

constexpr int kActThreads = 256;
constexpr int kActCtasPerSm = 4;     // amax pass; the quantization pass runs 3 per SM

template <bool kRHT>
__device__ __forceinline__ void act_block(const uint16_t* x, int64_t b, uint32_t signs, float v[16]) {
  uint32_t w[8];
  ld_nc_v8(x + b * 16, w);
#pragma unroll
  for (int i = 0; i < 8; ++i) { v[2 * i] = bf16lo(w[i]); v[2 * i + 1] = bf16hi(w[i]); }
  if (kRHT) rht16_block(v, signs);
}

__device__ __forceinline__ float block_max_all(float m, float* red) {
  for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  float r = 0.0f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = max_nan(r, red[i]);
  return r;
}

template <bool kRHT>
__global__ void __launch_bounds__(kActThreads) act_amax_kernel(const uint16_t* __restrict__ x, int64_t nblocks,
                                                               uint32_t signs, float* __restrict__ part) {
  __shared__ float red[32];
  float m = 0.0f;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblocks; b += (int64_t)gridDim.x * blockDim.x) {
    float v[16];
    act_block<kRHT>(x, b, signs, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) m = max_nan(m, fabsf(v[i]));
  }
  m = block_max_all(m, red);
  if (threadIdx.x == 0) part[blockIdx.x] = m;
}

// Byte offset of block scale (r, kb) in the tensor-core layout with kbt K tiles.
__device__ __forceinline__ int64_t mma_offset(int64_t r, int64_t kb, int64_t kbt) {
  return (((r >> 7) * kbt + (kb >> 2)) << 9) + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

template <bool kRHT>
__global__ void __launch_bounds__(kActThreads, 3) act_quant_kernel(const uint16_t* __restrict__ x, int64_t M,
                                                                   int64_t KB, uint32_t signs,
                                                                   const float* __restrict__ part, int nparts,
                                                                   uint8_t* __restrict__ codes,
                                                                   uint8_t* __restrict__ sf,
                                                                   float* __restrict__ tensor_scale,
                                                                   int* __restrict__ dev_status) {
  __shared__ float2 tab[128];
  __shared__ float red[32];
  float m = 0.0f;
  for (int i = threadIdx.x; i < nparts; i += blockDim.x) m = max_nan(m, part[i]);
  const float amax = block_max_all(m, red);
  const bool nonfinite = !finite_f(amax);
  const float g = nonfinite ? __int_as_float(0x7fc00000) : __fdiv_rn(amax, kTensorDenom);
  const float k6 = __frcp_rn(__fmul_rn(6.0f, g)), k4 = __frcp_rn(__fmul_rn(4.0f, g));
  for (int e = threadIdx.x; e < 128; e += blockDim.x) {
    const float E = e4m3_value((uint32_t)e);  // code 127 -> NaN -> unusable
    const float Sc = __fmul_rn(E, g);
    const float inv = __frcp_rn(Sc);
    const bool ok = (E > 0.0f) && (Sc > 0.0f) && finite_f(inv);
    tab[e] = make_float2(ok ? inv : 0.0f, ok ? __fmul_rn(E, E) : 0.0f);
  }
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *tensor_scale = g;
    if (dev_status) *dev_status = nonfinite ? NVFP4_DEV_NONFINITE : NVFP4_DEV_OK;
  }
  const int64_t nblocks = M * KB, kbt = (KB + 3) / 4;
  // block b is (row r, block kb) with b = r KB + kb; the grid stride moves both by
  // constants, so they advance without a division per block
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t b0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t dr = stride / KB, dkb = stride - dr * KB;
  int64_t r = b0 / KB, kb = b0 - r * KB;
  for (int64_t b = b0; b < nblocks; b += stride) {
    float z[16];
    act_block<kRHT>(x, b, signs, z);
    uint2 code;
    uint32_t sc;
    quant_block(z, tab, k6, k4, nonfinite, code, sc);
    reinterpret_cast<uint2*>(codes)[b] = code;
    sf[mma_offset(r, kb, kbt)] = (uint8_t)sc;
    r += dr;
    kb += dkb;
    if (kb >= KB) {
      kb -= KB;
      ++r;
    }
  }
  // the layout's padding: rows [M, roundup(M, 128)) and blocks [KB, roundup(KB, 4)) of the others
  const int64_t Mp = (M + 127) / 128 * 128, KBp = kbt * 4;
  const int64_t npad = Mp * KBp - M * KB;
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < npad; p += (int64_t)gridDim.x * blockDim.x) {
    int64_t r, kb;
    const int64_t tail = M * (KBp - KB);  // padding blocks of the real rows
    if (p < tail) {
      r = p / (KBp - KB);
      kb = KB + (p - r * (KBp - KB));
    } else {
      const int64_t q = p - tail;
      r = M + q / KBp;
      kb = q - (r - M) * KBp;
    }
    sf[mma_offset(r, kb, kbt)] = 0;
  }
}

int act_ctas() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n * kActCtasPerSm;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace nvfp4

extern "C" {

size_t nvfp4_act_quant_workspace_bytes(void) {
  const int n = nvfp4::act_ctas();
  return n > 0 ? ((size_t)n * sizeof(float) + 255) / 256 * 256 : 0;
}

nvfp4_status nvfp4_act_quant_mma(const void* x, int64_t M, int64_t K, int use_rht, uint32_t signs, uint8_t* codes,
                                 uint8_t* scales_mma, float* tensor_scale, int* dev_status, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (M < 1 || K < 16 || (K % 16) != 0) return NVFP4_ESHAPE;
  if (K > ((int64_t)1 << 46) / M) return NVFP4_ESHAPE;
  if (use_rht != 0 && use_rht != 1) return NVFP4_EINVAL;
  if (signs > 0xFFFFu) return NVFP4_EINVAL;
  if (!x || !codes || !scales_mma || !tensor_scale) return NVFP4_EINVAL;
  if (!nvfp4::aligned_to(x, 32) || !nvfp4::aligned_to(codes, 16) || !nvfp4::aligned_to(scales_mma, 16) ||
      !nvfp4::aligned_to(tensor_scale, 4) || !nvfp4::aligned_to(dev_status, 4))
    return NVFP4_EALIGN;
  const int ctas = nvfp4::act_ctas();
  if (ctas <= 0) return NVFP4_ECUDA;
  if (!workspace || !nvfp4::aligned_to(workspace, 256) || workspace_bytes < nvfp4_act_quant_workspace_bytes())
    return NVFP4_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  float* part = static_cast<float*>(workspace);
  const int64_t KB = K / 16, nb = M * KB;
  if (use_rht) {
    nvfp4::act_amax_kernel<true><<<ctas, nvfp4::kActThreads, 0, s>>>(xb, nb, signs, part);
    nvfp4::act_quant_kernel<true><<<ctas / 4 * 3, nvfp4::kActThreads, 0, s>>>(xb, M, KB, signs, part, ctas, codes,
                                                                              scales_mma, tensor_scale, dev_status);
  } else {
    nvfp4::act_amax_kernel<false><<<ctas, nvfp4::kActThreads, 0, s>>>(xb, nb, signs, part);
    nvfp4::act_quant_kernel<false><<<ctas / 4 * 3, nvfp4::kActThreads, 0, s>>>(xb, M, KB, signs, part, ctas, codes,
                                                                               scales_mma, tensor_scale, dev_status);
  }
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

}  // extern "C"
