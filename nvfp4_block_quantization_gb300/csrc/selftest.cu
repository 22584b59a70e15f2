// selftest.cu -- exposes the conversion instructions of the quantizers (sm_103a)
// so that a test can compare them with a software statement of the formats.
//
// The quantizers round with cvt.rn.satfinite.e2m1x2.f32 (E2M1 codes) and
// cvt.rn.satfinite.e4m3x2.f32 (E4M3 block scales) and decode with
// cvt.rn.f16x2.e2m1x2 and cvt.rn.f16x2.e4m3x2; this kernel runs exactly those
// wrappers (common.cuh) on caller-provided values.
#include "nvfp4.h"
#include "common.cuh"

namespace nvfp4 {
namespace {

__global__ void __launch_bounds__(256) selftest_cvt_kernel(const float* __restrict__ x, int64_t n,
                                                           uint8_t* __restrict__ e2m1, uint16_t* __restrict__ e4m3,
                                                           uint32_t* __restrict__ e2m1_dec, float* __restrict__ e4m3_val) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float v = x[i];
    e2m1[i] = (uint8_t)e2m1x2(v, v);    // both lanes of the paired conversion
    e4m3[i] = (uint16_t)e4m3x2(v, v);
  }
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < 256) {
    e2m1_dec[t] = e2m1x2_to_f16x2((uint32_t)t);
    e4m3_val[t] = e4m3_value((uint32_t)t);
  }
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_selftest_cvt(const float* x, int64_t n, uint8_t* e2m1_codes, uint16_t* e4m3_codes,
                                           uint32_t* e2m1_pair_f16x2, float* e4m3_values, void* stream) {
  if (n < 0) return NVFP4_ESHAPE;
  if (!e2m1_pair_f16x2 || !e4m3_values || (n > 0 && (!x || !e2m1_codes || !e4m3_codes))) return NVFP4_EINVAL;
  if ((reinterpret_cast<uintptr_t>(x) % 4) || (reinterpret_cast<uintptr_t>(e4m3_codes) % 2) ||
      (reinterpret_cast<uintptr_t>(e2m1_pair_f16x2) % 4) || (reinterpret_cast<uintptr_t>(e4m3_values) % 4))
    return NVFP4_EALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return NVFP4_ECUDA;
  const int64_t want = (n + 255) / 256;
  const int grid = (int)(want < 1 ? 1 : (want > (int64_t)sms * 8 ? (int64_t)sms * 8 : want));
  nvfp4::selftest_cvt_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, n, e2m1_codes, e4m3_codes,
                                                                                   e2m1_pair_f16x2, e4m3_values);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}
