// four_over_six.cuh -- the Four-Over-Six block decision shared by the 1-D
// quantization kernels (sm_103a).
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page), "full-stack NVFP4" paragraph: per 16-element block, two FP8
// (E4M3) block-scale candidates map the block's absolute maximum to 6 and to 4;
// the block is quantized to E2M1 under both and the candidate with the lower
// squared error is kept, ties to 6.
#pragma once

#include "common.cuh"

namespace nvfp4 {

// Four-Over-Six on one block z[16].  The two candidates' sequential error
// chains run side by side in one packed f32x2 accumulator (lane x: scale 6,
// lane y: scale 4); each lane is exactly the element-order fused chain
// acc = fma(d, d, acc) of its candidate, d = fl(Q - y) (exact here: y and Q are
// within a factor of two of each other), err = fl(E^2 * acc).
__device__ __forceinline__ void quant_block(const float z[16], const float2* tab, float k6, float k4, bool nonfinite,
                                            uint2& code, uint32_t& sc) {
  const float ma = max3_abs(max3_abs(max3_abs(z[0], z[1], z[2]), max3_abs(z[3], z[4], z[5]), max3_abs(z[6], z[7], z[8])),
                            max3_abs(z[9], z[10], z[11]), max3_abs(max3_abs(z[12], z[13], z[14]), z[15], 0.0f));
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

}  // namespace nvfp4
