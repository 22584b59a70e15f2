// rht16.cuh -- the random Hadamard transform of one 16-element block, shared by
// the standalone transform and the fused activation quantizer (sm_103a).
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page), training step 4: random Hadamard transforms against outliers
// in the NVFP4 GEMM path.  y = (x D) H / 4: element i negated where bit i of
// `signs` is set, then the radix-2 Walsh-Hadamard butterflies with strides 1, 2,
// 4, 8 (each pair (a, b) -> (fl(a + b), fl(a - b))), then the exact * 1/4.
#pragma once

#include <cstdint>

namespace nvfp4 {

__device__ __forceinline__ void rht16_block(float v[16], uint32_t signs) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if ((signs >> i) & 1u) v[i] = -v[i];
#pragma unroll
  for (int h = 1; h < 16; h <<= 1)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if ((i & h) == 0) {
        const float a = v[i], c = v[i + h];
        v[i] = __fadd_rn(a, c);
        v[i + h] = __fsub_rn(a, c);
      }
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], 0.25f);
}

}  // namespace nvfp4
