// common.cuh -- device helpers shared by the NVFP4 kernels (sm_103a).
//
// Conversions use the Blackwell cvt instructions; their rounding (round to
// nearest even, saturation to the largest finite value, sign of zero kept)
// and lane order (first operand -> high nibble/byte) were checked on GB300
// against a software statement of the formats over every non-NaN fp32 input.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace nvfp4 {

constexpr float kTensorDenom = 2688.0f;  // 6 (largest E2M1) * 448 (largest E4M3)

// Two fp32 values -> one byte of two E2M1 codes: `lo` in bits 0..3, `hi` in bits 4..7.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u16.u8 %0, t; }" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One byte of two E2M1 codes -> their values as f16x2 (low half = low nibble).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t h;
  uint16_t b = (uint16_t)byte;
  asm("{ .reg .b8 t; cvt.u8.u16 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h) : "h"(b));
  return h;
}

// Two fp32 values -> two E4M3 bytes: `lo` in bits 0..7, `hi` in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Value of one E4M3 byte (0x7F/0xFF decode to NaN).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h;
  uint16_t c = (uint16_t)(code & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(c));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

__device__ __forceinline__ float f16lo(uint32_t h2) { return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))); }
__device__ __forceinline__ float f16hi(uint32_t h2) { return __half2float(__ushort_as_half((unsigned short)(h2 >> 16))); }

// bf16 pair (one 32-bit word) -> two fp32 (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max that propagates NaN (a NaN anywhere makes the result NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float min_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ bool finite_f(float x) { return fabsf(x) <= 3.402823466e38f; }

// Error-free transformation of an addition (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bp = __fsub_rn(s, a);
  float ap = __fsub_rn(s, bp);
  e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

// Per-tensor constants of the Four-Over-Six quantizer plus the candidate
// table indexed by E4M3 code: inv[e] = fl(1 / fl(E * g)) when usable, else 0;
// e2[e] = E * E.
struct QuantTable {
  float inv[128];
  float e2[128];
};

// Fills `tab` (shared memory) with threads [0, 128) of the block; the caller
// synchronizes afterwards.
__device__ __forceinline__ void build_table(QuantTable* tab, float g) {
  int e = threadIdx.x;
  if (e < 128) {
    float E = e4m3_value((uint32_t)e);  // code 127 -> NaN -> unusable
    float S = __fmul_rn(E, g);
    float inv = __frcp_rn(S);
    bool ok = (E > 0.0f) && (S > 0.0f) && finite_f(inv);
    tab->inv[e] = ok ? inv : 0.0f;
    tab->e2[e] = ok ? __fmul_rn(E, E) : 0.0f;
  }
}

}  // namespace nvfp4
