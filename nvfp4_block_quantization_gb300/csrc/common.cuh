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
#include <atomic>

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

// max(|a|, |b|, |c|) in one instruction (a NaN operand is ignored).
__device__ __forceinline__ float max3_abs(float a, float b, float c) {
  float r;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ bool finite_f(float x) { return fabsf(x) <= 3.402823466e38f; }

// Lane-wise min / max of two bf16 pairs; a NaN in either input makes that lane NaN.
__device__ __forceinline__ uint32_t bf16x2_min_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

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

// Eight fp32 values -> one word of eight E2M1 codes (byte j = y[2j] low nibble,
// y[2j+1] high nibble) plus the four decoded f16x2 pairs (low half = even element).
__device__ __forceinline__ uint32_t e2m1x8(const float y[8], uint32_t q[4]) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %8, %7;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %10, %9;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %12, %11;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %4, b3;\n\t}"
      : "=r"(w), "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3])
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
  return w;
}

// (Q_lo - y0, Q_hi - y1) for the f16 pair q2: one rounding each (mixed-precision subtract).
// The sign is opposite to y - Q; only the square of the difference is used.
__device__ __forceinline__ void f16x2_minus(uint32_t q2, float y0, float y1, float& d0, float& d1) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "sub.rn.f32.f16 %0, l, %3;\n\tsub.rn.f32.f16 %1, h, %4;\n\t}"
      : "=f"(d0), "=f"(d1) : "r"(q2), "f"(y0), "f"(y1));
}

// fl(x_lo - m0), fl(x_hi - m1) for the bf16 pair w (exact widening, one rounding).
__device__ __forceinline__ void bf16x2_minus(uint32_t w, float m0, float m1, float& z0, float& z1) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "sub.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, h, %4;\n\t}"
      : "=f"(z0), "=f"(z1) : "r"(w), "f"(m0), "f"(m1));
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Named barrier over `n` threads (a multiple of 32) of the block.
__device__ __forceinline__ void named_barrier(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// 32-byte read-only streaming load (no L1 allocation).
__device__ __forceinline__ void ld_nc_v8(const void* p, uint32_t v[8]) {
  asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "l"(p));
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}


// Host: raises kernel `f`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device (a bit of `done` per device id below 64; others every call).
template <typename F>
inline cudaError_t smem_limit_once(F* f, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

}  // namespace nvfp4
