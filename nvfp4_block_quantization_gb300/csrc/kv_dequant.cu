// kv_dequant.cu -- NVFP4 KV-cache read: codes + E4M3 scales + per-group tensor
// scale (and optionally the smoothing mean) back to bf16 (sm_103a).
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page), inference steps 7 and 9: the NVFP4 KV cache written per chunk
// is read back by attention over the global sink, shot sink and rolling frames.
// Each token t uses the tensor scale (and mean) of its group t / tokens_per_group,
// so a cache assembled from frames of different chunks dequantizes in one pass.
#include "common.cuh"
#include "kv_kernels.cuh"

namespace nvfp4 {

// Empty chunk: nothing to quantize; the tensor scale and the mean are 0.
__global__ void kv_empty_kernel(const __grid_constant__ KvBatch b, int C, int* dev_status, int first_launch) {
  const KvJob& J = b.job[blockIdx.x];
  for (int c = threadIdx.x; c < C; c += blockDim.x)
    if (J.mean_out) J.mean_out[c] = J.mean_in ? J.mean_in[c] : 0.0f;
  if (threadIdx.x == 0) {
    *J.tensor_scale = 0.0f;
    if (blockIdx.x == 0 && dev_status && first_launch) *dev_status = 0;
  }
}

cudaError_t launch_kv_empty(const KvBatch& b, int C, int* dev_status, int first_launch, cudaStream_t s) {
  kv_empty_kernel<<<b.n, 256, 0, s>>>(b, C, dev_status, first_launch);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- dequant
//
// Launch: grid (gx, gy), CTAs of cw * rpp threads.  Thread (c, r) owns block
// column blockIdx.x * cw + c (16 channels) of the contiguous row range
// [blockIdx.y * R, (blockIdx.y + 1) * R), rows r, r + rpp, ...; its group's
// tensor scale and 16 means stay in registers and are reloaded only when a row
// crosses into the next group.  Codes and scale bytes of kAhead rows are loaded
// before any of them is expanded; a warp reads 256 contiguous code bytes and 32
// scale bytes per row and writes 1 KB of bf16 contiguously (one 32-byte store
// per thread when the output is 32-byte aligned).
constexpr int kAhead = 4;

// One 32-byte streaming store (the address must be 32-byte aligned); the output
// is not read again by this pass.
__device__ __forceinline__ void st_v8(void* p, const uint32_t w[8]) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

template <bool kMean, bool kWide>
__global__ void __launch_bounds__(256) kv_dequant_kernel(const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ scales,
                                                         const float* __restrict__ tensor_scale,
                                                         const float* __restrict__ mean, int64_t tpg, int64_t T,
                                                         int C, int cw, int rpp, int64_t rows_per_cta,
                                                         __nv_bfloat16* __restrict__ out) {
  const int nbr = C / 16;
  const int c = threadIdx.x % cw, rl = threadIdx.x / cw;
  const int cb = blockIdx.x * cw + c;
  if (cb >= nbr || rl >= rpp) return;
  const int64_t ra = (int64_t)blockIdx.y * rows_per_cta;
  const int64_t rb = ra + rows_per_cta < T ? ra + rows_per_cta : T;
  const uint2* c8 = reinterpret_cast<const uint2*>(codes) + cb;
  const uint8_t* s8 = scales + cb;
  uint4* o = reinterpret_cast<uint4*>(out + (size_t)cb * 16);
  const size_t orow = (size_t)C / 8;  // uint4 per output row
  int64_t gend = -1;                  // first row of the next group
  float g = 0.0f, mu[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) mu[i] = 0.0f;
  for (int64_t r = ra + rl; r < rb; r += (int64_t)kAhead * rpp) {
    uint2 cwd[kAhead];
    uint32_t sc[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int64_t row = r + (int64_t)u * rpp;
      if (row < rb) {
        cwd[u] = __ldg(c8 + (size_t)row * nbr);
        sc[u] = __ldg(s8 + (size_t)row * nbr);
      }
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int64_t row = r + (int64_t)u * rpp;
      if (row >= rb) break;
      if (row >= gend) {  // entering a new group (rare): its tensor scale and means
        const int64_t grp = row / tpg;
        gend = (grp + 1) * tpg;
        g = __ldg(tensor_scale + grp);
        if (kMean) {  // four 16-byte loads when aligned (the API requires only 4 bytes)
          const float* m = mean + (size_t)grp * C + (size_t)cb * 16;
          if ((reinterpret_cast<uintptr_t>(m) & 15) == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 v = __ldg(reinterpret_cast<const float4*>(m) + i);
              mu[4 * i] = v.x; mu[4 * i + 1] = v.y; mu[4 * i + 2] = v.z; mu[4 * i + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) mu[i] = __ldg(m + i);
          }
        }
      }
      const float S = __fmul_rn(e4m3_value(sc[u]), g);
      uint32_t w[8];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const uint32_t byte = ((p < 4 ? cwd[u].x : cwd[u].y) >> (8 * (p & 3))) & 0xFFu;
        const uint32_t q = e2m1x2_to_f16x2(byte);
        float v0 = __fmul_rn(f16lo(q), S);
        float v1 = __fmul_rn(f16hi(q), S);
        if (kMean) {
          v0 = __fadd_rn(v0, mu[2 * p]);
          v1 = __fadd_rn(v1, mu[2 * p + 1]);
        }
        __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
        w[p] = *reinterpret_cast<uint32_t*>(&h);
      }
      uint4* dst = o + (size_t)row * orow;
      if (kWide) {
        st_v8(dst, w);
      } else {
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
  }
}

cudaError_t launch_kv_dequant(const uint8_t* codes, const uint8_t* scales, const float* g, const float* mean,
                              int64_t tpg, int64_t T, int C, void* out, int sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int nbr = C / 16;
  const int cw = nbr < 256 ? nbr : 256;
  const int rpp = 256 / cw;
  const int gx = (nbr + cw - 1) / cw;
  // CTAs over contiguous row ranges, 32 per SM in total (16 when the means are
  // re-added: each CTA loads its group's 16 means per thread at start, so fewer,
  // longer CTAs do better); measured on the 21-frame cache
  const int per_sm = mean ? 16 : 32;
  int64_t gy = ((int64_t)per_sm * (sms > 0 ? sms : 1) + gx - 1) / gx;
  const int64_t max_gy = (T + rpp - 1) / rpp;
  if (gy > max_gy) gy = max_gy;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  const int64_t rows_per_cta = (T + gy - 1) / gy;
  gy = (T + rows_per_cta - 1) / rows_per_cta;
  const dim3 grid(gx, (unsigned)gy);
  const dim3 block(cw * rpp);
  auto* o = static_cast<__nv_bfloat16*>(out);
  const bool wide = (reinterpret_cast<uintptr_t>(out) % 32) == 0;
  if (mean && wide)
    kv_dequant_kernel<true, true><<<grid, block, 0, s>>>(codes, scales, g, mean, tpg, T, C, cw, rpp, rows_per_cta, o);
  else if (mean)
    kv_dequant_kernel<true, false><<<grid, block, 0, s>>>(codes, scales, g, mean, tpg, T, C, cw, rpp, rows_per_cta, o);
  else if (wide)
    kv_dequant_kernel<false, true><<<grid, block, 0, s>>>(codes, scales, g, mean, tpg, T, C, cw, rpp, rows_per_cta, o);
  else
    kv_dequant_kernel<false, false><<<grid, block, 0, s>>>(codes, scales, g, mean, tpg, T, C, cw, rpp, rows_per_cta, o);
  return cudaGetLastError();
}

}  // namespace nvfp4
