// w2d_kernels.cu -- NVFP4 weight quantizer with 16x16 2-D blocks (sm_103a).
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page), training pipeline step 4: weights carry 2-D block scales.
// Each 16x16 tile gets one E4M3 scale chosen by Four-Over-Six; the tile's error
// accumulates its 256 squared errors in row-major order.
//
//   w2d_amax       per-CTA absolute maximum (NaN-propagating) over each matrix.
//   w2d_amax_seq   (batched calls) every CTA takes its slice of each matrix in
//                  turn and publishes that matrix's amax once all CTAs have
//                  folded theirs in, so quantization of the first matrices
//                  overlaps the amax pass over the later ones.
//   w2d_quant      two threads per tile: tile amax, both candidates' errors,
//                  the choice, then the chosen codes.
#include "bulk.cuh"
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

// The job of CTA `bx` in a launch that gives job j the CTAs [begin_j, begin_j + n_j).
__device__ __forceinline__ int w2d_job_of(const W2dBatch& b, int bx, bool quant) {
  int j = 0;
  while (j + 1 < b.n && bx >= (quant ? b.job[j + 1].quant_begin : b.job[j + 1].amax_begin)) ++j;
  return j;
}

// NaN-propagating maximum over the block's threads; the result is valid in
// thread 0.  `red` holds one value per warp.
__device__ __forceinline__ float block_max_nan(float m, float* red) {
  for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
  }
  return m;
}

// Absolute maximum (NaN-propagating) of the 16-byte chunks [a, b) of one matrix,
// eight loads in flight per thread; the result is valid in thread 0.
template <bool kBF16>
__device__ __forceinline__ float range_amax(const uint4* p, int64_t a, int64_t b, float* red) {
  constexpr int U = 8;
  uint32_t mw = 0u;  // bf16: max of |x| pairs
  float mf = 0.0f;   // fp32
  for (int64_t i = a + threadIdx.x; i < b; i += (int64_t)U * blockDim.x) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = i + (int64_t)u * blockDim.x < b ? ld_nc_v4(p + i + (int64_t)u * blockDim.x)
                                                                        : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (kBF16) {
        mw = bf16x2_max_nan(mw, bf16x2_max_nan(v[u].x & 0x7fff7fffu, v[u].y & 0x7fff7fffu));
        mw = bf16x2_max_nan(mw, bf16x2_max_nan(v[u].z & 0x7fff7fffu, v[u].w & 0x7fff7fffu));
      } else {
        mf = max_nan(mf, max_nan(max_nan(fabsf(__uint_as_float(v[u].x)), fabsf(__uint_as_float(v[u].y))),
                                 max_nan(fabsf(__uint_as_float(v[u].z)), fabsf(__uint_as_float(v[u].w)))));
      }
    }
  }
  return block_max_nan(kBF16 ? max_nan(bf16lo(mw), bf16hi(mw)) : mf, red);
}

// Absolute maximum (NaN-propagating) of each matrix, per CTA: CTA c of job j
// reads the contiguous range of 16-byte chunks [c n / k, (c + 1) n / k) of the
// job's k CTAs with 8 loads in flight per thread; the partial goes to
// amax_part[blockIdx.x] (a job's partials are contiguous).
template <bool kBF16>
__global__ void __launch_bounds__(256) w2d_amax_kernel(const __grid_constant__ W2dBatch bt, float* amax_part,
                                                       int* dev_status) {
  __shared__ float red[32];
  if (blockIdx.x == 0 && threadIdx.x == 0 && dev_status && bt.reset_status) *dev_status = 0;
  const W2dJob& J = bt.job[w2d_job_of(bt, blockIdx.x, false)];
  const int lc = blockIdx.x - J.amax_begin;
  const int64_t nv = J.M * J.N / 16 * (kBF16 ? 2 : 4);  // 16-byte chunks
  const int64_t a = (int64_t)lc * nv / J.amax_ctas, b = (int64_t)(lc + 1) * nv / J.amax_ctas;
  const float m = range_amax<kBF16>(static_cast<const uint4*>(J.w), a, b, red);
  if (threadIdx.x == 0) amax_part[blockIdx.x] = m;
}

// Batched amax, one matrix after another: CTA c of the grid folds the chunks
// [c n / P, (c + 1) n / P) of each matrix into the matrix's amax word
// (ctr[1 + 2 j], the bits of |x|: as unsigned integers they order like the
// values, NaN above every number) and then counts itself on the matrix's ready
// word (ctr[2 + 2 j], release).  The quantization grid may start at once.
template <bool kBF16>
__global__ void __launch_bounds__(256) w2d_amax_seq_kernel(const __grid_constant__ W2dBatch bt, unsigned* ctr,
                                                           int* dev_status) {
  __shared__ float red[32];
  if (blockIdx.x == 0 && threadIdx.x == 0 && dev_status && bt.reset_status) *dev_status = 0;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int j = 0; j < bt.n; ++j) {
    const W2dJob& J = bt.job[j];
    const int64_t nv = J.M * J.N / 16 * (kBF16 ? 2 : 4);  // 16-byte chunks
    const int64_t a = (int64_t)blockIdx.x * nv / gridDim.x, b = (int64_t)(blockIdx.x + 1) * nv / gridDim.x;
    const float m = range_amax<kBF16>(static_cast<const uint4*>(J.w), a, b, red);
    if (threadIdx.x == 0) {
      atomicMax(ctr + 1 + 2 * j, __float_as_uint(m) & 0x7fffffffu);
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr + 2 + 2 * j) : "memory");
    }
    __syncthreads();  // red is reused by the next matrix
  }
}

// Quantization: two threads per 16x16 tile (lanes 2p and 2p + 1 of a warp), one
// per candidate (even lane: scale mapping the tile amax to 6, odd lane: to 4).
// Each finds the tile amax (rows 0-7 / 8-15, combined with its partner), picks
// its candidate's E4M3 scale, and quantizes the whole tile under it, keeping
// the 256 codes in registers and the error as one fused multiply-add per
// element in row-major order.  The pair then compares errors (lower wins, ties
// to 6) and the winner stores its codes and the scale byte.  A warp covers 16
// adjacent tiles: 512 contiguous bytes of every tile row.
// kSeq (overlapped batched launch): thread 0 waits (bounded) until the job's
// ready word counts every amax CTA, and the amax is the job's amax word; once
// every CTA has read what it needs, the last of them returns ctr to zero.
template <bool kBF16, bool kSeq>
__global__ void __launch_bounds__(256) w2d_quant_kernel(const __grid_constant__ W2dBatch bt, const float* amax_part,
                                                        unsigned* ctr, int* dev_status) {
  __shared__ QuantTable tab;
  __shared__ float red[32];
  const int jb = w2d_job_of(bt, blockIdx.x, true);
  const W2dJob& J = bt.job[jb];
  const void* w = J.w;
  const int64_t M = J.M, N = J.N;
  uint8_t* codes = J.codes;
  uint8_t* scales = J.scales;
  const int lq = blockIdx.x - J.quant_begin;  // this CTA within the job's CTAs
  if (kSeq) {
    if (threadIdx.x == 0) {
      const uint64_t t0 = bulk_timer_ns();
      bool ok = true;
      for (unsigned it = 0; ld_acquire_u32(ctr + 2 + 2 * jb) < (unsigned)bt.amax_grid; ++it) {
        if (bulk_timer_ns() - t0 > kBulkWaitNs) {
          ok = false;
          if (dev_status) atomicOr(dev_status, NVFP4_DEV_TIMEOUT_FLAG);
          break;
        }
        __nanosleep(it < 8 ? 128 : 512);
      }
      red[0] = ok ? __uint_as_float(*reinterpret_cast<volatile const unsigned*>(ctr + 1 + 2 * jb))
                  : __int_as_float(0x7fc00000);
    }
  } else {
    float m = 0.0f;
    for (int i = threadIdx.x; i < J.amax_ctas; i += blockDim.x) m = max_nan(m, amax_part[J.amax_begin + i]);
    m = block_max_nan(m, red);
    __syncthreads();
    if (threadIdx.x == 0) red[0] = m;
  }
  __syncthreads();
  const float amax = red[0];
  const bool nonfinite = !finite_f(amax);
  const float g = nonfinite ? __int_as_float(0x7fc00000) : __fdiv_rn(amax, kTensorDenom);
  const int half = threadIdx.x & 1;  // 0: candidate 6, 1: candidate 4
  const float kM = __frcp_rn(__fmul_rn(half ? 4.0f : 6.0f, g));
  build_table(&tab, g);
  __syncthreads();
  if (lq == 0 && threadIdx.x == 0) {
    *J.tensor_scale = g;
    if (nonfinite && dev_status) atomicOr(dev_status, NVFP4_DEV_NONFINITE_FLAG);
  }
  if (kSeq && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ctr, 1u) + 1u == gridDim.x) {  // every CTA has read its amax word
      __threadfence();
      for (int j = 0; j < bt.n; ++j) {
        ctr[1 + 2 * j] = 0u;
        ctr[2 + 2 * j] = 0u;
      }
      ctr[0] = 0u;
    }
  }

  const unsigned pair_mask = 3u << (threadIdx.x & 30);
  const int64_t TN = N / 16;
  const int64_t ntiles = (M / 16) * TN;
  const int64_t npairs = (int64_t)J.quant_ctas * (blockDim.x / 2);
  for (int64_t tl = ((int64_t)lq * blockDim.x + threadIdx.x) / 2; tl < ntiles; tl += npairs) {
    const int64_t ti = tl / TN, tj = tl - ti * TN;
    const int64_t base = ti * 16 * N + tj * 16;
    // tile amax: this lane's 8 rows, then the partner's
    float ab = 0.0f;
#pragma unroll 2
    for (int r = 8 * half; r < 8 * half + 8; ++r) {
      float v[16];
      load_row16<kBF16>(w, base + r * N, v);
      ab = max3_abs(ab, max3_abs(max3_abs(v[0], v[1], v[2]), max3_abs(v[3], v[4], v[5]), max3_abs(v[6], v[7], v[8])),
                    max3_abs(max3_abs(v[9], v[10], v[11]), max3_abs(v[12], v[13], v[14]), v[15]));
    }
    ab = fmaxf(ab, __shfl_xor_sync(pair_mask, ab, 1));
    // this lane's candidate
    const uint32_t e = e4m3x2(__fmul_rn(ab, kM), 0.0f) & 0x7Fu;
    const float inv = tab.inv[e];
    uint2 cw[16];
    float acc = 0.0f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float v[16];
      load_row16<kBF16>(w, base + r * N, v);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float y[8];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float2 yy = __fmul2_rn(make_float2(v[8 * h + 2 * p], v[8 * h + 2 * p + 1]), make_float2(inv, inv));
          y[2 * p] = yy.x;
          y[2 * p + 1] = yy.y;
        }
        uint32_t q[4];
        const uint32_t c = e2m1x8(y, q);
        if (h == 0) cw[r].x = c; else cw[r].y = c;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          float d0, d1;
          f16x2_minus(q[p], y[2 * p], y[2 * p + 1], d0, d1);
          acc = __fmaf_rn(d0, d0, acc);
          acc = __fmaf_rn(d1, d1, acc);
        }
      }
    }
    const float err = __fmul_rn(tab.e2[e], acc);
    const bool ok = inv > 0.0f && ab > 0.0f && !nonfinite;
    const float err_o = __shfl_xor_sync(pair_mask, err, 1);
    const bool ok_o = __shfl_xor_sync(pair_mask, ok ? 1 : 0, 1) != 0;
    const bool ok6 = half ? ok_o : ok, ok4 = half ? ok : ok_o;
    const float err6 = half ? err_o : err, err4 = half ? err : err_o;
    const bool pick4 = ok4 && (!ok6 || err4 < err6);
    // the winner writes; with no usable candidate the even lane writes zeros (or the NaN filler)
    const bool writer = half ? pick4 : !pick4;
    if (writer) {
      const bool use = half ? true : ok6;
#pragma unroll
      for (int r = 0; r < 16; ++r)
        reinterpret_cast<uint2*>(codes + (base + r * N) / 2)[0] = use ? cw[r] : make_uint2(0u, 0u);
      scales[tl] = nonfinite ? 0x7Fu : (uint8_t)(use ? e : 0u);
    }
  }
}

// Dequant: thread (c, r) owns 16-column block blockIdx.x * cw + c of the
// contiguous row range [blockIdx.y * R, (blockIdx.y + 1) * R), rows r, r + rpp,
// ...; codes and scale bytes of four rows are fetched ahead and each block's 16
// bf16 values go out in one 32-byte streaming store (two 16-byte stores when the
// output is only 16-byte aligned).
template <bool kWide>
__global__ void __launch_bounds__(256) w2d_dequant_kernel(const uint8_t* __restrict__ codes,
                                                          const uint8_t* __restrict__ scales,
                                                          const float* __restrict__ tensor_scale, int64_t M,
                                                          int64_t N, int cw, int rpp, int64_t rows_per_cta,
                                                          __nv_bfloat16* __restrict__ out) {
  constexpr int kAhead = 4;
  const int64_t nbr = N / 16;
  const int c = threadIdx.x % cw, rl = threadIdx.x / cw;
  const int64_t cb = (int64_t)blockIdx.x * cw + c;
  if (cb >= nbr || rl >= rpp) return;
  const int64_t ra = (int64_t)blockIdx.y * rows_per_cta;
  const int64_t rb = ra + rows_per_cta < M ? ra + rows_per_cta : M;
  const uint2* c8 = reinterpret_cast<const uint2*>(codes) + cb;
  const uint8_t* s8 = scales + cb;
  uint4* o = reinterpret_cast<uint4*>(out + cb * 16);
  const size_t orow = (size_t)N / 8;  // uint4 per output row
  const float g = __ldg(tensor_scale);
  for (int64_t r = ra + rl; r < rb; r += (int64_t)kAhead * rpp) {
    uint2 cwd[kAhead];
    uint32_t sc[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int64_t row = r + (int64_t)u * rpp;
      if (row < rb) {
        cwd[u] = __ldg(c8 + (size_t)row * nbr);
        sc[u] = __ldg(s8 + (size_t)(row / 16) * nbr);
      }
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int64_t row = r + (int64_t)u * rpp;
      if (row >= rb) break;
      const float S = __fmul_rn(e4m3_value(sc[u]), g);
      uint32_t wd[8];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const uint32_t byte = ((p < 4 ? cwd[u].x : cwd[u].y) >> (8 * (p & 3))) & 0xFFu;
        const uint32_t q = e2m1x2_to_f16x2(byte);
        __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(f16lo(q), S), __fmul_rn(f16hi(q), S));
        wd[p] = *reinterpret_cast<uint32_t*>(&h);
      }
      uint4* dst = o + (size_t)row * orow;
      if (kWide) {
        asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(wd[0]), "r"(wd[1]),
                     "r"(wd[2]), "r"(wd[3]), "r"(wd[4]), "r"(wd[5]), "r"(wd[6]), "r"(wd[7])
                     : "memory");
      } else {
        dst[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        dst[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
      }
    }
  }
}

cudaError_t launch_w2d_batch(const W2dBatch& b, bool bf16, int amax_ctas, int quant_ctas, float* amax_part,
                             int* dev_status, cudaStream_t s) {
  if (bf16) w2d_amax_kernel<true><<<amax_ctas, 256, 0, s>>>(b, amax_part, dev_status);
  else w2d_amax_kernel<false><<<amax_ctas, 256, 0, s>>>(b, amax_part, dev_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (bf16) w2d_quant_kernel<true, false><<<quant_ctas, 256, 0, s>>>(b, amax_part, nullptr, dev_status);
  else w2d_quant_kernel<false, false><<<quant_ctas, 256, 0, s>>>(b, amax_part, nullptr, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_w2d_batch_overlapped(const W2dBatch& b, bool bf16, int quant_ctas, unsigned* ctr, int* dev_status,
                                        cudaStream_t s) {
  if (bf16) w2d_amax_seq_kernel<true><<<b.amax_grid, 256, 0, s>>>(b, ctr, dev_status);
  else w2d_amax_seq_kernel<false><<<b.amax_grid, 256, 0, s>>>(b, ctr, dev_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(quant_ctas);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start beside the amax grid
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float* no_part = nullptr;
  if (bf16) return cudaLaunchKernelEx(&cfg, w2d_quant_kernel<true, true>, b, no_part, ctr, dev_status);
  return cudaLaunchKernelEx(&cfg, w2d_quant_kernel<false, true>, b, no_part, ctr, dev_status);
}

cudaError_t launch_w2d_quant(const void* w, bool bf16, const W2dGeom& geo, uint8_t* codes, uint8_t* scales,
                             float* tensor_scale, int* dev_status, float* amax_part, int quant_ctas,
                             cudaStream_t s) {
  W2dBatch b;
  b.n = 1;
  b.reset_status = 1;
  W2dJob& j = b.job[0];
  j.w = w;
  j.M = geo.M;
  j.N = geo.N;
  j.codes = codes;
  j.scales = scales;
  j.tensor_scale = tensor_scale;
  j.amax_begin = 0;
  j.amax_ctas = geo.amax_ctas;
  j.quant_begin = 0;
  j.quant_ctas = quant_ctas;
  return launch_w2d_batch(b, bf16, geo.amax_ctas, quant_ctas, amax_part, dev_status, s);
}

cudaError_t launch_w2d_dequant(const uint8_t* codes, const uint8_t* scales, const float* g, int64_t M, int64_t N,
                               void* out, int sms, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  const int64_t nbr = N / 16;
  const int cw = nbr < 256 ? (int)nbr : 256;
  const int rpp = 256 / cw;
  const int64_t gx = (nbr + cw - 1) / cw;
  int64_t gy = ((int64_t)32 * (sms > 0 ? sms : 1) + gx - 1) / gx;  // 32 CTAs per SM in total
  const int64_t max_gy = (M + rpp - 1) / rpp;
  if (gy > max_gy) gy = max_gy;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  const int64_t rows_per_cta = (M + gy - 1) / gy;
  gy = (M + rows_per_cta - 1) / rows_per_cta;
  const dim3 grid((unsigned)gx, (unsigned)gy), block(cw * rpp);
  auto* o = static_cast<__nv_bfloat16*>(out);
  if ((reinterpret_cast<uintptr_t>(out) % 32) == 0)
    w2d_dequant_kernel<true><<<grid, block, 0, s>>>(codes, scales, g, M, N, cw, rpp, rows_per_cta, o);
  else
    w2d_dequant_kernel<false><<<grid, block, 0, s>>>(codes, scales, g, M, N, cw, rpp, rows_per_cta, o);
  return cudaGetLastError();
}

}  // namespace nvfp4
