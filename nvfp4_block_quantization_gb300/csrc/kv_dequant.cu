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

cudaError_t launch_kv_dequant(const uint8_t* codes, const uint8_t* scales, const float* g, const float* mean,
                              int64_t tpg, int64_t T, int C, void* out, int ctas, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  kv_dequant_kernel<<<ctas, 256, 0, s>>>(codes, scales, g, mean, tpg, T, C, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace nvfp4
