// kv_exchange.cu -- packing an NVFP4 KV-cache tensor into per-rank head shards
// for a sequence-parallel exchange, and unpacking them (sm_103a).
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page): under Ulysses sequence parallelism an all-to-all moves
// attention inputs between a sequence split and a head split, and the page
// credits the 4-bit KV cache with the time saved at SP = 2 and 4 (the
// "weaknesses" item on Table 6), i.e. with moving packed NVFP4 instead of bf16.
// Here a rank's quantized tensor [T][H][..] (codes, E4M3 scales, its tensor
// scale and, for smoothed K, its mean) is cut into P head shards of H / P heads,
// each laid out as one contiguous segment, so that one all-to-all of equal
// segments moves shard p to rank p:
//   [16 B: tensor scale g, fp32, then zeros]
//   [mean of the shard's heads, (H / P) * D fp32]       (only with a mean)
//   [codes, T * (H / P) * D / 2 bytes]                  (padded to 16 B)
//   [scales, T * (H / P) * D / 16 bytes]                (padded to 16 B)
// Unpacking P received segments (segment r from rank r, holding that rank's
// T_r = T tokens) stacks them along the token axis: [P * T][H / P][..], with
// one tensor scale (and mean) per source rank, which is how the cache read
// (nvfp4_kv_dequant with tokens_per_group = T) takes per-group scales.
#include "nvfp4.h"
#include "kv_kernels.cuh"

namespace nvfp4 {
namespace {

size_t pad16(size_t v) { return (v + 15) / 16 * 16; }

struct ShardGeo {
  int64_t T;
  int H, D, P, hs;
  size_t mean_bytes, code_bytes, scale_bytes, seg_bytes;
};

ShardGeo shard_geo(int64_t T, int H, int D, int P, bool with_mean) {
  ShardGeo s;
  s.T = T;
  s.H = H;
  s.D = D;
  s.P = P;
  s.hs = H / P;
  s.mean_bytes = with_mean ? (size_t)s.hs * D * 4 : 0;
  s.code_bytes = pad16((size_t)T * s.hs * D / 2);
  s.scale_bytes = pad16((size_t)T * s.hs * D / 16);
  s.seg_bytes = 16 + s.mean_bytes + s.code_bytes + s.scale_bytes;
  return s;
}

bool shard_ok(int64_t T, int H, int D, int P) {
  return T >= 0 && T <= ((int64_t)1 << 30) && H >= 1 && D >= 16 && D % 16 == 0 && P >= 1 && H % P == 0 &&
         (int64_t)H * D <= (1 << 24);
}

// Copies n bytes (n a multiple of 8, both pointers 8-byte aligned) or, when not,
// byte by byte.
__device__ __forceinline__ void copy_bytes(uint8_t* dst, const uint8_t* src, int n) {
  if ((n & 7) == 0 && ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 7) == 0) {
    for (int i = 0; i < n; i += 8) *reinterpret_cast<uint2*>(dst + i) = *reinterpret_cast<const uint2*>(src + i);
  } else {
    for (int i = 0; i < n; ++i) dst[i] = src[i];
  }
}

// One thread per (shard p, token t, head within the shard h): that row's codes and scales.
// pack = 1: tensor rows -> segments; pack = 0: segments -> stacked rows.
__global__ void __launch_bounds__(256) shard_rows_kernel(uint8_t* codes, uint8_t* scales, uint8_t* seg, ShardGeo s,
                                                         int pack) {
  const int64_t rows = (int64_t)s.P * s.T * s.hs;
  const int cb = s.D / 2, sb = s.D / 16;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows; i += (int64_t)gridDim.x * blockDim.x) {
    const int h = (int)(i % s.hs);
    const int64_t t = (i / s.hs) % s.T;
    const int p = (int)(i / ((int64_t)s.hs * s.T));
    uint8_t* base = seg + (size_t)p * s.seg_bytes + 16 + s.mean_bytes;
    uint8_t* sc = base + (size_t)(t * s.hs + h) * cb;
    uint8_t* ss = base + s.code_bytes + (size_t)(t * s.hs + h) * sb;
    if (pack) {
      // source row: token t, head p * hs + h of the [T][H] tensor
      const size_t r = (size_t)t * s.H + (size_t)p * s.hs + h;
      copy_bytes(sc, codes + r * cb, cb);
      copy_bytes(ss, scales + r * sb, sb);
    } else {
      // destination row: token p * T + t of the stacked [P T][hs] tensor
      const size_t r = ((size_t)p * s.T + t) * s.hs + h;
      copy_bytes(codes + r * cb, sc, cb);
      copy_bytes(scales + r * sb, ss, sb);
    }
  }
}

// Tensor scales and means: one CTA per shard.
__global__ void shard_meta_kernel(float* g, float* mean, uint8_t* seg, ShardGeo s, int pack) {
  const int p = blockIdx.x;
  uint8_t* base = seg + (size_t)p * s.seg_bytes;
  float* sg = reinterpret_cast<float*>(base);
  float* sm = reinterpret_cast<float*>(base + 16);
  const int n = s.hs * s.D;
  if (pack) {
    if (threadIdx.x < 4) sg[threadIdx.x] = threadIdx.x == 0 ? *g : 0.0f;
    if (mean)
      for (int i = threadIdx.x; i < n; i += blockDim.x) sm[i] = mean[(size_t)p * n + i];
  } else {
    if (threadIdx.x == 0) g[p] = sg[0];
    if (mean)
      for (int i = threadIdx.x; i < n; i += blockDim.x) mean[(size_t)p * n + i] = sm[i];
  }
}

cudaError_t launch_shards(uint8_t* codes, uint8_t* scales, float* g, float* mean, uint8_t* seg, const ShardGeo& s,
                          int pack, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t rows = (int64_t)s.P * s.T * s.hs;
  if (rows > 0) {
    const int64_t want = (rows + 255) / 256;
    const int grid = (int)(want > (int64_t)sms * 16 ? (int64_t)sms * 16 : want);
    shard_rows_kernel<<<grid, 256, 0, st>>>(codes, scales, seg, s, pack);
  }
  shard_meta_kernel<<<s.P, 256, 0, st>>>(g, mean, seg, s, pack);
  return cudaGetLastError();
}

}  // namespace
}  // namespace nvfp4

extern "C" {

size_t nvfp4_kv_shard_bytes(int64_t T, int H, int D, int P, int with_mean) {
  if (!nvfp4::shard_ok(T, H, D, P)) return 0;
  return nvfp4::shard_geo(T, H, D, P, with_mean != 0).seg_bytes;
}

nvfp4_status nvfp4_kv_pack_head_shards(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                                       const float* mean, int64_t T, int H, int D, int P, void* out, void* stream) {
  if (!nvfp4::shard_ok(T, H, D, P)) return NVFP4_ESHAPE;
  if (!tensor_scale || !out || (T > 0 && (!codes || !scales))) return NVFP4_EINVAL;
  if ((reinterpret_cast<uintptr_t>(out) % 16) || (reinterpret_cast<uintptr_t>(tensor_scale) % 4) ||
      (reinterpret_cast<uintptr_t>(mean) % 4))
    return NVFP4_EALIGN;
  const nvfp4::ShardGeo s = nvfp4::shard_geo(T, H, D, P, mean != nullptr);
  cudaError_t e = nvfp4::launch_shards(const_cast<uint8_t*>(codes), const_cast<uint8_t*>(scales),
                                       const_cast<float*>(tensor_scale), const_cast<float*>(mean),
                                       static_cast<uint8_t*>(out), s, 1, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

nvfp4_status nvfp4_kv_unpack_head_shards(const void* in, int64_t T, int H, int D, int P, int with_mean,
                                         uint8_t* codes, uint8_t* scales, float* tensor_scales, float* means,
                                         void* stream) {
  if (!nvfp4::shard_ok(T, H, D, P)) return NVFP4_ESHAPE;
  if (!in || !tensor_scales || (T > 0 && (!codes || !scales)) || (with_mean != 0) != (means != nullptr))
    return NVFP4_EINVAL;
  if ((reinterpret_cast<uintptr_t>(in) % 16) || (reinterpret_cast<uintptr_t>(tensor_scales) % 4) ||
      (reinterpret_cast<uintptr_t>(means) % 4))
    return NVFP4_EALIGN;
  const nvfp4::ShardGeo s = nvfp4::shard_geo(T, H, D, P, with_mean != 0);
  cudaError_t e = nvfp4::launch_shards(codes, scales, tensor_scales, means,
                                       const_cast<uint8_t*>(static_cast<const uint8_t*>(in)), s, 0,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

}  // extern "C"
