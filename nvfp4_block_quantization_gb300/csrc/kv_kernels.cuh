// kv_kernels.cuh -- internal (non-ABI) declarations shared by the kernels and
// the C-ABI layer.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

constexpr int kCTile = 4096;       // channels covered by one stats CTA (8 per thread, <= 512 threads)
constexpr int kMaxJobs = 64;       // tensors per batched launch
constexpr int NVFP4_DEV_NONFINITE_FLAG = 1;

// One tensor of a launch: the caller's pointers plus its workspace slices.
struct KvJob {
  const void* x;
  const float* mean_in;
  float* mean_out;
  uint8_t* codes;
  uint8_t* scales;
  float* tensor_scale;
  float4* part;      // [nchunks][C] {sum, compensation, min, max} (smoothed tensors)
  float* amax_part;  // per-CTA maxima feeding the tensor amax
  float* mean;       // [C] mean used for smoothing
  int smooth;
  int namax;         // number of valid amax_part entries
};

struct KvBatch {
  KvJob job[kMaxJobs];
  int n;
};

// Launch geometry shared by the three kernels.
struct KvGeom {
  int64_t T;
  int C;               // H * D
  int nchunks;         // token chunks of the stats pass
  int rows_per_chunk;
  int nctiles;         // channel tiles of the stats pass
  int ctile_threads;   // threads per stats CTA
  int nfin;            // finalize CTAs (256 channels each)
};

// status_reset (may be NULL) is set to 0 before anything else; status_or (may be NULL) receives flags.
cudaError_t launch_kv_quant(const KvBatch& b, const KvGeom& geo, bool bf16, int* status_reset, int* status_or,
                            int quant_ctas, cudaStream_t s);
cudaError_t launch_kv_dequant(const uint8_t* codes, const uint8_t* scales, const float* g, const float* mean,
                              int64_t tpg, int64_t T, int C, void* out, int ctas, cudaStream_t s);

// 16x16-tile weight quantizer.
struct W2dGeom {
  int64_t M, N;
  int amax_ctas;
};
cudaError_t launch_w2d_quant(const void* w, bool bf16, const W2dGeom& geo, uint8_t* codes, uint8_t* scales,
                             float* tensor_scale, int* dev_status, float* amax_part, int quant_ctas,
                             cudaStream_t s);
cudaError_t launch_w2d_dequant(const uint8_t* codes, const uint8_t* scales, const float* g, int64_t M, int64_t N,
                               void* out, int ctas, cudaStream_t s);

}  // namespace nvfp4
