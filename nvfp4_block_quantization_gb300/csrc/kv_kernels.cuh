// kv_kernels.cuh -- internal (non-ABI) declarations shared by the kernels and
// the C-ABI layer.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nvfp4 {

constexpr int kMaxJobs = 64;      // tensors per launch
constexpr int kMaxGroupW = 128;   // channels per statistics group
constexpr int kStatsConsumers = 256;  // statistics threads per CTA (plus one producer warp)
constexpr int kStatsTileRows = 64;
constexpr int kStatsCtasPerSm = 2;
constexpr int NVFP4_DEV_NONFINITE_FLAG = 1;

// One tensor of a launch: the caller's pointers plus its workspace slices.
struct KvJob {
  const void* x;
  const float* mean_in;
  float* mean_out;
  uint8_t* codes;
  uint8_t* scales;
  float* tensor_scale;
  float4* part;   // [P][smax][W] {sum, low part, min, max} per CTA segment (smoothed tensors)
  float* mean;    // [C] mean used for smoothing
  unsigned* ctr;  // [0] amax bits, [1 + k] arrivals at channel group k
  int smooth;
};

struct KvBatch {
  CUtensorMap map[kMaxJobs];  // 2-D TMA map of each job's x[T][C]: box W channels x kStatsTileRows rows
  KvJob job[kMaxJobs];
  int n;
};

// Statistics partition: the ngroups * T (channel group, row) units of a tensor
// are cut into P contiguous ranges, one per statistics CTA.
struct KvGeom {
  int64_t T;
  int64_t U;     // ngroups * T units
  int C;         // H * D
  int W;         // channels per group
  int ngroups;
  int P;         // statistics CTAs per tensor
  int smax;      // row segments per CTA, upper bound
  unsigned* header;  // [0] quant CTAs finished, [1] status flags
  int* dev_status;
  int first_launch;  // 1: write *dev_status, 0: OR into it
};

// Quantization launch shape: CTAs of cw * rpp threads cover cw block columns of
// rpp rows; gx CTAs across the columns, gy down the rows, one z slice per job.
struct KvQuantShape {
  int cw, rpp, gx, gy;
};

cudaError_t launch_kv_stats(const KvBatch& b, const KvGeom& g, bool bf16, cudaStream_t s);
cudaError_t make_tile_map(CUtensorMap* map, const void* x, bool bf16, int64_t T, int C, int W);
cudaError_t launch_kv_quant(const KvBatch& b, const KvGeom& g, const KvQuantShape& q, bool bf16, cudaStream_t s);
KvQuantShape kv_quant_shape(int64_t T, int C, int n_jobs, int sms);
cudaError_t launch_kv_empty(const KvBatch& b, int C, int* dev_status, int first_launch, cudaStream_t s);
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
