// kv_kernels.cuh -- internal (non-ABI) declarations shared by the kernels and
// the C-ABI layer.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nvfp4 {

constexpr int kMaxJobs = 64;          // tensors per fused launch
constexpr int kFusedStatsWarps = 8;   // warps streaming the statistics pass
constexpr int kFusedQuantWarps = 16;  // warps quantizing (one 16-element block per thread per tile)
constexpr int kFusedMaxW = 128;       // channels per group
constexpr int NVFP4_DEV_NONFINITE_FLAG = 1;

// One tensor of a fused launch: the caller's pointers plus its workspace slices.
struct FusedJob {
  const void* x;
  const float* mean_in;
  float* mean_out;
  uint8_t* codes;
  uint8_t* scales;
  float* tensor_scale;
  float4* part;   // [P][smax][W] {sum, low part, min, max} per CTA segment (smoothed tensors)
  float* mean;    // [C] mean used for smoothing
  unsigned* ctr;  // [0] amax bits, [1] ready count, [2 + k] arrivals at channel group k
  int smooth;
};

struct FusedBatch {
  CUtensorMap map[kMaxJobs];  // 2-D TMA map of each job's x: box W channels x 64 rows
  FusedJob job[kMaxJobs];
  int n;
};

struct FusedGeom {
  int64_t T;
  int64_t U;       // ngroups * T (group, row) units
  int C;           // H * D
  int W;           // channels per group
  int ngroups;
  int P;           // CTAs (all resident)
  int smax;        // row segments per CTA, upper bound
  unsigned spin_limit;
  unsigned* header;  // [0] exit counter, [1] status flags
  int* dev_status;
  int first_launch;  // 1: write *dev_status, 0: OR into it
};

cudaError_t launch_kv_fused(const FusedBatch& b, const FusedGeom& g, bool bf16, cudaStream_t s);
cudaError_t make_tile_map(CUtensorMap* map, const void* x, bool bf16, int64_t T, int C, int W);
int fused_ctas_per_sm(bool bf16);
cudaError_t launch_kv_empty(const FusedBatch& b, int C, int* dev_status, int first_launch, cudaStream_t s);
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
