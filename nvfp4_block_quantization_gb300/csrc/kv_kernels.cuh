// kv_kernels.cuh -- internal (non-ABI) declarations shared by the kernels and
// the C-ABI layer.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

constexpr int kMaxJobs = 64;             // tensors per launch
constexpr int kStatsConsumers = 384;     // statistics consumer threads per CTA, upper bound
constexpr int kStatsStages = 4;          // statistics ring stages
constexpr int kStatsStageBytes = 24576;  // bytes per stage
constexpr int NVFP4_DEV_NONFINITE_FLAG = 1;
constexpr int NVFP4_DEV_TIMEOUT_FLAG = 2;

// One tensor of a launch: the caller's pointers plus its workspace slices.
struct KvJob {
  const void* x;
  const float* mean_in;
  float* mean_out;
  uint8_t* codes;
  uint8_t* scales;
  float* tensor_scale;
  float4* part;   // [P][rpp][C] {sum, low part, min, max} per statistics thread (smoothed tensors)
  float* mean;    // [C] mean used for smoothing
  unsigned* ctr;  // [0] amax bits, [1] statistics CTAs that published their partials, [2] ... that finished the job
  int smooth;
};

struct KvBatch {
  KvJob job[kMaxJobs];
  int n;
};

// Statistics partition: the rows are cut into stages of rows_per_stage rows (a
// multiple of rpp) and CTA c of P takes stages c, c + P, c + 2 P, ...; its
// tpr * rpp consumer threads each own an 8-channel chunk (tpr per row) of every
// rpp-th row.
struct KvGeom {
  int64_t T;
  int C;    // H * D
  int P;    // statistics CTAs (one per SM)
  int tpr;  // threads per row: min(C / 8, kStatsConsumers)
  int rpp;  // rows in parallel: kStatsConsumers / tpr
  int rows_per_stage;
  double inv_T;  // binary64 reciprocal of T: mean = fl32(sum * inv_T)
  float denom;   // tensor scale g = fl(amax / denom): 2688 (6 * 448), or 1792 (4 * 448) with headroom
  unsigned* header;  // [0] quant CTAs finished, [1] status flags
  int* dev_status;
  int first_launch;  // 1: write *dev_status, 0: OR into it
};

// Quantization launch shape: CTAs of cw * rpp threads cover cw block columns of
// rpp rows.  A 1-D grid: first gx * gy_early CTAs for each job but the last (they
// run beside the statistics grid, one per SM in total), then gx * gy_last CTAs
// for the last job (two per SM once the statistics grid has finished).
struct KvQuantShape {
  int cw, rpp, gx, gy_early, gy_last;
  int ctas;  // total CTAs
};

cudaError_t launch_kv_stats(const KvBatch& b, const KvGeom& g, bool bf16, cudaStream_t s);
cudaError_t launch_kv_quant(const KvBatch& b, const KvGeom& g, const KvQuantShape& q, bool bf16, cudaStream_t s);
KvQuantShape kv_quant_shape(int64_t T, int C, int n_jobs, int sms);
cudaError_t launch_kv_empty(const KvBatch& b, int C, int* dev_status, int first_launch, cudaStream_t s);
cudaError_t launch_kv_dequant(const uint8_t* codes, const uint8_t* scales, const float* g, const float* mean,
                              int64_t tpg, int64_t T, int C, void* out, int sms, cudaStream_t s);

// 16x16-tile weight quantizer.
struct W2dGeom {
  int64_t M, N;
  int amax_ctas;
};

// One matrix of a weight launch: its CTAs are [amax_begin, amax_begin + amax_ctas) of
// the amax grid (its partials sit at those indices of the workspace) and
// [quant_begin, quant_begin + quant_ctas) of the quantization grid.
constexpr int kMaxW2dJobs = 64;
struct W2dJob {
  const void* w;
  int64_t M, N;
  uint8_t* codes;
  uint8_t* scales;
  float* tensor_scale;
  int amax_begin, amax_ctas, quant_begin, quant_ctas;
};
struct W2dBatch {
  W2dJob job[kMaxW2dJobs];
  int n;
  int reset_status;  // 1: the launch starts *dev_status at 0 (first launch of a call)
  int amax_grid;     // overlapped launch: CTAs of the amax grid (each covers a slice of every job)
};
cudaError_t launch_w2d_batch(const W2dBatch& b, bool bf16, int amax_ctas, int quant_ctas, float* amax_part,
                             int* dev_status, cudaStream_t s);
// Overlapped launch pair: the amax grid takes the jobs one after another and
// publishes each job's amax as soon as it is complete; the quantization grid
// (a programmatic dependent) starts on a job as soon as its amax is.  ctr holds
// 1 + 2 * kMaxW2dJobs words, zero before the launch and zero again after it.
cudaError_t launch_w2d_batch_overlapped(const W2dBatch& b, bool bf16, int quant_ctas, unsigned* ctr, int* dev_status,
                                        cudaStream_t s);
cudaError_t launch_w2d_quant(const void* w, bool bf16, const W2dGeom& geo, uint8_t* codes, uint8_t* scales,
                             float* tensor_scale, int* dev_status, float* amax_part, int quant_ctas,
                             cudaStream_t s);
cudaError_t launch_w2d_dequant(const uint8_t* codes, const uint8_t* scales, const float* g, int64_t M, int64_t N,
                               void* out, int sms, cudaStream_t s);

}  // namespace nvfp4
