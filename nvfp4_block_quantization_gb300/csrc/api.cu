// api.cu -- the extern "C" entry points declared in include/nvfp4.h.
//
// Every entry point validates its arguments synchronously (nothing is
// enqueued on an error), carves its workspace, and enqueues the kernels on the
// caller's stream.  No allocation, no synchronization, no printing.
#include <algorithm>
#include <cstring>

#include "nvfp4.h"
#include "kv_kernels.cuh"

namespace {

using namespace nvfp4;

constexpr size_t kWsAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

bool kv_shape_ok(int64_t T, int H, int D) {
  if (T < 0 || H < 1 || D < 16 || (D % 16) != 0) return false;
  const int64_t C = (int64_t)H * D;
  if (C > (1 << 24)) return false;                        // channel indices fit in int with headroom
  if (T > 0 && C > ((int64_t)1 << 46) / T) return false;  // unit arithmetic (units * CTAs) fits in int64
  return true;
}

// Plan of one KV launch pair: statistics partition and the workspace layout.
//   header (256 B): quant CTAs finished, status flags
//   per job: counters (2 words), mean [C], partials [P][rpp][C] float4
struct KvPlan {
  KvGeom geo;
  size_t ctr_bytes, mean_bytes, part_bytes, job_bytes, header_bytes;
};

int stats_ctas() { return device_sms(); }

KvPlan kv_plan(int64_t T, int H, int D, int ctas) {
  KvPlan p;
  std::memset(&p, 0, sizeof(p));
  KvGeom& g = p.geo;
  g.T = T;
  g.C = H * D;
  g.P = std::max(ctas, 1);
  g.tpr = std::min(g.C / 8, kStatsConsumers);
  g.rpp = kStatsConsumers / g.tpr;
  g.rows_per_stage = g.rpp;  // set per element size at launch (stats_stage_rows)
  g.inv_T = T > 0 ? 1.0 / (double)T : 0.0;
  p.header_bytes = kWsAlign;
  p.ctr_bytes = kWsAlign;
  p.mean_bytes = align_up((size_t)g.C * sizeof(float), kWsAlign);
  p.part_bytes = align_up((size_t)g.P * g.rpp * g.C * sizeof(float4), kWsAlign);
  p.job_bytes = p.ctr_bytes + p.mean_bytes + p.part_bytes;
  return p;
}

// Rows per statistics stage: a multiple of rpp whose slabs fill a stage.
int stats_stage_rows(const KvGeom& g, bool bf16) {
  const size_t slab_bytes = (size_t)8 * g.tpr * (bf16 ? 2 : 4);
  return g.rpp * (int)std::max<size_t>(1, (size_t)kStatsStageBytes / (slab_bytes * g.rpp));
}

size_t kv_batch_workspace(const KvPlan& p, int n_jobs) { return p.header_bytes + p.job_bytes * (size_t)n_jobs; }

int quant_grid(int64_t nblocks, int sms) {
  const int64_t per_cta = 256;
  const int64_t need = (nblocks + per_cta - 1) / per_cta;
  return (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)std::max(sms, 1) * 8));
}

nvfp4_status check_job(const nvfp4_kv_job& j, int64_t T) {
  if (!j.tensor_scale) return NVFP4_EINVAL;
  if (T > 0 && (!j.x || !j.codes || !j.scales)) return NVFP4_EINVAL;
  if (j.smooth != 0 && j.smooth != 1) return NVFP4_EINVAL;
  if (!j.smooth && (j.mean_in || j.mean_out)) return NVFP4_EINVAL;
  if (!aligned(j.x, 32) || !aligned(j.codes, 16) || !aligned(j.scales, 16)) return NVFP4_EALIGN;
  if (!aligned(j.tensor_scale, 4) || !aligned(j.mean_in, 4) || !aligned(j.mean_out, 4)) return NVFP4_EALIGN;
  return NVFP4_OK;
}

enum KvPhase : int { kPhaseStats = 1, kPhaseQuant = 2, kPhaseBoth = 3 };

constexpr float kDenomStandard = 6.0f * 448.0f;  // g maps the tensor amax to 6 x the largest E4M3
constexpr float kDenomHeadroom = 4.0f * 448.0f;  // g leaves every block's 4-candidate under 448

nvfp4_status kv_run(const nvfp4_kv_job* jobs, int n_jobs, nvfp4_in_dtype dt, int64_t T, int H, int D,
                    int* dev_status, void* workspace, size_t workspace_bytes, void* stream, int phases,
                    float denom = kDenomStandard) {
  if (!jobs || n_jobs < 1) return NVFP4_EINVAL;
  if (dt != NVFP4_IN_BF16 && dt != NVFP4_IN_FP32) return NVFP4_EINVAL;
  if (!kv_shape_ok(T, H, D)) return NVFP4_ESHAPE;
  for (int i = 0; i < n_jobs; ++i) {
    nvfp4_status st = check_job(jobs[i], T);
    if (st != NVFP4_OK) return st;
  }
  if (!aligned(dev_status, 4)) return NVFP4_EALIGN;
  const bool bf16 = dt == NVFP4_IN_BF16;
  const int ctas = stats_ctas();
  if (ctas <= 0) return NVFP4_ECUDA;
  const KvPlan plan = kv_plan(T, H, D, ctas);
  const size_t need = kv_batch_workspace(plan, n_jobs);
  if (!workspace || workspace_bytes < need || !aligned(workspace, kWsAlign)) return NVFP4_EWORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  for (int first = 0; first < n_jobs; first += kMaxJobs) {
    KvBatch b;
    std::memset(&b, 0, sizeof(b));
    b.n = std::min(kMaxJobs, n_jobs - first);
    // unsmoothed tensors first: their statistics finish soonest (no reduction), so
    // their quantization starts while the smoothed ones are still being streamed
    int order[kMaxJobs], no = 0;
    for (int pass = 0; pass <= 1; ++pass)
      for (int i = 0; i < b.n; ++i)
        if ((jobs[first + i].smooth != 0) == (pass == 1)) order[no++] = first + i;
    for (int i = 0; i < b.n; ++i) {
      const nvfp4_kv_job& src = jobs[order[i]];
      KvJob& j = b.job[i];
      char* base = ws + plan.header_bytes + plan.job_bytes * (size_t)order[i];
      j.x = src.x;
      j.smooth = src.smooth;
      j.mean_in = src.mean_in;
      j.mean_out = src.mean_out;
      j.codes = src.codes;
      j.scales = src.scales;
      j.tensor_scale = src.tensor_scale;
      j.ctr = reinterpret_cast<unsigned*>(base);
      j.mean = reinterpret_cast<float*>(base + plan.ctr_bytes);
      j.part = reinterpret_cast<float4*>(base + plan.ctr_bytes + plan.mean_bytes);
    }
    KvGeom g = plan.geo;
    g.denom = denom;
    g.rows_per_stage = stats_stage_rows(g, bf16);
    g.header = reinterpret_cast<unsigned*>(ws);
    g.dev_status = dev_status;
    g.first_launch = first == 0 ? 1 : 0;
    if (T == 0) {
      if ((phases & kPhaseStats) && launch_kv_empty(b, g.C, dev_status, g.first_launch, s) != cudaSuccess)
        return NVFP4_ECUDA;
      continue;
    }
    if ((phases & kPhaseStats) && launch_kv_stats(b, g, bf16, s) != cudaSuccess) return NVFP4_ECUDA;
    if (phases & kPhaseQuant) {
      const KvQuantShape q = kv_quant_shape(T, g.C, b.n, device_sms());
      if (launch_kv_quant(b, g, q, bf16, s) != cudaSuccess) return NVFP4_ECUDA;
    }
  }
  return NVFP4_OK;
}

}  // namespace

extern "C" {

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_EINVAL: return "NVFP4_EINVAL: invalid argument";
    case NVFP4_ESHAPE: return "NVFP4_ESHAPE: unsupported shape";
    case NVFP4_EALIGN: return "NVFP4_EALIGN: misaligned pointer";
    case NVFP4_EWORKSPACE: return "NVFP4_EWORKSPACE: workspace missing, too small or misaligned";
    case NVFP4_ECUDA: return "NVFP4_ECUDA: CUDA error";
    case NVFP4_ECAPACITY: return "NVFP4_ECAPACITY: no free chunk slot in the KV-cache pool";
  }
  return "NVFP4_UNKNOWN";
}

int nvfp4_version(void) { return 100; }

size_t nvfp4_kv_workspace_bytes(int64_t T, int H, int D) { return nvfp4_kv_batched_workspace_bytes(1, T, H, D); }

size_t nvfp4_kv_batched_workspace_bytes(int n_jobs, int64_t T, int H, int D) {
  if (n_jobs < 1 || !kv_shape_ok(T, H, D)) return 0;
  const int ctas = stats_ctas();
  if (ctas <= 0) return 0;
  return kv_batch_workspace(kv_plan(T, H, D, ctas), n_jobs);
}

nvfp4_status nvfp4_kv_smooth_quant(const void* x, nvfp4_in_dtype dt, int64_t T, int H, int D, int smooth,
                                   const float* mean_in, float* mean_out, uint8_t* codes, uint8_t* scales,
                                   float* tensor_scale, int* dev_status, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  nvfp4_kv_job j;
  j.x = x;
  j.smooth = smooth;
  j.mean_in = mean_in;
  j.mean_out = mean_out;
  j.codes = codes;
  j.scales = scales;
  j.tensor_scale = tensor_scale;
  return kv_run(&j, 1, dt, T, H, D, dev_status, workspace, workspace_bytes, stream, kPhaseBoth);
}

nvfp4_status nvfp4_kv_smooth_quant_batched(const nvfp4_kv_job* jobs, int n_jobs, nvfp4_in_dtype dt, int64_t T,
                                           int H, int D, int* dev_status, void* workspace, size_t workspace_bytes,
                                           void* stream) {
  return kv_run(jobs, n_jobs, dt, T, H, D, dev_status, workspace, workspace_bytes, stream, kPhaseBoth);
}

nvfp4_status nvfp4_kv_smooth_quant_headroom(const nvfp4_kv_job* jobs, int n_jobs, nvfp4_in_dtype dt, int64_t T,
                                            int H, int D, int* dev_status, void* workspace, size_t workspace_bytes,
                                            void* stream) {
  return kv_run(jobs, n_jobs, dt, T, H, D, dev_status, workspace, workspace_bytes, stream, kPhaseBoth,
                kDenomHeadroom);
}

nvfp4_status nvfp4_kv_stats_batched(const nvfp4_kv_job* jobs, int n_jobs, nvfp4_in_dtype dt, int64_t T, int H,
                                    int D, void* workspace, size_t workspace_bytes, void* stream) {
  return kv_run(jobs, n_jobs, dt, T, H, D, nullptr, workspace, workspace_bytes, stream, kPhaseStats);
}

nvfp4_status nvfp4_kv_quant_batched(const nvfp4_kv_job* jobs, int n_jobs, nvfp4_in_dtype dt, int64_t T, int H,
                                    int D, int* dev_status, void* workspace, size_t workspace_bytes, void* stream) {
  return kv_run(jobs, n_jobs, dt, T, H, D, dev_status, workspace, workspace_bytes, stream, kPhaseQuant);
}

nvfp4_status nvfp4_kv_dequant(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                              const float* mean, int64_t tokens_per_group, int64_t T, int H, int D, void* out_bf16,
                              void* stream) {
  if (!kv_shape_ok(T, H, D)) return NVFP4_ESHAPE;
  if (tokens_per_group < 1) return NVFP4_ESHAPE;
  if (!tensor_scale) return NVFP4_EINVAL;
  if (T > 0 && (!codes || !scales || !out_bf16)) return NVFP4_EINVAL;
  if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(out_bf16, 16)) return NVFP4_EALIGN;
  if (!aligned(tensor_scale, 4) || !aligned(mean, 4)) return NVFP4_EALIGN;
  const int sms = device_sms();
  if (sms <= 0) return NVFP4_ECUDA;
  cudaError_t e = launch_kv_dequant(codes, scales, tensor_scale, mean, tokens_per_group, T, H * D, out_bf16, sms,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

size_t nvfp4_w2d_workspace_bytes(int64_t M, int64_t N) {
  if (M < 0 || N < 16 || (M % 16) != 0 || (N % 16) != 0) return 0;
  if (M > 0 && N > ((int64_t)1 << 46) / M) return 0;
  const int sms = device_sms();
  if (sms <= 0) return 0;
  return align_up((size_t)sms * 4 * sizeof(float), kWsAlign);
}

}  // extern "C"

namespace {

// Scratch of nvfp4_weight_quant_2d_static: one amax partial per amax CTA (4 per SM).
// A file-scope device array, so the call needs no workspace and allocates nothing.
// Every slot is written by its CTA before the quantization kernel reads it, so
// nothing in it has to start at zero.  All calls on one device share it.
constexpr int kW2dStaticPartials = 4096;  // room for 1024 SMs
static __device__ __align__(256) float g_w2d_static_scratch[kW2dStaticPartials];
// Device address of the scratch in the current context, looked up on every call
// (cudaGetSymbolAddress with the caller's device current), so that a call after a
// device reset -- which loads the module into a new context -- never reuses an
// address of the old one; nullptr if the lookup fails.
float* w2d_static_scratch() {
  void* q = nullptr;
  if (cudaGetSymbolAddress(&q, g_w2d_static_scratch) != cudaSuccess || !q) return nullptr;
  return static_cast<float*>(q);
}

}  // namespace

extern "C" {

nvfp4_status nvfp4_weight_quant_2d_static(const void* w, nvfp4_in_dtype dt, int64_t M, int64_t N, uint8_t* codes,
                                          uint8_t* scales, float* tensor_scale, int* dev_status, void* stream) {
  if (dt != NVFP4_IN_BF16 && dt != NVFP4_IN_FP32) return NVFP4_EINVAL;
  if (M < 0 || N < 16 || (M % 16) != 0 || (N % 16) != 0) return NVFP4_ESHAPE;
  if (M > 0 && N > ((int64_t)1 << 46) / M) return NVFP4_ESHAPE;  // (chunk index) * (CTAs) fits in int64
  if (!tensor_scale) return NVFP4_EINVAL;
  if (M > 0 && (!w || !codes || !scales)) return NVFP4_EINVAL;
  if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 16)) return NVFP4_EALIGN;
  if (!aligned(tensor_scale, 4) || !aligned(dev_status, 4)) return NVFP4_EALIGN;
  const int sms = device_sms();
  if (sms <= 0) return NVFP4_ECUDA;
  if (sms * 4 > kW2dStaticPartials) return NVFP4_EWORKSPACE;  // more amax CTAs than the scratch holds
  float* scratch = w2d_static_scratch();
  if (!scratch) return NVFP4_ECUDA;
  W2dGeom geo;
  geo.M = M;
  geo.N = N;
  geo.amax_ctas = sms * 4;
  const int64_t ntiles = (M / 16) * (N / 16);
  const int qctas = quant_grid(2 * ntiles, sms);  // two threads per tile
  cudaError_t e = launch_w2d_quant(w, dt == NVFP4_IN_BF16, geo, codes, scales, tensor_scale, dev_status, scratch,
                                   qctas, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

nvfp4_status nvfp4_weight_quant_2d(const void* w, nvfp4_in_dtype dt, int64_t M, int64_t N, uint8_t* codes,
                                   uint8_t* scales, float* tensor_scale, int* dev_status, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (dt != NVFP4_IN_BF16 && dt != NVFP4_IN_FP32) return NVFP4_EINVAL;
  if (M < 0 || N < 16 || (M % 16) != 0 || (N % 16) != 0) return NVFP4_ESHAPE;
  if (M > 0 && N > ((int64_t)1 << 46) / M) return NVFP4_ESHAPE;  // (chunk index) * (CTAs) fits in int64
  if (!tensor_scale) return NVFP4_EINVAL;
  if (M > 0 && (!w || !codes || !scales)) return NVFP4_EINVAL;
  if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 16)) return NVFP4_EALIGN;
  if (!aligned(tensor_scale, 4) || !aligned(dev_status, 4)) return NVFP4_EALIGN;
  const int sms = device_sms();
  if (sms <= 0) return NVFP4_ECUDA;
  const size_t need = align_up((size_t)sms * 4 * sizeof(float), kWsAlign);
  if (!workspace || workspace_bytes < need || !aligned(workspace, kWsAlign)) return NVFP4_EWORKSPACE;
  W2dGeom geo;
  geo.M = M;
  geo.N = N;
  geo.amax_ctas = sms * 4;
  const int64_t ntiles = (M / 16) * (N / 16);
  const int qctas = quant_grid(2 * ntiles, sms);  // two threads per tile
  cudaError_t e = launch_w2d_quant(w, dt == NVFP4_IN_BF16, geo, codes, scales, tensor_scale, dev_status,
                                   static_cast<float*>(workspace), qctas, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

size_t nvfp4_w2d_batched_workspace_bytes(int n_jobs) {
  if (n_jobs < 1) return 0;
  return align_up((size_t)(1 + 2 * kMaxW2dJobs) * sizeof(unsigned), kWsAlign);
}

nvfp4_status nvfp4_weight_quant_2d_batched(const nvfp4_w2d_job* jobs, int n_jobs, nvfp4_in_dtype dt, int* dev_status,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  if (!jobs || n_jobs < 1) return NVFP4_EINVAL;
  if (dt != NVFP4_IN_BF16 && dt != NVFP4_IN_FP32) return NVFP4_EINVAL;
  for (int i = 0; i < n_jobs; ++i) {
    const nvfp4_w2d_job& j = jobs[i];
    if (j.M < 0 || j.N < 16 || (j.M % 16) != 0 || (j.N % 16) != 0) return NVFP4_ESHAPE;
    if (j.M > 0 && j.N > ((int64_t)1 << 46) / j.M) return NVFP4_ESHAPE;
    if (!j.tensor_scale) return NVFP4_EINVAL;
    if (j.M > 0 && (!j.w || !j.codes || !j.scales)) return NVFP4_EINVAL;
    if (!aligned(j.w, 16) || !aligned(j.codes, 16) || !aligned(j.scales, 16)) return NVFP4_EALIGN;
    if (!aligned(j.tensor_scale, 4)) return NVFP4_EALIGN;
  }
  if (!aligned(dev_status, 4)) return NVFP4_EALIGN;
  const size_t need = align_up((size_t)(1 + 2 * kMaxW2dJobs) * sizeof(unsigned), kWsAlign);
  if (!workspace || workspace_bytes < need || !aligned(workspace, kWsAlign)) return NVFP4_EWORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return NVFP4_ECUDA;
  const bool bf16 = dt == NVFP4_IN_BF16;
  for (int first = 0; first < n_jobs; first += kMaxW2dJobs) {
    W2dBatch b;
    std::memset(&b, 0, sizeof(b));
    b.n = std::min(kMaxW2dJobs, n_jobs - first);
    b.reset_status = first == 0 ? 1 : 0;
    b.amax_grid = sms * 4;
    // smallest matrices first: their amax is complete soonest, so their
    // quantization starts while the amax pass reads the larger ones
    int order[kMaxW2dJobs];
    for (int i = 0; i < b.n; ++i) order[i] = first + i;
    std::stable_sort(order, order + b.n, [&](int x, int y) { return jobs[x].M * jobs[x].N < jobs[y].M * jobs[y].N; });
    int q = 0;
    for (int i = 0; i < b.n; ++i) {
      const nvfp4_w2d_job& src = jobs[order[i]];
      W2dJob& j = b.job[i];
      j.w = src.w;
      j.M = src.M;
      j.N = src.N;
      j.codes = src.codes;
      j.scales = src.scales;
      j.tensor_scale = src.tensor_scale;
      j.quant_ctas = quant_grid(2 * (src.M / 16) * (src.N / 16), sms);  // two threads per tile
      j.quant_begin = q;
      q += j.quant_ctas;
    }
    if (launch_w2d_batch_overlapped(b, bf16, q, static_cast<unsigned*>(workspace), dev_status,
                                    static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return NVFP4_ECUDA;
  }
  return NVFP4_OK;
}

nvfp4_status nvfp4_weight_dequant_2d(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                                     int64_t M, int64_t N, void* out_bf16, void* stream) {
  if (M < 0 || N < 16 || (M % 16) != 0 || (N % 16) != 0) return NVFP4_ESHAPE;
  if (!tensor_scale) return NVFP4_EINVAL;
  if (M > 0 && (!codes || !scales || !out_bf16)) return NVFP4_EINVAL;
  if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(out_bf16, 16) || !aligned(tensor_scale, 4))
    return NVFP4_EALIGN;
  const int sms = device_sms();
  if (sms <= 0) return NVFP4_ECUDA;
  cudaError_t e = launch_w2d_dequant(codes, scales, tensor_scale, M, N, out_bf16, sms,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

}  // extern "C"
