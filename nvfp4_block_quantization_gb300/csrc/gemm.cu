// gemm.cu -- the W4A4 NVFP4 GEMM path (sm_103a): Y = X W^T with X quantized by
// the 1-D quantizer (one E4M3 scale per 16 elements of a row) and W by the 2-D
// quantizer (one E4M3 scale per 16x16 tile), each with its fp32 tensor scale.
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page): training step 4 runs the GEMMs in NVFP4 with 2-D block
// scales for weights and 1-D block scales for activations; inference step 6
// merges the weights into a W4A4 model.
//
// The contraction is a dense block-scaled FP4 GEMM, so it runs on the tensor
// cores through cuBLASLt (E2M1 operands, VEC16 UE4M3 block scales, fp32
// accumulation).  This file adds what the library needs around it:
//   - the block scales rearranged into the tensor cores' scale layout: tiles of
//     128 rows x 4 blocks (512 bytes, rows r % 32 at 16-byte steps, r / 32 at
//     4-byte steps, the block within the tile at 1-byte steps), K tiles
//     fastest, zeros in the padding; a weight tile's scale is repeated for its
//     16 rows;
//   - alpha = gX * gW computed on the device, so the call never reads device
//     memory on the host;
//   - a caller-owned plan holding the cuBLASLt handle, descriptors and the
//     chosen algorithm.
#include <cstring>
#include <new>

#include <cublasLt.h>

#include "nvfp4.h"
#include "common.cuh"
#include "rht16.cuh"

struct nvfp4_gemm_plan {
  int64_t M, N, K;
  cublasLtHandle_t handle;
  cublasLtMatmulDesc_t op;
  cublasLtMatrixLayout_t lw, lx, ly;
  cublasLtMatmulAlgo_t algo;
  size_t algo_workspace;
};

namespace nvfp4 {
namespace {

constexpr size_t kGemmWorkspace = (size_t)32 << 20;  // cuBLASLt workspace offered to the heuristic
constexpr size_t kScalarBytes = 256;                 // alpha and beta at the front of the workspace

int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// One thread per output word: the four blocks of one row inside one tile sit
// in consecutive bytes, so word w of tile (rt, ct) holds blocks 4 ct .. 4 ct + 3
// of row 128 rt + (w % 4) * 32 + w / 4.  Stores are in output order (coalesced);
// the gather from the row-major input is four byte loads.
//   kTile: the input is a 16x16-tile scale grid [rows / 16][kblocks].
template <bool kTile>
__global__ void __launch_bounds__(256) scales_to_mma_kernel(const uint8_t* __restrict__ in, int64_t rows,
                                                            int64_t kblocks, uint32_t* __restrict__ out,
                                                            int64_t out_words) {
  const int64_t kbt = (kblocks + 3) / 4;
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < out_words; o += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = o >> 7;
    const int w = (int)(o & 127);
    const int64_t rt = tile / kbt, ct = tile - rt * kbt;
    const int64_t r = rt * 128 + (w & 3) * 32 + (w >> 2), kb0 = ct * 4;
    uint32_t v = 0;
    if (r < rows) {
      const uint8_t* src = in + (kTile ? (r >> 4) : r) * kblocks;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (kb0 + c < kblocks) v |= (uint32_t)src[kb0 + c] << (8 * c);
    }
    out[o] = v;
  }
}

// Random Hadamard transform of 16-element blocks along the rows (rht16_block):
// one thread per block, widened exactly to fp32 first.
template <bool kBF16>
__global__ void __launch_bounds__(256) rht16_kernel(const void* __restrict__ x, int64_t nblocks, uint32_t signs,
                                                    float* __restrict__ out) {
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblocks; b += (int64_t)gridDim.x * blockDim.x) {
    float v[16];
    if (kBF16) {
      uint32_t w[8];
      ld_nc_v8(static_cast<const uint16_t*>(x) + b * 16, w);
#pragma unroll
      for (int i = 0; i < 8; ++i) { v[2 * i] = bf16lo(w[i]); v[2 * i + 1] = bf16hi(w[i]); }
    } else {
      uint32_t w[16];
      ld_nc_v8(static_cast<const float*>(x) + b * 16, w);
      ld_nc_v8(static_cast<const float*>(x) + b * 16 + 8, w + 8);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(w[i]);
    }
    rht16_block(v, signs);
    float4* o = reinterpret_cast<float4*>(out + b * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
}

__global__ void alpha_kernel(const float* __restrict__ gx, const float* __restrict__ gw, float* __restrict__ ab) {
  ab[0] = __fmul_rn(*gx, *gw);
  ab[1] = 0.0f;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

nvfp4_status launch_scales(const uint8_t* in, int64_t rows, int64_t kblocks, bool tile, uint8_t* out, void* stream) {
  const int64_t bytes = nvfp4_mma_scales_bytes(rows, kblocks * 16);
  if (bytes == 0) return NVFP4_OK;
  const int sms = sm_count();
  if (sms <= 0) return NVFP4_ECUDA;
  const int64_t words = bytes / 4;  // a whole number of 512-byte tiles
  int64_t grid = (words + 255) / 256;
  if (grid > (int64_t)sms * 16) grid = (int64_t)sms * 16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* o = reinterpret_cast<uint32_t*>(out);
  if (tile) scales_to_mma_kernel<true><<<(unsigned)grid, 256, 0, s>>>(in, rows, kblocks, o, words);
  else scales_to_mma_kernel<false><<<(unsigned)grid, 256, 0, s>>>(in, rows, kblocks, o, words);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

void destroy(nvfp4_gemm_plan* p) {
  if (!p) return;
  if (p->ly) cublasLtMatrixLayoutDestroy(p->ly);
  if (p->lx) cublasLtMatrixLayoutDestroy(p->lx);
  if (p->lw) cublasLtMatrixLayoutDestroy(p->lw);
  if (p->op) cublasLtMatmulDescDestroy(p->op);
  if (p->handle) cublasLtDestroy(p->handle);
  delete p;
}

}  // namespace
}  // namespace nvfp4

extern "C" {

int64_t nvfp4_mma_scales_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 16 || (K % 16) != 0) return 0;
  return nvfp4::round_up(rows, 128) * nvfp4::round_up(K / 16, 4);
}

nvfp4_status nvfp4_scales_to_mma(const uint8_t* scales, int64_t rows, int64_t K, uint8_t* out, void* stream) {
  if (rows < 0 || K < 16 || (K % 16) != 0) return NVFP4_ESHAPE;
  if (rows > 0 && (!scales || !out)) return NVFP4_EINVAL;
  if (!nvfp4::aligned_to(out, 16)) return NVFP4_EALIGN;
  return nvfp4::launch_scales(scales, rows, K / 16, false, out, stream);
}

nvfp4_status nvfp4_w2d_scales_to_mma(const uint8_t* scales, int64_t N, int64_t K, uint8_t* out, void* stream) {
  if (N < 0 || (N % 16) != 0 || K < 16 || (K % 16) != 0) return NVFP4_ESHAPE;
  if (N > 0 && (!scales || !out)) return NVFP4_EINVAL;
  if (!nvfp4::aligned_to(out, 16)) return NVFP4_EALIGN;
  return nvfp4::launch_scales(scales, N, K / 16, true, out, stream);
}

nvfp4_status nvfp4_rht16(const void* x, nvfp4_in_dtype dt, int64_t rows, int64_t K, uint32_t signs, float* out,
                         void* stream) {
  if (dt != NVFP4_IN_BF16 && dt != NVFP4_IN_FP32) return NVFP4_EINVAL;
  if (rows < 0 || K < 16 || (K % 16) != 0) return NVFP4_ESHAPE;
  if (rows > 0 && K > ((int64_t)1 << 46) / rows) return NVFP4_ESHAPE;
  if (signs > 0xFFFFu) return NVFP4_EINVAL;
  if (rows == 0) return NVFP4_OK;
  if (!x || !out) return NVFP4_EINVAL;
  if (!nvfp4::aligned_to(x, 32) || !nvfp4::aligned_to(out, 16)) return NVFP4_EALIGN;
  const int sms = nvfp4::sm_count();
  if (sms <= 0) return NVFP4_ECUDA;
  const int64_t nb = rows * (K / 16);
  int64_t grid = (nb + 255) / 256;
  if (grid > (int64_t)sms * 16) grid = (int64_t)sms * 16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dt == NVFP4_IN_BF16) nvfp4::rht16_kernel<true><<<(unsigned)grid, 256, 0, s>>>(x, nb, signs, out);
  else nvfp4::rht16_kernel<false><<<(unsigned)grid, 256, 0, s>>>(x, nb, signs, out);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

size_t nvfp4_gemm_workspace_bytes(void) { return nvfp4::kScalarBytes + nvfp4::kGemmWorkspace; }

nvfp4_status nvfp4_gemm_plan_create(int64_t M, int64_t N, int64_t K, nvfp4_gemm_plan** plan) {
  if (!plan) return NVFP4_EINVAL;
  *plan = nullptr;
  if (M < 1 || N < 16 || (N % 16) != 0 || K < 32 || (K % 32) != 0) return NVFP4_ESHAPE;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return NVFP4_ESHAPE;
  nvfp4_gemm_plan* p = new (std::nothrow) nvfp4_gemm_plan;
  if (!p) return NVFP4_ECUDA;
  std::memset(p, 0, sizeof(*p));
  p->M = M;
  p->N = N;
  p->K = K;
  bool ok = cublasLtCreate(&p->handle) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatmulDescCreate(&p->op, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS;
  // Y^T (N x M, column-major) = W (N x K) * X^T: both operands K-contiguous
  const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
  const int32_t mode = CUBLASLT_MATMUL_MATRIX_SCALE_VEC16_UE4M3;
  const cublasLtPointerMode_t pm = CUBLASLT_POINTER_MODE_DEVICE;
  const void* placeholder = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));  // set per call
  ok = ok && cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta)) == CUBLAS_STATUS_SUCCESS &&
       cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb)) == CUBLAS_STATUS_SUCCESS &&
       cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_A_SCALE_MODE, &mode, sizeof(mode)) == CUBLAS_STATUS_SUCCESS &&
       cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_B_SCALE_MODE, &mode, sizeof(mode)) == CUBLAS_STATUS_SUCCESS &&
       cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_A_SCALE_POINTER, &placeholder, sizeof(placeholder)) == CUBLAS_STATUS_SUCCESS &&
       cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &placeholder, sizeof(placeholder)) == CUBLAS_STATUS_SUCCESS &&
       cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_POINTER_MODE, &pm, sizeof(pm)) == CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatrixLayoutCreate(&p->lw, CUDA_R_4F_E2M1, (uint64_t)K, (uint64_t)N, K) == CUBLAS_STATUS_SUCCESS &&
       cublasLtMatrixLayoutCreate(&p->lx, CUDA_R_4F_E2M1, (uint64_t)K, (uint64_t)M, K) == CUBLAS_STATUS_SUCCESS &&
       cublasLtMatrixLayoutCreate(&p->ly, CUDA_R_16BF, (uint64_t)N, (uint64_t)M, N) == CUBLAS_STATUS_SUCCESS;
  cublasLtMatmulPreference_t pref = nullptr;
  cublasLtMatmulHeuristicResult_t res;
  std::memset(&res, 0, sizeof(res));
  int found = 0;
  const size_t cap = nvfp4::kGemmWorkspace;
  ok = ok && cublasLtMatmulPreferenceCreate(&pref) == CUBLAS_STATUS_SUCCESS &&
       cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &cap, sizeof(cap)) == CUBLAS_STATUS_SUCCESS &&
       cublasLtMatmulAlgoGetHeuristic(p->handle, p->op, p->lw, p->lx, p->ly, p->ly, pref, 1, &res, &found) == CUBLAS_STATUS_SUCCESS &&
       found >= 1;
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (!ok) {
    nvfp4::destroy(p);
    return NVFP4_ECUDA;
  }
  p->algo = res.algo;
  p->algo_workspace = res.workspaceSize;
  *plan = p;
  return NVFP4_OK;
}

void nvfp4_gemm_plan_destroy(nvfp4_gemm_plan* plan) { nvfp4::destroy(plan); }

nvfp4_status nvfp4_gemm_w4a4(nvfp4_gemm_plan* plan, const uint8_t* x_codes, const uint8_t* x_scales_mma,
                             const float* x_tensor_scale, const uint8_t* w_codes, const uint8_t* w_scales_mma,
                             const float* w_tensor_scale, void* y_bf16, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!plan) return NVFP4_EINVAL;
  if (!x_codes || !x_scales_mma || !x_tensor_scale || !w_codes || !w_scales_mma || !w_tensor_scale || !y_bf16)
    return NVFP4_EINVAL;
  if (!nvfp4::aligned_to(x_codes, 16) || !nvfp4::aligned_to(w_codes, 16) || !nvfp4::aligned_to(x_scales_mma, 16) ||
      !nvfp4::aligned_to(w_scales_mma, 16) || !nvfp4::aligned_to(y_bf16, 16) ||
      !nvfp4::aligned_to(x_tensor_scale, 4) || !nvfp4::aligned_to(w_tensor_scale, 4))
    return NVFP4_EALIGN;
  if (!workspace || !nvfp4::aligned_to(workspace, 256) || workspace_bytes < nvfp4_gemm_workspace_bytes())
    return NVFP4_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* ab = static_cast<float*>(workspace);  // [0] alpha = gX * gW, [1] beta = 0
  nvfp4::alpha_kernel<<<1, 1, 0, s>>>(x_tensor_scale, w_tensor_scale, ab);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ECUDA;
  if (cublasLtMatmulDescSetAttribute(plan->op, CUBLASLT_MATMUL_DESC_A_SCALE_POINTER, &w_scales_mma,
                                     sizeof(w_scales_mma)) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatmulDescSetAttribute(plan->op, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &x_scales_mma,
                                     sizeof(x_scales_mma)) != CUBLAS_STATUS_SUCCESS)
    return NVFP4_ECUDA;
  char* gemm_ws = static_cast<char*>(workspace) + nvfp4::kScalarBytes;
  const cublasStatus_t st = cublasLtMatmul(plan->handle, plan->op, ab, w_codes, plan->lw, x_codes, plan->lx, ab + 1,
                                           y_bf16, plan->ly, y_bf16, plan->ly, &plan->algo, gemm_ws,
                                           nvfp4::kGemmWorkspace, s);
  return st == CUBLAS_STATUS_SUCCESS ? NVFP4_OK : NVFP4_ECUDA;
}

}  // extern "C"
