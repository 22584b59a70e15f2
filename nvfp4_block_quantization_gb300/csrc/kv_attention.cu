// kv_attention.cu -- attention that reads the NVFP4 KV cache directly
// (sm_103a): a few query tokens per head attend over one view of the
// multi-shot cache; K and V are dequantized in registers from the pool's codes,
// scales, tensor scales and (for K) means, so the cache is read at 0.5625 bytes
// per element instead of the 2 of a bf16 cache.
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page), inference steps 7 and 9: attention reads the NVFP4 KV cache
// over the global sink, the shot sink and the rolling frames.
//
// Per view token t (pool row frame_row[t / L_f] + t % L_f, slot
// frame_slot[t / L_f]) and channel d of head h, with S = fl(E * g[slot]) the
// scale of d's 16-channel block:
//   k = Q_k S_k + mean[slot][h][d],  v = Q_v S_v,
// s_i(t) = scale * q_i[h] . k and o_i = sum_t softmax_t(s_i) v_t, in fp32.  The
// block scale is common to the block's 16 channels, so q . k over a block is
// evaluated as S_k (q . Q_k) + q . mean (the second sum once per slot), and p v as
// (p S_v) Q_v: the same values up to fp32 rounding order.
//
// Split-KV: CTA (h, s) takes the view tokens [s R, (s + 1) R) of head h (R from 256 to
// 2048 tokens, sized so that the H x S grid is one wave of resident CTAs); a group
// of D / 16 lanes owns a few tokens per step (one 16-channel scale block per lane
// and token: one 8-byte code load and one scale byte each, all issued before any
// is used),
// reduces the dot products over its group with shuffles, and keeps an online
// softmax (running max m, sum l, weighted V o) per query.
// The CTA merges its groups' states and writes one partial per query; the
// combine kernel merges the splits.
#include <algorithm>
#include <cstring>

#include "nvfp4.h"
#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kAttnMaxQ = 4;
constexpr int kAttnTokensPerSplit = 256;  // the shortest split: the workspace holds ceil(T / 256) partials
constexpr int kAttnMaxTokensPerSplit = 2048;  // the longest: a lane group's fp32 sums stay at most 128 terms

struct AttnView {
  int64_t row[NVFP4_MAX_VIEW_FRAMES];
  int meta[NVFP4_MAX_VIEW_FRAMES];
};

// The E2M1 values of four code bytes (eight elements; byte j holds elements 2j in its low nibble
// and 2j + 1 in its high one), the word split into bytes inside the conversion sequence.
__device__ __forceinline__ void decode8(uint32_t w, float* out) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 h0, h1, h2, h3;\n\t"
      ".reg .b16 l0, u0, l1, u1, l2, u2, l3, u3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %8;\n\t"
      "cvt.rn.f16x2.e2m1x2 h0, b0;\n\tcvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h2, b2;\n\tcvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
      "mov.b32 {l0, u0}, h0;\n\tmov.b32 {l1, u1}, h1;\n\tmov.b32 {l2, u2}, h2;\n\tmov.b32 {l3, u3}, h3;\n\t"
      "cvt.f32.f16 %0, l0;\n\tcvt.f32.f16 %1, u0;\n\tcvt.f32.f16 %2, l1;\n\tcvt.f32.f16 %3, u1;\n\t"
      "cvt.f32.f16 %4, l2;\n\tcvt.f32.f16 %5, u2;\n\tcvt.f32.f16 %6, l3;\n\tcvt.f32.f16 %7, u3;\n\t}"
      : "=f"(out[0]), "=f"(out[1]), "=f"(out[2]), "=f"(out[3]), "=f"(out[4]), "=f"(out[5]), "=f"(out[6]),
        "=f"(out[7])
      : "r"(w));
}

// The E2M1 values of one token's 16-channel block (one scale block) from its 8 code bytes.
__device__ __forceinline__ void decode16(uint2 codes, float out[16]) {
  decode8(codes.x, out);
  decode8(codes.y, out + 8);
}

// Register caps: 128 for one query (16 warps per SM), 168 for two, 255 otherwise.
template <int D, int NQ>
__global__ void __launch_bounds__(kAttnThreads, NQ == 1 ? 4 : (NQ == 2 ? 3 : 2)) attn_split_kernel(
    const float* __restrict__ q, const uint8_t* __restrict__ kc, const uint8_t* __restrict__ ks,
    const float* __restrict__ kg, const float* __restrict__ kmean, const uint8_t* __restrict__ vc,
    const uint8_t* __restrict__ vs, const float* __restrict__ vg, int64_t L, int64_t T, int64_t R, int H,
    float scale, float* __restrict__ part, const __grid_constant__ AttnView view) {
  constexpr int G = D / 16;         // lanes per token: one 16-channel scale block each
  constexpr int TPW = 32 / G;       // tokens per warp step
  constexpr int W = kAttnThreads / 32;
  const int h = blockIdx.x, s = blockIdx.y, S = gridDim.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / G, gl = lane % G;  // token slot in the warp step, lane in the group
  const int C = H * D;
  // this lane's 16 channels of head h: d0 = 16 gl
  float qv[NQ][16];
#pragma unroll
  for (int i = 0; i < NQ; ++i)
#pragma unroll
    for (int j = 0; j < 16; ++j) qv[i][j] = __ldg(q + (size_t)i * C + (size_t)h * D + 16 * gl + j);
  float m[NQ], l[NQ], o[NQ][16];
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) o[i][j] = 0.0f;
  }
  const int64_t t_begin = (int64_t)s * R;
  const int64_t t_end = t_begin + R < T ? t_begin + R : T;
  // U tokens per group per step: their code and scale loads are all issued before
  // any of them is used
  constexpr int U = NQ <= 2 ? 4 : 2;
  int64_t fend = -1, delta = 0;
  int slot = -1, mslot = -1;
  float gk = 0.0f, gv = 0.0f;
  float cq[NQ];  // sum over this lane's 16 channels of q_i * mean (K's means of the current slot)
#pragma unroll
  for (int i = 0; i < NQ; ++i) cq[i] = 0.0f;
  for (int64_t t0 = t_begin + (int64_t)warp * TPW * U; t0 < t_end; t0 += (int64_t)W * TPW * U) {
    uint2 kcode[U], vcode[U];
    uint32_t ke[U], ve[U];
    int sl[U];
    bool on[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t t = t0 + (int64_t)u * TPW + grp;
      on[u] = t < t_end;  // uniform within the group
      sl[u] = slot;
      if (on[u]) {
        if (t >= fend) {
          const int64_t f = t / L;
          fend = (f + 1) * L;
          delta = view.row[f] - f * L;
          slot = view.meta[f];
        }
        sl[u] = slot;
        const size_t cell = ((size_t)(t + delta) * H + h);  // (pool row, head)
        kcode[u] = __ldg(reinterpret_cast<const uint2*>(kc + cell * (D / 2)) + gl);
        vcode[u] = __ldg(reinterpret_cast<const uint2*>(vc + cell * (D / 2)) + gl);
        ke[u] = __ldg(ks + cell * (D / 16) + gl);
        ve[u] = __ldg(vs + cell * (D / 16) + gl);
      }
    }
    // first the K dot products of all U tokens (independent chains, two per token and query),
    // with each token's V block scale taken while its slot's tensor scales are current
    float sc[U][NQ], Sv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      Sv[u] = 0.0f;
#pragma unroll
      for (int i = 0; i < NQ; ++i) sc[u][i] = 0.0f;
      if (on[u]) {
        if (sl[u] != mslot) {  // a frame of another slot: its tensor scales (and K means)
          mslot = sl[u];
          gk = __ldg(kg + mslot);
          gv = __ldg(vg + mslot);
          if (kmean) {
            float mu[16];
            const float4* mp = reinterpret_cast<const float4*>(kmean + (size_t)mslot * C + (size_t)h * D + 16 * gl);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const float4 a = __ldg(mp + k4);
              mu[4 * k4] = a.x; mu[4 * k4 + 1] = a.y; mu[4 * k4 + 2] = a.z; mu[4 * k4 + 3] = a.w;
            }
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
              float a = 0.0f;
#pragma unroll
              for (int j = 0; j < 16; ++j) a = __fmaf_rn(qv[i][j], mu[j], a);
              cq[i] = a;
            }
          }
        }
        // q . k over the block = S_k * (q . Q_k) + q . mean: the scale is common to the block
        const float Sk = __fmul_rn(e4m3_value(ke[u]), gk);
        Sv[u] = __fmul_rn(e4m3_value(ve[u]), gv);
        float kq[16];
        decode16(kcode[u], kq);
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            a0 = __fmaf_rn(qv[i][j], kq[j], a0);
            a1 = __fmaf_rn(qv[i][j + 1], kq[j + 1], a1);
          }
          sc[u][i] = __fmaf_rn(__fadd_rn(a0, a1), Sk, cq[i]);
        }
      }
    }
    // the dot products' shuffle trees over the group
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < NQ; ++i)
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) sc[u][i] += __shfl_xor_sync(0xffffffffu, sc[u][i], off);
    // then each token in turn: the online softmax update, dequantize V and accumulate
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (on[u]) {
        // p * v = (p * S_v) * Q_v: the scale is folded into the weight
        float vq[16];
        decode16(vcode[u], vq);
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          const float sv = __fmul_rn(sc[u][i], scale);
          if (sv > m[i]) {  // a new running maximum: rescale what has been summed so far
            const float corr = __expf(m[i] - sv);
            l[i] = __fmul_rn(l[i], corr);
#pragma unroll
            for (int j = 0; j < 16; ++j) o[i][j] = __fmul_rn(o[i][j], corr);
            m[i] = sv;
          }
          const float p = __expf(sv - m[i]);
          l[i] = __fadd_rn(l[i], p);
          const float pS = __fmul_rn(p, Sv[u]);
#pragma unroll
          for (int j = 0; j < 16; ++j) o[i][j] = __fmaf_rn(pS, vq[j], o[i][j]);
        }
      }
    }
  }
  // merge the CTA's groups (W warps x TPW groups) per query in shared memory
  __shared__ float sm_m[W * TPW][NQ], sm_l[W * TPW][NQ];
  __shared__ float sm_o[W * TPW][NQ][D];
  const int gid = warp * TPW + grp;
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    if (gl == 0) {
      sm_m[gid][i] = m[i];
      sm_l[gid][i] = l[i];
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) sm_o[gid][i][16 * gl + j] = o[i][j];
  }
  __syncthreads();
  for (int x = threadIdx.x; x < NQ * D; x += blockDim.x) {
    const int i = x / D, d = x - i * D;
    float M = -INFINITY;
    for (int g2 = 0; g2 < W * TPW; ++g2) M = fmaxf(M, sm_m[g2][i]);
    float Ls = 0.0f, Os = 0.0f;
    for (int g2 = 0; g2 < W * TPW; ++g2) {
      const float w = sm_m[g2][i] == -INFINITY ? 0.0f : __expf(sm_m[g2][i] - M);
      Ls = __fmaf_rn(sm_l[g2][i], w, Ls);
      Os = __fmaf_rn(sm_o[g2][i][d], w, Os);
    }
    float* pp = part + (((size_t)h * S + s) * NQ + i) * (D + 2);
    pp[2 + d] = Os;
    if (d == 0) {
      pp[0] = M;
      pp[1] = Ls;
    }
  }
}

// out[i][h][d] = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M) over the splits.
// CTA (h, i): the splits' partials are loaded by the whole CTA into shared
// memory, kCombineChunk splits at a time (coalesced, eight loads in flight per thread), and
// each chunk is merged into a running (max, sum, weighted V) per channel.
constexpr int kCombineChunk = 64;
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ part, int S, int NQ, int H,
                                                           float* __restrict__ out) {
  __shared__ float sp[kCombineChunk][D + 2];
  const int h = blockIdx.x, i = blockIdx.y;
  float M = -INFINITY, Ls = 0.0f, Os = 0.0f;  // thread d < D: channel d
  const int d = threadIdx.x;
  for (int c0 = 0; c0 < S; c0 += kCombineChunk) {
    const int n = S - c0 < kCombineChunk ? S - c0 : kCombineChunk;
    __syncthreads();  // the previous chunk has been read
    // eight loads in flight per thread before any is stored
    for (int x0 = threadIdx.x; x0 < n * (D + 2); x0 += 8 * blockDim.x) {
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int x = x0 + k * blockDim.x, sj = x / (D + 2), r = x - sj * (D + 2);
        v[k] = x < n * (D + 2) ? part[(((size_t)h * S + c0 + sj) * NQ + i) * (D + 2) + r] : 0.0f;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int x = x0 + k * blockDim.x, sj = x / (D + 2), r = x - sj * (D + 2);
        if (x < n * (D + 2)) sp[sj][r] = v[k];
      }
    }
    __syncthreads();
    if (d < D) {
      float Mc = M;
      for (int sj = 0; sj < n; ++sj) Mc = fmaxf(Mc, sp[sj][0]);
      if (Mc != -INFINITY) {
        const float corr = M == -INFINITY ? 0.0f : __expf(M - Mc);
        Ls = __fmul_rn(Ls, corr);
        Os = __fmul_rn(Os, corr);
        for (int sj = 0; sj < n; ++sj) {
          const float w = sp[sj][0] == -INFINITY ? 0.0f : __expf(sp[sj][0] - Mc);
          Ls = __fmaf_rn(sp[sj][1], w, Ls);
          Os = __fmaf_rn(sp[sj][2 + d], w, Os);
        }
        M = Mc;
      }
    }
  }
  if (d < D) out[(size_t)i * H * D + (size_t)h * D + d] = Os / Ls;
}

// Tokens per split: the H x S grid fills one wave of the CTAs that fit on the GPU at
// once (fewer partials for the combine, no partial last wave); a multiple of the
// 64 tokens a CTA takes per step, between kAttnTokensPerSplit and kAttnMaxTokensPerSplit.
template <int D, int NQ>
cudaError_t split_tokens(int64_t T, int H, int64_t* R) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_split_kernel<D, NQ>, kAttnThreads, 0);
  if (e != cudaSuccess) return e;
  const int64_t per_head = std::max<int64_t>(1, (int64_t)sms * std::max(per_sm, 1) / H);
  const int64_t r = (T + per_head - 1) / per_head;
  *R = std::min<int64_t>(kAttnMaxTokensPerSplit, std::max<int64_t>(kAttnTokensPerSplit, (r + 63) / 64 * 64));
  return cudaSuccess;
}

template <int D, int NQ>
cudaError_t launch_attn(const float* q, const uint8_t* kc, const uint8_t* ks, const float* kg, const float* km,
                        const uint8_t* vc, const uint8_t* vs, const float* vg, int64_t L, int64_t T, int H,
                        float scale, float* part, const AttnView& view, float* out, cudaStream_t st) {
  int64_t R = 0;
  cudaError_t e0 = split_tokens<D, NQ>(T, H, &R);
  if (e0 != cudaSuccess) return e0;
  const int S = (int)((T + R - 1) / R);  // at most ceil(T / 256): the caller checked that it fits
  attn_split_kernel<D, NQ><<<dim3(H, S), kAttnThreads, 0, st>>>(q, kc, ks, kg, km, vc, vs, vg, L, T, R, H, scale,
                                                                part, view);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<D><<<dim3(H, NQ), 256, 0, st>>>(part, S, NQ, H, out);
  return cudaGetLastError();
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace nvfp4

extern "C" {

size_t nvfp4_kv_attention_workspace_bytes(int n_frames, int64_t tokens_per_frame, int H, int D, int n_q) {
  if (n_frames < 1 || tokens_per_frame < 1 || H < 1 || D < 1 || n_q < 1) return 0;
  const int64_t T = (int64_t)n_frames * tokens_per_frame;
  const int64_t S = (T + nvfp4::kAttnTokensPerSplit - 1) / nvfp4::kAttnTokensPerSplit;
  return ((size_t)H * S * n_q * (D + 2) * sizeof(float) + 255) / 256 * 256;
}

nvfp4_status nvfp4_kv_attention_decode(const float* q, int n_q, const uint8_t* k_codes, const uint8_t* k_scales,
                                       const float* k_g, const float* k_mean, const uint8_t* v_codes,
                                       const uint8_t* v_scales, const float* v_g, int64_t pool_rows, int n_meta,
                                       const int64_t* frame_row, const int* frame_meta, int n_frames,
                                       int64_t tokens_per_frame, int H, int D, float scale, float* out,
                                       void* workspace, size_t workspace_bytes, void* stream) {
  if (n_q < 1 || n_q > nvfp4::kAttnMaxQ) return NVFP4_ESHAPE;
  if (D != 64 && D != 128) return NVFP4_ESHAPE;
  if (H < 1 || (int64_t)H * D > (1 << 24)) return NVFP4_ESHAPE;
  if (n_frames < 1 || n_frames > NVFP4_MAX_VIEW_FRAMES || tokens_per_frame < 1 || pool_rows < 1 || n_meta < 1)
    return NVFP4_ESHAPE;
  if (tokens_per_frame > ((int64_t)1 << 40) / NVFP4_MAX_VIEW_FRAMES) return NVFP4_ESHAPE;
  if ((int64_t)H * D > ((int64_t)1 << 46) / pool_rows) return NVFP4_ESHAPE;
  if (!q || !k_codes || !k_scales || !k_g || !v_codes || !v_scales || !v_g || !frame_row || !frame_meta || !out)
    return NVFP4_EINVAL;
  if (!nvfp4::aligned_to(k_codes, 16) || !nvfp4::aligned_to(v_codes, 16) || !nvfp4::aligned_to(q, 4) ||
      !nvfp4::aligned_to(k_g, 4) || !nvfp4::aligned_to(v_g, 4) || !nvfp4::aligned_to(out, 4) ||
      !nvfp4::aligned_to(k_mean, 16))
    return NVFP4_EALIGN;
  if (!workspace || !nvfp4::aligned_to(workspace, 256) ||
      workspace_bytes < nvfp4_kv_attention_workspace_bytes(n_frames, tokens_per_frame, H, D, n_q))
    return NVFP4_EWORKSPACE;
  nvfp4::AttnView view;
  std::memset(&view, 0, sizeof(view));
  for (int i = 0; i < n_frames; ++i) {  // every frame inside the pool, every slot inside the metadata
    if (frame_row[i] < 0 || frame_row[i] > pool_rows - tokens_per_frame) return NVFP4_ESHAPE;
    if (frame_meta[i] < 0 || frame_meta[i] >= n_meta) return NVFP4_ESHAPE;
    view.row[i] = frame_row[i];
    view.meta[i] = frame_meta[i];
  }
  const int64_t T = (int64_t)n_frames * tokens_per_frame;
  const int64_t S64 = (T + nvfp4::kAttnTokensPerSplit - 1) / nvfp4::kAttnTokensPerSplit;  // most splits
  if (S64 > 65535) return NVFP4_ESHAPE;
  float* part = static_cast<float*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
#define NVFP4_ATTN(DD, QQ)                                                                                     \
  e = nvfp4::launch_attn<DD, QQ>(q, k_codes, k_scales, k_g, k_mean, v_codes, v_scales, v_g, tokens_per_frame, T, \
                                 H, scale, part, view, out, st)
  if (D == 128) {
    if (n_q == 1) NVFP4_ATTN(128, 1); else if (n_q == 2) NVFP4_ATTN(128, 2);
    else if (n_q == 3) NVFP4_ATTN(128, 3); else NVFP4_ATTN(128, 4);
  } else {
    if (n_q == 1) NVFP4_ATTN(64, 1); else if (n_q == 2) NVFP4_ATTN(64, 2);
    else if (n_q == 3) NVFP4_ATTN(64, 3); else NVFP4_ATTN(64, 4);
  }
#undef NVFP4_ATTN
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

}  // extern "C"
