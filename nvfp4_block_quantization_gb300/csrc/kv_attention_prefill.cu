// kv_attention_prefill.cu -- attention of a block of query tokens over the NVFP4
// KV cache on the 5th-generation tensor cores (sm_103a): S = Q K^T and O = P V
// with tcgen05.mma, K and V dequantized tile by tile into shared memory.
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page), inference steps 7 and 9: each new chunk of tokens attends over
// the cached view (global sink, shot sink, rolling frames) read from the NVFP4
// KV cache.
//
// Per head h, query i and view token t (pool row frame_row[t / L_f] + t % L_f,
// slot frame_meta[t / L_f]), channel d in 16-channel block b:
//   k_td = Q_td E_k[t, b] g_k[slot] + mean[slot][h][d],   v_td = Q_td E_v[t, b] g_v[slot]
//   out[i][h] = sum_t softmax_t(scale * q_i . k_t) v_t
// An E2M1 value times an E4M3 value has at most 6 significant bits, so
// K'_td = Q_td E_k and V'_td = Q_td E_v are exact in bf16, and the queries are
// bf16.  The tensor cores take the exact products:
//   s_it = scale * (g_k[slot_t] * (q_i . K'_t) + q_i . mean[slot_t][h])
// with q . K' summed in fp32 by the MMA and q . mean computed once per slot of the
// view in fp32.  Two passes over the view per 128-query tile: the first finds
// each row's maximum m and sum l = sum_t exp(s - m); the second writes
//   P'_it = bf16(exp(s_it - m_i) * g_v[slot_t] / G)     (G = max g_v over the view)
// and accumulates O = P' V' in TMEM; out = G * O / l.  Beyond fp32 arithmetic
// only P' is rounded (bf16, relative 2^-9).
//
// One CTA per (128 queries, head), two CTAs per SM, 128 threads: all threads
// dequantize a 128-key tile into shared memory, one thread issues the MMAs,
// thread r owns query row r (TMEM lane r) for the softmax and the epilogue.
// Operand tiles use the no-swizzle K-major layout of 8-row x 16-byte core
// matrices; the transposed V' tile pads its K stride to 144 bytes so that its
// 16-byte stores from eight lanes hit eight different bank groups.
#include <cstring>

#include "nvfp4.h"
#include "bulk.cuh"
#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int kPfTile = 128;           // queries per CTA, keys per tile
constexpr int kPfD = 128;              // head dimension
constexpr int kPfThreads = 128;
constexpr int kPfMaxSlots = 16;        // distinct pool slots in one view
constexpr uint32_t kLboStd = 128, kSboStd = 2048;  // [128 rows][256 B]: core matrices 128 B apart along K
constexpr uint32_t kLboV = 144, kSboV = 2304;      // the padded V' tile
constexpr int kTileStd = 32768;
constexpr int kTileV = 36864;
constexpr int kPfSmem = 2 * kTileStd + kTileV + kPfMaxSlots * kPfTile * 4 + 3 * kPfTile * 4 + 256;

struct PfView {
  int64_t row[NVFP4_MAX_VIEW_FRAMES];
  int vslot[NVFP4_MAX_VIEW_FRAMES];  // index into slot[] of the frame's pool slot
  int slot[kPfMaxSlots];             // the view's distinct pool slots
  int n_vslots;
};

struct PfArgs {
  const uint16_t* q;  // bf16 [n_q][H][D]
  const uint8_t* k_codes;
  const uint8_t* k_scales;
  const float* k_g;
  const float* k_mean;  // [n_meta][H][D] or null
  const uint8_t* v_codes;
  const uint8_t* v_scales;
  const float* v_g;
  float* out;  // fp32 [n_q][H][D]
  int* dev_status;
  int64_t n_q, n_keys, L_f;
  int H;
  float scale;
};

__device__ __forceinline__ uint32_t core_off(uint32_t r, uint32_t chunk, uint32_t lbo, uint32_t sbo) {
  return (r >> 3) * sbo + chunk * lbo + (r & 7) * 16;
}

__device__ __forceinline__ uint64_t pf_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

__device__ __forceinline__ void pf_ld32(uint32_t taddr, float v[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 values of one block (8 code bytes, E4M3 scale byte) as exact bf16 pairs:
// w[j] holds channels 2j (low half) and 2j + 1.
__device__ __forceinline__ void decode_block_bf16(uint2 codes, uint32_t scale_byte, uint32_t w[8]) {
  const float E = e4m3_value(scale_byte);
  const uint32_t c[2] = {codes.x, codes.y};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t h2 = e2m1x2_to_f16x2((c[j >> 2] >> (8 * (j & 3))) & 0xFFu);
    const __nv_bfloat162 b = __float22bfloat162_rn(make_float2(__fmul_rn(f16lo(h2), E), __fmul_rn(f16hi(h2), E)));
    w[j] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// The view token of key t: its pool row and the view-slot index of its chunk.
__device__ __forceinline__ void key_location(const PfView& view, int64_t L_f, int64_t t, int64_t& row, int& vs) {
  const int64_t f = t / L_f;
  row = view.row[f] + (t - f * L_f);
  vs = view.vslot[f];
}

__global__ void __launch_bounds__(kPfThreads, 2) attn_prefill_kernel(const __grid_constant__ PfView view,
                                                                     PfArgs a) {
  extern __shared__ __align__(128) uint8_t pf_smem[];
  uint8_t* Qs = pf_smem;                     // Q tile, bf16 [query][d]
  uint8_t* KPs = Qs + kTileStd;              // K' tile [key][d] bf16, then P' [query][key] bf16
  uint8_t* Vt = KPs + kTileStd;              // V'^T tile [d][key] bf16, padded
  float* qm = reinterpret_cast<float*>(Vt + kTileV);  // [view slot][query]: q . mean
  float* key_gk = qm + kPfMaxSlots * kPfTile;         // per key of the tile: g_k
  float* key_gv = key_gk + kPfTile;                    // g_v / G
  int* key_vs = reinterpret_cast<int*>(key_gv + kPfTile);  // view slot of the key, -1 past the view
  uint64_t* bar = reinterpret_cast<uint64_t*>(key_vs + kPfTile);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  float* Gs = reinterpret_cast<float*>(tmem_slot + 1);
  int* failed = reinterpret_cast<int*>(Gs + 1);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = blockIdx.y;
  const int64_t q0 = (int64_t)blockIdx.x * kPfTile;
  const int H = a.H;
  const int64_t rowq = q0 + tid;  // this thread's query
  const bool q_ok = rowq < a.n_q;

  if (tid == 0) {
    mbar_init(bar, 1);
    *failed = 0;
    float G = 0.0f;
    for (int s = 0; s < view.n_vslots; ++s) G = fmaxf(G, a.v_g[view.slot[s]]);
    *Gs = G;
    mbar_fence_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Q tile: thread r writes query row r (zeros past n_q); q . mean per view slot
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.q + (rowq * H + h) * kPfD);
    float qf[kPfD];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = q_ok ? ld_nc_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(Qs + core_off(tid, c, kLboStd, kSboStd)) = v;
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        qf[8 * c + 2 * j] = bf16lo(w[j]);
        qf[8 * c + 2 * j + 1] = bf16hi(w[j]);
      }
    }
    for (int s = 0; s < view.n_vslots; ++s) {
      float acc = 0.0f;
      if (a.k_mean) {
        const float* mrow = a.k_mean + ((int64_t)view.slot[s] * H + h) * kPfD;
#pragma unroll 8
        for (int d = 0; d < kPfD; ++d) acc = __fmaf_rn(qf[d], mrow[d], acc);
      }
      qm[s * kPfTile + tid] = acc;
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_S = tmem, t_O = tmem + 128;
  const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
  const float G = *Gs;
  const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kPfTile >> 3) << 17) |
                         ((uint32_t)(kPfTile >> 4) << 24);  // bf16 x bf16 -> fp32, K-major, M = N = 128
  const int n_tiles = (int)((a.n_keys + kPfTile - 1) / kPfTile);
  uint32_t phase = 0;

  // thread roles in the dequantization (all 128 threads)
  const int kr = tid & 7, kb = (tid >> 3) & 7, kg2 = tid >> 6;  // K' tile: key row, block, key-group parity
  const int vkg = tid & 15, vb = tid >> 4;                       // V'^T tile: key group of 8, block

  float m = -INFINITY, l = 0.0f;

  for (int pass = 0; pass < 2; ++pass) {
    for (int tile = 0; tile < n_tiles; ++tile) {
      const int64_t t0 = (int64_t)tile * kPfTile;
      // ---- K' tile: keys kr + 8 (kg2 + 2 j), block kb ----
#pragma unroll 2
      for (int j = 0; j < 8; ++j) {
        const int key = kr + 8 * (kg2 + 2 * j);
        const int64_t t = t0 + key;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (t < a.n_keys) {
          int64_t prow;
          int vs;
          key_location(view, a.L_f, t, prow, vs);
          const int64_t base = prow * H + h;
          const uint2 codes = *reinterpret_cast<const uint2*>(a.k_codes + base * (kPfD / 2) + kb * 8);
          decode_block_bf16(codes, a.k_scales[base * (kPfD / 16) + kb], w);
          if (kb == 0) {
            key_gk[key] = a.k_g[view.slot[vs]];
            key_vs[key] = vs;
          }
        } else if (kb == 0) {
          key_gk[key] = 0.0f;
          key_vs[key] = -1;
        }
        *reinterpret_cast<uint4*>(KPs + core_off(key, 2 * kb, kLboStd, kSboStd)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(KPs + core_off(key, 2 * kb + 1, kLboStd, kSboStd)) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      // ---- V'^T tile (second pass): keys 8 vkg .. 8 vkg + 7, block vb ----
      if (pass == 1) {
        uint32_t w[8][8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int key = 8 * vkg + j;
          const int64_t t = t0 + key;
#pragma unroll
          for (int i = 0; i < 8; ++i) w[j][i] = 0u;
          if (t < a.n_keys) {
            int64_t prow;
            int vs;
            key_location(view, a.L_f, t, prow, vs);
            const int64_t base = prow * H + h;
            const uint2 codes = *reinterpret_cast<const uint2*>(a.v_codes + base * (kPfD / 2) + vb * 8);
            decode_block_bf16(codes, a.v_scales[base * (kPfD / 16) + vb], w[j]);
            if (vb == 0) key_gv[key] = G > 0.0f ? __fdiv_rn(a.v_g[view.slot[vs]], G) : 0.0f;
          } else if (vb == 0) {
            key_gv[key] = 0.0f;
          }
        }
        // channel 16 vb + i of keys 8 vkg .. 8 vkg + 7: one 16-byte chunk of V'^T's row
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t o[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const uint32_t lo = (i & 1) ? (w[2 * p][i >> 1] >> 16) : (w[2 * p][i >> 1] & 0xFFFFu);
            const uint32_t hi = (i & 1) ? (w[2 * p + 1][i >> 1] >> 16) : (w[2 * p + 1][i >> 1] & 0xFFFFu);
            o[p] = lo | (hi << 16);
          }
          *reinterpret_cast<uint4*>(Vt + core_off(16 * vb + i, vkg, kLboV, kSboV)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncthreads();
      // ---- S = Q K'^T ----
      if (tid == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t qa = smem_u32(Qs), ka = smem_u32(KPs);
#pragma unroll
        for (int k = 0; k < kPfD / 16; ++k) {
          const uint64_t da = pf_desc(qa + k * 2 * kLboStd, kLboStd, kSboStd);
          const uint64_t db = pf_desc(ka + k * 2 * kLboStd, kLboStd, kSboStd);
          const uint32_t acc = k > 0 ? 1u : 0u;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
              ::"r"(t_S), "l"(da), "l"(db), "r"(idesc), "r"(acc) : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                     : "memory");
      }
      if (!mbar_wait(bar, phase)) atomicExch(failed, 1);
      phase ^= 1u;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // ---- scores of this thread's query row ----
      float s[kPfTile];
#pragma unroll
      for (int c = 0; c < 4; ++c) pf_ld32(t_S + lane_addr + 32 * c, s + 32 * c);
#pragma unroll
      for (int k = 0; k < kPfTile; ++k) {
        const int vs = key_vs[k];
        s[k] = vs >= 0 ? __fmul_rn(a.scale, __fadd_rn(__fmul_rn(key_gk[k], s[k]), qm[vs * kPfTile + tid]))
                       : -INFINITY;
      }
      if (pass == 0) {
        float mt = m;
#pragma unroll
        for (int k = 0; k < kPfTile; ++k) mt = fmaxf(mt, s[k]);
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < kPfTile; ++k) sum = __fadd_rn(sum, expf(s[k] - mt));
        l = __fadd_rn(__fmul_rn(l, expf(m - mt)), sum);
        m = mt;
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();  // the next tile's dequantization rewrites K' and the key arrays
      } else {
        // P' row of this query (K' has been consumed by the finished MMAs)
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          uint32_t o[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int k = 8 * c + 2 * p;
            const float p0 = __fmul_rn(expf(s[k] - m), key_gv[k]);
            const float p1 = __fmul_rn(expf(s[k + 1] - m), key_gv[k + 1]);
            const __nv_bfloat162 b = __float22bfloat162_rn(make_float2(p0, p1));
            o[p] = *reinterpret_cast<const uint32_t*>(&b);
          }
          *reinterpret_cast<uint4*>(KPs + core_off(tid, c, kLboStd, kSboStd)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        // ---- O += P' V' ----
        if (tid == 0) {
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t pa = smem_u32(KPs), va = smem_u32(Vt);
#pragma unroll
          for (int k = 0; k < kPfTile / 16; ++k) {
            const uint64_t da = pf_desc(pa + k * 2 * kLboStd, kLboStd, kSboStd);
            const uint64_t db = pf_desc(va + k * 2 * kLboV, kLboV, kSboV);
            const uint32_t acc = (tile > 0 || k > 0) ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                ::"r"(t_O), "l"(da), "l"(db), "r"(idesc), "r"(acc) : "memory");
          }
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                       : "memory");
        }
        if (!mbar_wait(bar, phase)) atomicExch(failed, 1);
        phase ^= 1u;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      }
      if (*reinterpret_cast<volatile int*>(failed)) break;
    }
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(failed)) break;
  }
  // ---- out = G O / l ----
  if (!*reinterpret_cast<volatile int*>(failed)) {
    float o[kPfD];
#pragma unroll
    for (int c = 0; c < 4; ++c) pf_ld32(t_O + lane_addr + 32 * c, o + 32 * c);
    if (q_ok) {
      const float f = n_tiles > 0 ? __fdiv_rn(G, l) : 0.0f;
      float4* dst = reinterpret_cast<float4*>(a.out + (rowq * H + h) * kPfD);
#pragma unroll
      for (int c = 0; c < kPfD / 4; ++c)
        dst[c] = make_float4(__fmul_rn(o[4 * c], f), __fmul_rn(o[4 * c + 1], f), __fmul_rn(o[4 * c + 2], f),
                             __fmul_rn(o[4 * c + 3], f));
    }
  } else if (tid == 0 && a.dev_status) {
    atomicOr(a.dev_status, NVFP4_DEV_TIMEOUT);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem) : "memory");
}

bool pf_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace nvfp4

extern "C" {

nvfp4_status nvfp4_kv_attention_prefill(const void* q_bf16, int64_t n_q, const uint8_t* k_codes,
                                        const uint8_t* k_scales, const float* k_g, const float* k_mean,
                                        const uint8_t* v_codes, const uint8_t* v_scales, const float* v_g,
                                        int64_t pool_rows, int n_meta, const int64_t* frame_row,
                                        const int* frame_meta, int n_frames, int64_t tokens_per_frame, int H, int D,
                                        float scale, float* out, int* dev_status, void* stream) {
  if (D != nvfp4::kPfD || H < 1 || H > 65535) return NVFP4_ESHAPE;
  if (n_q < 1 || n_q > ((int64_t)1 << 31) * nvfp4::kPfTile) return NVFP4_ESHAPE;
  if (n_frames < 1 || n_frames > NVFP4_MAX_VIEW_FRAMES || tokens_per_frame < 1 || pool_rows < 1 || n_meta < 1)
    return NVFP4_ESHAPE;
  if (tokens_per_frame > ((int64_t)1 << 40) / NVFP4_MAX_VIEW_FRAMES) return NVFP4_ESHAPE;
  if ((int64_t)H * D > ((int64_t)1 << 46) / pool_rows || (int64_t)H * D > ((int64_t)1 << 46) / n_q)
    return NVFP4_ESHAPE;
  if (!q_bf16 || !k_codes || !k_scales || !k_g || !v_codes || !v_scales || !v_g || !frame_row || !frame_meta || !out)
    return NVFP4_EINVAL;
  if (!nvfp4::pf_aligned(q_bf16, 16) || !nvfp4::pf_aligned(k_codes, 8) || !nvfp4::pf_aligned(v_codes, 8) ||
      !nvfp4::pf_aligned(k_g, 4) || !nvfp4::pf_aligned(v_g, 4) || !nvfp4::pf_aligned(out, 16) ||
      !nvfp4::pf_aligned(k_mean, 4) || !nvfp4::pf_aligned(dev_status, 4))
    return NVFP4_EALIGN;
  nvfp4::PfView view;
  std::memset(&view, 0, sizeof(view));
  for (int i = 0; i < n_frames; ++i) {  // every frame inside the pool, every slot inside the metadata
    if (frame_row[i] < 0 || frame_row[i] > pool_rows - tokens_per_frame) return NVFP4_ESHAPE;
    if (frame_meta[i] < 0 || frame_meta[i] >= n_meta) return NVFP4_ESHAPE;
    view.row[i] = frame_row[i];
    int vs = 0;
    while (vs < view.n_vslots && view.slot[vs] != frame_meta[i]) ++vs;
    if (vs == view.n_vslots) {
      if (view.n_vslots == nvfp4::kPfMaxSlots) return NVFP4_ESHAPE;  // too many chunks in one view
      view.slot[view.n_vslots++] = frame_meta[i];
    }
    view.vslot[i] = vs;
  }
  nvfp4::PfArgs a;
  a.q = static_cast<const uint16_t*>(q_bf16);
  a.k_codes = k_codes;
  a.k_scales = k_scales;
  a.k_g = k_g;
  a.k_mean = k_mean;
  a.v_codes = v_codes;
  a.v_scales = v_scales;
  a.v_g = v_g;
  a.out = out;
  a.dev_status = dev_status;
  a.n_q = n_q;
  a.n_keys = (int64_t)n_frames * tokens_per_frame;
  a.L_f = tokens_per_frame;
  a.H = H;
  a.scale = scale;
  if (cudaFuncSetAttribute(nvfp4::attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, nvfp4::kPfSmem) !=
      cudaSuccess)
    return NVFP4_ECUDA;
  const dim3 grid((unsigned)((n_q + nvfp4::kPfTile - 1) / nvfp4::kPfTile), (unsigned)H);
  nvfp4::attn_prefill_kernel<<<grid, nvfp4::kPfThreads, nvfp4::kPfSmem, static_cast<cudaStream_t>(stream)>>>(view, a);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

}  // extern "C"
