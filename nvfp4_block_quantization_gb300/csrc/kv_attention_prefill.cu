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
// view in fp32, all in base-2 units (times log2 e).  One pass over the view with
// an online maximum: per key tile, P'_it = bf16(2^(t_it - m_i) g_v[slot_t] / G)
// (G = max g_v over the view) is accumulated as O += P' V' in TMEM and
// l_i += sum_t 2^(t_it - m_i).  The running maximum m_i moves only when a tile's
// scores exceed it by more than 8 (then O's row and l are rescaled), so P' stays
// below 2^8 and rescaling is rare.  out = G O / l.  Beyond fp32 arithmetic only
// P' is rounded (bf16, relative 2^-9); 2^x is the hardware approximation
// (relative error below 2^-22).
//
// One CTA per (256 queries, head), 256 threads: all threads dequantize each
// 128-key tile into shared memory once for both 128-query halves; thread 0
// issues the MMAs of both halves (TMEM: S of half 0 and 1 in columns 0-255, O in
// 256-511); warp w owns query rows 32 (w % 4) .. of half w / 4 (its TMEM lane
// quadrant) for the softmax and the epilogue.  Operand tiles use the no-swizzle
// K-major layout of 8-row x 16-byte core matrices; the transposed V' tile pads
// its K stride to 144 bytes so that its stores spread over the banks.
#include <cstring>

#include "nvfp4.h"
#include "bulk.cuh"
#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int kPfTile = 128;           // queries per half, keys per tile
constexpr int kPfHalves = 2;           // query halves per CTA sharing each K'/V' tile
constexpr int kPfD = 128;              // head dimension
constexpr int kPfThreads = 128 * kPfHalves;
constexpr int kPfMaxSlots = 16;        // distinct pool slots in one view
constexpr uint32_t kLboStd = 128, kSboStd = 2048;  // [128 rows][256 B]: core matrices 128 B apart along K
constexpr uint32_t kLboV = 144, kSboV = 2304;      // the padded V' tile
constexpr int kTileStd = 32768;
constexpr int kTileV = 36864;
constexpr float kRescaleStep = 8.0f;  // base-2 units the running maximum may lag behind
// Q (2 halves), K', P' (2 halves), V'^T, q . mean per thread, key tables, barriers
constexpr int kPfSmem = kPfHalves * kTileStd + kTileStd + kPfHalves * kTileStd + kTileV + kPfMaxSlots * kPfThreads * 4 +
                        4 * kPfTile * 4 + 256;
static_assert(kPfSmem <= 232448, "shared memory per CTA");

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

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void pf_st32(uint32_t taddr, const float v[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      ::"r"(taddr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
      "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]),
      "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]),
      "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}

__device__ __forceinline__ void pf_mma_tile(uint32_t d_tmem, uint32_t a_smem, uint32_t a_lbo, uint32_t a_sbo,
                                            uint32_t b_smem, uint32_t b_lbo, uint32_t b_sbo, uint32_t idesc,
                                            bool accumulate) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {  // K = 128 in steps of 16 (two core matrices along K)
    const uint64_t da = pf_desc(a_smem + k * 2 * a_lbo, a_lbo, a_sbo);
    const uint64_t db = pf_desc(b_smem + k * 2 * b_lbo, b_lbo, b_sbo);
    const uint32_t acc = (accumulate || k > 0) ? 1u : 0u;
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(da), "l"(db), "r"(idesc), "r"(acc) : "memory");
  }
}

// The codes and scales of one thread's share of a key tile, loaded ahead of use:
// four (key, block) units of K' and four keys x one block of V'.  x packs the
// scale byte (bits 0-7) and 1 + the key's view slot (bits 8-15; 0: past the view).
struct PfCodes {
  uint2 kc[4];
  uint32_t kx[4];
  uint2 vc[4];
  uint32_t vx[4];
};

__device__ __forceinline__ void pf_load_codes(const PfView& view, const PfArgs& a, int h, int64_t t0, int kr, int kb,
                                              int kg, int vkg, int vb, int vh, PfCodes& c) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int64_t t = t0 + kr + 8 * (kg + 4 * j);
    c.kc[j] = make_uint2(0u, 0u);
    c.kx[j] = 0u;
    if (t < a.n_keys) {
      int64_t prow;
      int vs;
      key_location(view, a.L_f, t, prow, vs);
      const int64_t base = prow * a.H + h;
      c.kc[j] = *reinterpret_cast<const uint2*>(a.k_codes + base * (kPfD / 2) + kb * 8);
      c.kx[j] = (uint32_t)a.k_scales[base * (kPfD / 16) + kb] | ((uint32_t)(vs + 1) << 8);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int64_t t = t0 + 8 * vkg + 4 * vh + j;
    c.vc[j] = make_uint2(0u, 0u);
    c.vx[j] = 0u;
    if (t < a.n_keys) {
      int64_t prow;
      int vs;
      key_location(view, a.L_f, t, prow, vs);
      const int64_t base = prow * a.H + h;
      c.vc[j] = *reinterpret_cast<const uint2*>(a.v_codes + base * (kPfD / 2) + vb * 8);
      c.vx[j] = (uint32_t)a.v_scales[base * (kPfD / 16) + vb] | ((uint32_t)(vs + 1) << 8);
    }
  }
}

__global__ void __launch_bounds__(kPfThreads, 1) attn_prefill_kernel(const __grid_constant__ PfView view,
                                                                     PfArgs a) {
  extern __shared__ __align__(128) uint8_t pf_smem[];
  uint8_t* Qs = pf_smem;                          // Q of both halves, bf16 [query][d]
  uint8_t* Kb = Qs + kPfHalves * kTileStd;        // K' tile [key][d]
  uint8_t* Pb = Kb + kTileStd;                    // P' of both halves [query][key]
  uint8_t* Vt = Pb + kPfHalves * kTileStd;        // V'^T tile [d][key], padded
  float* qm = reinterpret_cast<float*>(Vt + kTileV);  // [view slot][thread]: scale log2e q . mean
  float* key_a = qm + kPfMaxSlots * kPfThreads;        // per key: scale log2e g_k
  float* key_gv = key_a + kPfTile;                      // g_v / G (0 past the view)
  int* key_qm = reinterpret_cast<int*>(key_gv + kPfTile);  // offset of the key's slot in qm, -1 past the view
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(key_qm + 2 * kPfTile);
  uint64_t* bar_pv = bar_s + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_pv + 1);
  float* Gs = reinterpret_cast<float*>(tmem_slot + 1);
  int* failed = reinterpret_cast<int*>(Gs + 1);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int half = warp >> 2, quad = warp & 3;
  const int h = blockIdx.y;
  const int64_t rowq = (int64_t)blockIdx.x * (kPfTile * kPfHalves) + tid;  // this thread's query
  const bool q_ok = rowq < a.n_q;
  const int H = a.H;
  const float slog2e = a.scale * 1.4426950408889634f;

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_pv, 1);
    *failed = 0;
    float G = 0.0f;
    for (int s = 0; s < view.n_vslots; ++s) G = fmaxf(G, a.v_g[view.slot[s]]);
    *Gs = G;
    mbar_fence_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // roles in the dequantization
  const int kr = tid & 7, kb = (tid >> 3) & 7, kg = tid >> 6;    // K': key row, block, group (0..3)
  const int vkg = tid & 15, vb = (tid >> 4) & 7, vh = tid >> 7;  // V'^T: key group of 8, block, half
  PfCodes pre;
  pf_load_codes(view, a, h, 0, kr, kb, kg, vkg, vb, vh, pre);  // the first tile, in flight during the prologue

  // Q rows (zeros past n_q) and scale log2e q . mean per view slot
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.q + (rowq * H + h) * kPfD);
    uint8_t* qs = Qs + half * kTileStd;
    const int r = tid & 127;
    uint32_t qw[64];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = q_ok ? ld_nc_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(qs + core_off(r, c, kLboStd, kSboStd)) = v;
      qw[4 * c] = v.x; qw[4 * c + 1] = v.y; qw[4 * c + 2] = v.z; qw[4 * c + 3] = v.w;
    }
    for (int s = 0; s < view.n_vslots; ++s) {
      float acc = 0.0f;
      if (a.k_mean) {
        const float4* mrow = reinterpret_cast<const float4*>(a.k_mean + ((int64_t)view.slot[s] * H + h) * kPfD);
#pragma unroll 4
        for (int c = 0; c < kPfD / 4; ++c) {
          const float4 mv = mrow[c];
          acc = __fmaf_rn(bf16lo(qw[2 * c]), mv.x, acc);
          acc = __fmaf_rn(bf16hi(qw[2 * c]), mv.y, acc);
          acc = __fmaf_rn(bf16lo(qw[2 * c + 1]), mv.z, acc);
          acc = __fmaf_rn(bf16hi(qw[2 * c + 1]), mv.w, acc);
        }
      }
      qm[s * kPfThreads + tid] = __fmul_rn(slog2e, acc);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
  const uint32_t t_S = tmem + half * 128 + lane_addr, t_O = tmem + 256 + half * 128 + lane_addr;
  const float G = *Gs;
  const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kPfTile >> 3) << 17) |
                         ((uint32_t)(kPfTile >> 4) << 24);  // bf16 x bf16 -> fp32, K-major, M = N = 128
  const int n_tiles = (int)((a.n_keys + kPfTile - 1) / kPfTile);
  uint32_t ph_s = 0, ph_pv = 0;
  uint8_t* Pmine = Pb + half * kTileStd;

  // K' of the prefetched tile into Kb, with its per-key factors
  auto decode_k = [&]() {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int key = kr + 8 * (kg + 4 * j);
      const uint32_t x = pre.kx[j];
      uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (x >> 8) decode_block_bf16(pre.kc[j], x & 0xFFu, w);
      if (kb == 0) {
        const int vs = (int)(x >> 8) - 1;
        key_a[key] = vs >= 0 ? __fmul_rn(slog2e, a.k_g[view.slot[vs]]) : 0.0f;
        key_qm[key] = vs >= 0 ? vs * kPfThreads : -1;
      }
      *reinterpret_cast<uint4*>(Kb + core_off(key, 2 * kb, kLboStd, kSboStd)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(Kb + core_off(key, 2 * kb + 1, kLboStd, kSboStd)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
  };
  // V'^T of the prefetched tile into Vt, with the keys' g_v / G
  auto decode_v = [&]() {
    uint32_t w[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t x = pre.vx[j];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[j][i] = 0u;
      if (x >> 8) decode_block_bf16(pre.vc[j], x & 0xFFu, w[j]);
      if (vb == 0) {
        const int vs = (int)(x >> 8) - 1;
        key_gv[8 * vkg + 4 * vh + j] = (vs >= 0 && G > 0.0f) ? __fdiv_rn(a.v_g[view.slot[vs]], G) : 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {  // channel 16 vb + i of the four keys: 8 bytes of V'^T's row
      uint32_t o[2];
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const uint32_t lo = (i & 1) ? (w[2 * p][i >> 1] >> 16) : (w[2 * p][i >> 1] & 0xFFFFu);
        const uint32_t hi = (i & 1) ? (w[2 * p + 1][i >> 1] >> 16) : (w[2 * p + 1][i >> 1] & 0xFFFFu);
        o[p] = lo | (hi << 16);
      }
      *reinterpret_cast<uint2*>(Vt + core_off(16 * vb + i, vkg, kLboV, kSboV) + 8 * vh) = make_uint2(o[0], o[1]);
    }
  };
  auto issue_s = [&]() {  // S = Q K'^T for both halves
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    for (int hh = 0; hh < kPfHalves; ++hh)
      pf_mma_tile(tmem + hh * 128, smem_u32(Qs + hh * kTileStd), kLboStd, kSboStd, smem_u32(Kb), kLboStd, kSboStd,
                  idesc, false);
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar_s))
                 : "memory");
  };

  // tile 0
  decode_k();
  decode_v();
  if (n_tiles > 1) pf_load_codes(view, a, h, kPfTile, kr, kb, kg, vkg, vb, vh, pre);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (tid == 0) issue_s();

  float m = -INFINITY, l = 0.0f;
  for (int tile = 0; tile < n_tiles; ++tile) {
    const bool more = tile + 1 < n_tiles;
    if (!mbar_wait(bar_s, ph_s)) atomicExch(failed, 1);
    ph_s ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // ---- scores (base 2), running maximum, weights of this thread's query row ----
    float t[kPfTile];
#pragma unroll
    for (int c = 0; c < 4; ++c) pf_ld32(t_S + 32 * c, t + 32 * c);
    float mt = -INFINITY;
#pragma unroll
    for (int k = 0; k < kPfTile; ++k) {
      const int off = key_qm[k];
      t[k] = off >= 0 ? __fmaf_rn(key_a[k], t[k], qm[off + tid]) : -INFINITY;
      mt = fmaxf(mt, t[k]);
    }
    const bool grow = mt > m + kRescaleStep;
    if (__any_sync(0xffffffffu, grow)) {
      const float m_new = grow ? mt : m;
      const float f = grow ? ex2_approx(m - m_new) : 1.0f;  // 0 for the first tile (m = -inf)
      l = __fmul_rn(l, f);
      m = m_new;
      if (tile > 0) {  // O holds earlier tiles (their MMAs have finished): scale this row, warp-wide
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          pf_ld32(t_O + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __fmul_rn(o[i], f);
          pf_st32(t_O + 32 * c, o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
    }
    float sum = 0.0f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      uint32_t o[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int k = 8 * c + 2 * p;
        const float p0 = ex2_approx(t[k] - m), p1 = ex2_approx(t[k + 1] - m);
        sum = __fadd_rn(sum, __fadd_rn(p0, p1));
        const __nv_bfloat162 b = __float22bfloat162_rn(make_float2(__fmul_rn(p0, key_gv[k]), __fmul_rn(p1, key_gv[k + 1])));
        o[p] = *reinterpret_cast<const uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(Pmine + core_off(tid & 127, c, kLboStd, kSboStd)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    l = __fadd_rn(l, sum);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    // ---- O += P' V' for both halves; meanwhile the next K' ----
    if (tid == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      for (int hh = 0; hh < kPfHalves; ++hh)
        pf_mma_tile(tmem + 256 + hh * 128, smem_u32(Pb + hh * kTileStd), kLboStd, kSboStd, smem_u32(Vt), kLboV, kSboV,
                    idesc, tile > 0);
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar_pv))
                   : "memory");
    }
    if (more) decode_k();  // K' is free: S of this tile has finished
    if (!mbar_wait(bar_pv, ph_pv)) atomicExch(failed, 1);
    ph_pv ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (more) {
      decode_v();  // V'^T and P' are free: P' V' has finished
      if (tile + 2 < n_tiles) pf_load_codes(view, a, h, (int64_t)(tile + 2) * kPfTile, kr, kb, kg, vkg, vb, vh, pre);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();  // every wait of this tile is over: all threads see the same flag below
    if (*reinterpret_cast<volatile int*>(failed)) break;
    if (more && tid == 0) issue_s();
  }
  // ---- out = G O / l ----
  if (!*reinterpret_cast<volatile int*>(failed)) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const float f = n_tiles > 0 ? __fdiv_rn(G, l) : 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float o[32];
      pf_ld32(t_O + 32 * c, o);
      if (q_ok) {
        float4* dst = reinterpret_cast<float4*>(a.out + (rowq * H + h) * kPfD + 32 * c);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__fmul_rn(o[4 * i], f), __fmul_rn(o[4 * i + 1], f), __fmul_rn(o[4 * i + 2], f),
                               __fmul_rn(o[4 * i + 3], f));
      }
    }
  } else if (tid == 0 && a.dev_status) {
    atomicOr(a.dev_status, NVFP4_DEV_TIMEOUT);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
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
  if (n_q < 1 || n_q > ((int64_t)1 << 30) * nvfp4::kPfTile) return NVFP4_ESHAPE;
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
  const int64_t q_per_cta = nvfp4::kPfTile * nvfp4::kPfHalves;
  const dim3 grid((unsigned)((n_q + q_per_cta - 1) / q_per_cta), (unsigned)H);
  nvfp4::attn_prefill_kernel<<<grid, nvfp4::kPfThreads, nvfp4::kPfSmem, static_cast<cudaStream_t>(stream)>>>(view, a);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

}  // extern "C"
