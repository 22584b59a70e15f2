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
// One CTA per (256 queries, head), 18 warps in roles, every hand-off an mbarrier; keys in
// tiles of 64:
//   warps 0-3, 4-7    softmax of query half 0 / 1: thread r owns query row r of its half (TMEM
//                     lane r); per tile, the maximum of its 64 scores, then P' (bf16 pairs)
//                     written into TMEM over the S columns already read; O rescaled when needed.
//                     A tile whose keys share one view slot (most of them) takes the slot's
//                     factors as scalars and the extreme raw S with 3-input max, and forms P'
//                     in packed fp32x2 arithmetic;
//   warps 8, 9, 12, 13  K' decoders (sub-partitions 0 and 1), warps 10, 11, 16, 17 V'
//                     decoders: thread k owns key k of every other tile, loads its
//                     72 code and scale bytes a tile ahead, and writes its 128 bf16 channels,
//                     E2M1 magnitudes taken from byte-permute tables and multiplied by the block
//                     scale in bf16x2 (exact); the K' decoders also write each key's factors;
//   warps 14, 15      one thread per half (sub-partitions 2 and 3, beside the lighter V'
//                     decoders) issues that half's MMAs: S_h(j + 2) = Q_h K'(j + 2)^T
//                     into the S buffer that P'_h(j) V'(j) has just read, so S stays one tile
//                     ahead of the softmax.
// TMEM per half: two 64-column S buffers (P' over the first 32 columns of each) and a
// 128-column O.  K' and V' share one [key][d] layout of 8-row x 16-byte core matrices, four
// buffers each: K-major for S = Q K'^T, MN-major for P' V'.  Every wait is bounded; a timeout is
// reported in the status word and the CTA drains its MMAs before freeing TMEM.
// With a workspace, the units of the last, partial wave of CTAs run as two CTAs over the two
// halves of the keys; prefill_merge_kernel combines them.
#include <cstring>

#include "nvfp4.h"
#include "bulk.cuh"
#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int kPfQTile = 128;          // queries per half: the TMEM lanes
constexpr int kPfKTile = 64;           // keys per tile
constexpr int kPfHalves = 2;           // query halves per CTA sharing each K'/V' tile
constexpr int kPfRows = kPfQTile * kPfHalves;
constexpr int kPfD = 128;              // head dimension
constexpr int kPfSoftmaxWarps = 4 * kPfHalves;
constexpr int kPfDecodeWarps = 8;      // K' on sub-partitions 0 and 1, V' on 2 and 3
constexpr int kPfMmaWarp = kPfSoftmaxWarps + kPfDecodeWarps;  // the warp that allocates TMEM
constexpr int kPfThreads = 32 * (kPfMmaWarp + kPfHalves);  // plus one MMA-issuing warp per half
constexpr int kPfMaxSlots = 16;        // distinct pool slots in one view
constexpr int kPfBufs = 4;             // K' and V' tile buffers each
constexpr int kPfKeyBufs = 8;          // key-factor table buffers
constexpr uint32_t kLboStd = 128, kSboStd = 2048;  // [rows][256 B]: core matrices 128 B apart along d
// V' [key][d] as an MN-major B operand: LBO = 2048 between groups of 8 keys (the K direction),
// SBO = 128 between groups of 8 channels (the N direction).
constexpr uint32_t kLboV = 2048, kSboV = 128;
constexpr int kTileQ = kPfQTile * kPfD * 2;   // one half's Q, bf16
constexpr int kTileKV = kPfKTile * kPfD * 2;  // one K' or V' tile, bf16
constexpr float kRescaleStep = 8.0f;  // base-2 units the running maximum may lag behind
// Q (2 halves), K' and V' (4 buffers each), q . mean per row and slot, key tables, slot tables,
// barriers; P' lives in TMEM over the S it was computed from
constexpr int kPfSmem = kPfHalves * kTileQ + 2 * kPfBufs * kTileKV + kPfMaxSlots * kPfRows * 4 +
                        kPfKeyBufs * 3 * kPfKTile * 4 + 2 * kPfMaxSlots * 4 + 512;  // barriers etc. in the last 512 B
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
  // Key split of the last wave: units (head h, query tile qt) are numbered h * q_tiles + qt.
  // Units below n_full run whole; each later unit runs as two CTAs over keys [0, t_mid) and
  // [t_mid, n_keys), which write G O / l, m and l of their rows to `part` for the merge kernel.
  float* part;
  int64_t q_tiles, n_full, t_mid;
};

// One split half's rows in the workspace: out [256][128] fp32, then m [256] and l [256].
constexpr int64_t kPfPartFloats = (int64_t)kPfRows * kPfD + 2 * kPfRows;

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

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Issues a 32-column TMEM load without waiting for it (pf_wait_ld completes it).
__device__ __forceinline__ void pf_ld32_issue(uint32_t taddr, uint32_t r[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Marks 32 registers as written here, so that no use of them moves above a preceding wait::ld.
__device__ __forceinline__ void pf_tie32(uint32_t r[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                 "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]),
                 "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

__device__ __forceinline__ void pf_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 16 values of one block (8 code bytes, E4M3 scale byte) as exact bf16 pairs:
// w[j] holds channels 2j (low half) and 2j + 1.  No conversion instructions: the bf16 bytes of
// the eight E2M1 magnitudes (0, 0.5, 1, 1.5, 2, 3, 4, 6 = 0x0000, 0x3F00, 0x3F80, 0x3FC0, 0x4000,
// 0x4040, 0x4080, 0x40C0) are two 8-entry byte tables, read by one byte permute per four values;
// the code's sign bit is or-ed into the high byte; one packed bf16 multiply by the block scale E
// ends it.  |E2M1| has at most 2 significant bits and E4M3 at most 4, so the product is exact in
// bf16 and lies in [2^-10, 2688], inside its normal range.  A block is two words.
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t scale_byte) {  // E in both halves, exact in bf16
  return __byte_perm(__float_as_uint(e4m3_value(scale_byte)), 0u, 0x3232);
}

// Eight codes (one 32-bit word, code 2j + k in bits 8j + 4k .. + 3) times E2 -> w[0..3].
__device__ __forceinline__ void decode_word_bf16(uint32_t cw, uint32_t E2, uint32_t w[4]) {
  const uint32_t mag = cw & 0x77777777u, s4 = cw << 4;  // s4: even codes' sign bits at bit 7 of a byte
#pragma unroll
  for (int hq = 0; hq < 2; ++hq) {  // codes 4 hq .. 4 hq + 3
    const uint32_t sel = hq ? (mag >> 16) : mag;
    const uint32_t hi = __byte_perm(0x3F3F3F00u, 0x40404040u, sel);
    const uint32_t lo = __byte_perm(0xC0800000u, 0xC0804000u, sel);
    const uint32_t hs = hi | (__byte_perm(s4, cw, hq ? 0x7362 : 0x5140) & 0x80808080u);
    w[2 * hq] = bf16x2_mul(__byte_perm(lo, hs, 0x5140), E2);
    w[2 * hq + 1] = bf16x2_mul(__byte_perm(lo, hs, 0x7362), E2);
  }
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

__device__ __forceinline__ void pf_st16(uint32_t taddr, const uint32_t v[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// One tcgen05.mma of kind f16; `acc` 0 overwrites D.  An operand given as a 64-bit value is a
// shared-memory descriptor; as a 32-bit value, a TMEM address.
__device__ __forceinline__ void pf_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void pf_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc) : "memory");
}

// The descriptors of one K step follow from the first by adding the step's byte offset / 16 to
// the address field (bits 0-13): shared-memory addresses stay below 2^18, so it cannot carry.

// O (+)= P' V' with P' (A, bf16 pairs: lane = query row, column c = keys 2c and 2c + 1) in TMEM.
__device__ __forceinline__ void pf_mma_tile_ta(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem, uint32_t b_lbo,
                                               uint32_t b_sbo, uint32_t idesc, bool accumulate) {
  const uint64_t db = pf_desc(b_smem, b_lbo, b_sbo);
#pragma unroll
  for (int k = 0; k < kPfKTile / 16; ++k)  // K = the tile's keys in steps of 16 (8 TMEM columns of A, two core matrices of B)
    pf_mma_ta(d_tmem, a_tmem + 8 * k, db + (uint64_t)((k * 2 * b_lbo) >> 4), idesc, (accumulate || k > 0) ? 1u : 0u);
}

__device__ __forceinline__ void pf_mma_tile(uint32_t d_tmem, uint32_t a_smem, uint32_t a_lbo, uint32_t a_sbo,
                                            uint32_t b_smem, uint32_t b_lbo, uint32_t b_sbo, uint32_t idesc,
                                            bool accumulate) {
  const uint64_t da = pf_desc(a_smem, a_lbo, a_sbo), db = pf_desc(b_smem, b_lbo, b_sbo);
#pragma unroll
  for (int k = 0; k < kPfD / 16; ++k)  // K = d = 128 in steps of 16 (two core matrices along K)
    pf_mma(d_tmem, da + (uint64_t)((k * 2 * a_lbo) >> 4), db + (uint64_t)((k * 2 * b_lbo) >> 4), idesc,
           (accumulate || k > 0) ? 1u : 0u);
}

__device__ __forceinline__ bool pf_wait_warp(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ void pf_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__global__ void __launch_bounds__(kPfThreads, 1) attn_prefill_kernel(const __grid_constant__ PfView view,
                                                                     PfArgs a) {
  extern __shared__ __align__(128) uint8_t pf_smem[];
  uint8_t* Qs = pf_smem;                          // Q of both halves, bf16 [query][d]
  uint8_t* Kb = Qs + kPfHalves * kTileQ;          // K' tiles [buffer][key][d]
  uint8_t* Vb = Kb + kPfBufs * kTileKV;           // V' tiles [buffer][key][d]
  float* qm = reinterpret_cast<float*>(Vb + kPfBufs * kTileKV);  // [view slot][row]: scale log2e q . mean
  float* key_a = qm + kPfMaxSlots * kPfRows;               // [table buffer][key]: scale log2e g_k
  float* key_gv = key_a + kPfKeyBufs * kPfKTile;           // [table buffer][key]: g_v / G (0 past the view)
  int* key_off = reinterpret_cast<int*>(key_gv + kPfKeyBufs * kPfKTile);  // slot offset in qm, -1 past the view
  float* slot_a = reinterpret_cast<float*>(key_off + kPfKeyBufs * kPfKTile);
  float* slot_gv = slot_a + kPfMaxSlots;
  // Tile j uses K'/V' buffer j % 4 and, in each half, S buffer j % 2.  A barrier completes one phase
  // per use of its buffer, and every wait names the phase it needs by its parity.
  uint64_t* bar = reinterpret_cast<uint64_t*>(slot_gv + kPfMaxSlots);
  uint64_t* k_full = bar;        // [buffer] K'(j) and its key tables written   (2 decode warps)
  uint64_t* k_free = bar + 4;    // [buffer] both S(j) MMAs have read K'(j)      (a commit per half)
  uint64_t* v_full = bar + 8;    // [buffer] V'(j) written                       (2 decode warps)
  uint64_t* v_free = bar + 12;   // [buffer] both P' V'(j) MMAs have read V'(j)  (a commit per half)
  uint64_t* s_full = bar + 16;   // [half][S buffer] S(j) in TMEM                (commit)
  uint64_t* p_full = bar + 20;   // [half][S buffer] P'(j) in TMEM               (4 softmax warps)
  uint64_t* o_done = bar + 24;   // [half][S buffer] P' V'(j) added to O         (commit)
  uint64_t* drain = bar + 28;    // every MMA issued has finished                (a commit per half)
  uint64_t* key_ready = bar + 29;  // [table buffer] key factors of tile j written (2 decode warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 29 + kPfKeyBufs);
  float* Gs = reinterpret_cast<float*>(tmem_slot + 1);
  int* failed = reinterpret_cast<int*>(Gs + 1);
  volatile int* vfailed = failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t bid = blockIdx.x;
  const int64_t unit = bid < a.n_full ? bid : a.n_full + (bid - a.n_full) / 2;
  const int part = bid < a.n_full ? -1 : (int)((bid - a.n_full) & 1);  // -1: the whole view
  const int h = (int)(unit / a.q_tiles);
  const int64_t qt = unit - (int64_t)h * a.q_tiles;
  const int64_t t_begin = part == 1 ? a.t_mid : 0, t_end = part == 0 ? a.t_mid : a.n_keys;  // this CTA's keys
  const int H = a.H;
  const float slog2e = a.scale * 1.4426950408889634f;
  const int n_tiles = (int)((t_end - t_begin + kPfKTile - 1) / kPfKTile);

  if (tid == 0) {
    for (int i = 0; i < kPfBufs; ++i) {
      mbar_init(&k_full[i], 2);
      mbar_init(&k_free[i], kPfHalves);
      mbar_init(&v_full[i], 2);
      mbar_init(&v_free[i], kPfHalves);
    }
    for (int i = 0; i < 2 * kPfHalves; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(drain, kPfHalves);
    for (int i = 0; i < kPfKeyBufs; ++i) mbar_init(&key_ready[i], 2);
    *failed = 0;
    float G = 0.0f;
    for (int s = 0; s < view.n_vslots; ++s) G = fmaxf(G, a.v_g[view.slot[s]]);
    *Gs = G;
    for (int s = 0; s < view.n_vslots; ++s) {
      slot_a[s] = __fmul_rn(slog2e, a.k_g[view.slot[s]]);
      slot_gv[s] = G > 0.0f ? __fdiv_rn(a.v_g[view.slot[s]], G) : 0.0f;
    }
    mbar_fence_init();
  }
  if (warp == kPfMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // softmax threads: their Q row (zeros past n_q) and scale log2e q . mean per view slot
  const int64_t rowq = qt * kPfRows + tid;
  if (warp < kPfSoftmaxWarps) {
    const bool q_ok = rowq < a.n_q;
    const uint4* src = reinterpret_cast<const uint4*>(a.q + (rowq * H + h) * kPfD);
    uint8_t* qs = Qs + (tid >> 7) * kTileQ;
    uint32_t qw[64];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = q_ok ? ld_nc_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(qs + core_off(tid & 127, c, kLboStd, kSboStd)) = v;
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
      qm[s * kPfRows + tid] = __fmul_rn(slog2e, acc);
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q is an MMA operand
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  const float G = *Gs;

  if (warp < kPfSoftmaxWarps) {
    // ================= softmax of one query half =================
    const int half = warp >> 2;
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_half = tmem + half * 256 + lane_addr, t_O = t_half + 128;  // S buffers at +0, +64; O at +128
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int sb = j & 1, tb = j % kPfKeyBufs;
      const uint32_t t_S = t_half + 64 * sb;
      const float* ka = key_a + tb * kPfKTile;
      const float* kgv = key_gv + tb * kPfKTile;
      const int* koff = key_off + tb * kPfKTile;
      // a tile whose keys are all in the view and in one slot (with frames of at least 64 tokens
      // its first and last key decide it): the slot's factors are scalars
      if (!pf_wait_warp(&key_ready[tb], (j / kPfKeyBufs) & 1)) { ok = false; break; }
      const int o_first = koff[0], o_last = koff[kPfKTile - 1];
      const int uvs = (a.L_f >= kPfKTile && o_first == o_last && o_first >= 0) ? o_first / kPfRows : -1;
      const float ua = uvs >= 0 ? slot_a[uvs] : 0.0f, ub = uvs >= 0 ? qm[uvs * kPfRows + tid] : 0.0f;
      const float ugv = uvs >= 0 ? slot_gv[uvs] : 0.0f;
      if (!pf_wait_warp(&s_full[2 * half + sb], (j >> 1) & 1)) { ok = false; break; }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // pass 1: the tile's maximum of t = (scale log2e) (g_k S + q . mean)
      float mt = -INFINITY;
      if (uvs >= 0) {
        // one slot: t = fmaf(ua, S, ub) is monotonic in S (non-decreasing for ua >= 0), so the
        // maximum is fmaf(ua, S*, ub) with S* the largest S (the smallest for ua < 0)
        const bool up = ua >= 0.0f;
        float e0 = up ? -INFINITY : INFINITY, e1 = e0, e2 = e0, e3 = e0;
        uint32_t r0[32], r1[32];
        pf_ld32_issue(t_S, r0);
        pf_ld32_issue(t_S + 32, r1);
        pf_wait_ld();
        pf_tie32(r0);
        pf_tie32(r1);
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          if (up) {
            e0 = fmax3(e0, __uint_as_float(r0[i]), __uint_as_float(r0[i + 1]));
            e1 = fmax3(e1, __uint_as_float(r0[i + 2]), __uint_as_float(r0[i + 3]));
            e2 = fmax3(e2, __uint_as_float(r0[i + 4]), __uint_as_float(r0[i + 5]));
            e3 = fmax3(e3, __uint_as_float(r0[i + 6]), __uint_as_float(r0[i + 7]));
            e0 = fmax3(e0, __uint_as_float(r1[i]), __uint_as_float(r1[i + 1]));
            e1 = fmax3(e1, __uint_as_float(r1[i + 2]), __uint_as_float(r1[i + 3]));
            e2 = fmax3(e2, __uint_as_float(r1[i + 4]), __uint_as_float(r1[i + 5]));
            e3 = fmax3(e3, __uint_as_float(r1[i + 6]), __uint_as_float(r1[i + 7]));
          } else {
            e0 = fmin3(e0, __uint_as_float(r0[i]), __uint_as_float(r0[i + 1]));
            e1 = fmin3(e1, __uint_as_float(r0[i + 2]), __uint_as_float(r0[i + 3]));
            e2 = fmin3(e2, __uint_as_float(r0[i + 4]), __uint_as_float(r0[i + 5]));
            e3 = fmin3(e3, __uint_as_float(r0[i + 6]), __uint_as_float(r0[i + 7]));
            e0 = fmin3(e0, __uint_as_float(r1[i]), __uint_as_float(r1[i + 1]));
            e1 = fmin3(e1, __uint_as_float(r1[i + 2]), __uint_as_float(r1[i + 3]));
            e2 = fmin3(e2, __uint_as_float(r1[i + 4]), __uint_as_float(r1[i + 5]));
            e3 = fmin3(e3, __uint_as_float(r1[i + 6]), __uint_as_float(r1[i + 7]));
          }
        }
        mt = __fmaf_rn(ua, up ? fmax3(e0, e1, fmaxf(e2, e3)) : fmin3(e0, e1, fminf(e2, e3)), ub);
      } else {
#pragma unroll 1
        for (int c = 0; c < kPfKTile / 32; ++c) {
          float t[32];
          pf_ld32(t_S + 32 * c, t);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int k = 32 * c + i, off = koff[k];
            if (off >= 0) mt = fmaxf(mt, __fmaf_rn(ka[k], t[i], qm[off + tid]));
          }
        }
      }
      const bool grow = mt > m + kRescaleStep;
      if (__any_sync(0xffffffffu, grow)) {
        const float m_new = grow ? mt : m;
        const float f = grow ? ex2_approx(m - m_new) : 1.0f;  // 0 for the first tile (m = -inf)
        l = __fmul_rn(l, f);
        m = m_new;
        if (j > 0) {  // O holds tiles up to j - 1: once P' V'(j - 1) is in, scale this row
          if (!pf_wait_warp(&o_done[2 * half + (sb ^ 1)], ((j - 1) >> 1) & 1)) { ok = false; break; }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float o[32];
            pf_ld32(t_O + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __fmul_rn(o[i], f);
            pf_st32(t_O + 32 * c, o);
          }
        }
      }
      // pass 2: P' = bf16(2^(t - m) g_v / G) into TMEM over S (columns already read), and l
      float2 sa = make_float2(0.0f, 0.0f), sc = sa;
      if (uvs >= 0) {  // pairs of keys in packed fp32x2 arithmetic; t - m = fmaf(ua, S, ub - m)
        const float2 ua2 = make_float2(ua, ua), c2 = make_float2(__fsub_rn(ub, m), __fsub_rn(ub, m));
        const float2 g2 = make_float2(ugv, ugv);
#pragma unroll 1
        for (int c = 0; c < kPfKTile / 32; ++c) {
          float t[32];
          pf_ld32(t_S + 32 * c, t);
          uint32_t pw[16];
#pragma unroll
          for (int p = 0; p < 16; ++p) {
            const float2 x = __ffma2_rn(make_float2(t[2 * p], t[2 * p + 1]), ua2, c2);
            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            if (p & 1) sc = __fadd2_rn(sc, e); else sa = __fadd2_rn(sa, e);
            const float2 q = __fmul2_rn(e, g2);
            const __nv_bfloat162 b = __float22bfloat162_rn(q);
            pw[p] = *reinterpret_cast<const uint32_t*>(&b);
          }
          pf_st16(t_S + 16 * c, pw);  // keys 32 c .. 32 c + 31: columns 16 c .. 16 c + 15, S there already read
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kPfKTile / 32; ++c) {
          float t[32];
          pf_ld32(t_S + 32 * c, t);
          uint32_t pw[16];
#pragma unroll
          for (int p = 0; p < 16; ++p) {
            const int i = 2 * p, k = 32 * c + i;
            const int o0 = koff[k], o1 = koff[k + 1];
            const float p0 = o0 >= 0 ? ex2_approx(__fmaf_rn(ka[k], t[i], qm[o0 + tid]) - m) : 0.0f;
            const float p1 = o1 >= 0 ? ex2_approx(__fmaf_rn(ka[k + 1], t[i + 1], qm[o1 + tid]) - m) : 0.0f;
            if (p & 1) sc = __fadd2_rn(sc, make_float2(p0, p1)); else sa = __fadd2_rn(sa, make_float2(p0, p1));
            const __nv_bfloat162 b = __float22bfloat162_rn(make_float2(__fmul_rn(p0, kgv[k]), __fmul_rn(p1, kgv[k + 1])));
            pw[p] = *reinterpret_cast<const uint32_t*>(&b);
          }
          pf_st16(t_S + 16 * c, pw);
        }
      }
      const float sum = __fadd_rn(__fadd_rn(sa.x, sa.y), __fadd_rn(sc.x, sc.y));
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      l = __fadd_rn(l, sum);
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[2 * half + sb]);
      if (__any_sync(0xffffffffu, *vfailed != 0)) { ok = false; break; }
    }
    // ---- out = G O / l, once the last P' V' is in (its commit covers every earlier MMA) ----
    const int jl = n_tiles - 1;
    if (ok && pf_wait_warp(&o_done[2 * half + (jl & 1)], (jl >> 1) & 1)) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const float f = __fdiv_rn(G, l);
      float* P = part < 0 ? nullptr : a.part + ((unit - a.n_full) * 2 + part) * kPfPartFloats;
      if (P) {  // a split half: its rows' m and l beside its G O / l
        P[kPfRows * kPfD + tid] = m;
        P[kPfRows * kPfD + kPfRows + tid] = l;
      }
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float o[32];
        pf_ld32(t_O + 32 * c, o);
        if (rowq < a.n_q) {
          float4* dst = reinterpret_cast<float4*>(P ? P + (int64_t)tid * kPfD + 32 * c : a.out + (rowq * H + h) * kPfD + 32 * c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__fmul_rn(o[4 * i], f), __fmul_rn(o[4 * i + 1], f), __fmul_rn(o[4 * i + 2], f),
                                 __fmul_rn(o[4 * i + 3], f));
        }
      }
    } else {
      atomicExch(failed, 1);
    }
  } else if (warp != 14 && warp != 15) {
    // ================= K' and V' tiles, one key per thread =================
    // Warps 8, 9 and 12, 13 (sub-partitions 0 and 1) decode K' and write the key factors; warps
    // 10, 11 and 16, 17 decode V'.  Warps 8, 9 / 10, 11 take the even tiles, 12, 13 / 16, 17 the
    // odd ones.  Thread `key` owns key `key` of its tiles: the key's 64
    // code bytes and 8 scale bytes are loaded a tile ahead (nothing reads them until the tile is
    // decoded), and its 128 bf16 channels stored as 16 chunks of 16 bytes in the same [key][d]
    // core-matrix layout for both (K-major for S = Q K'^T, MN-major for P' V').
    const int dq = warp < 14 ? warp - kPfSoftmaxWarps : warp - 10;  // warps 8-13, 16, 17 -> 0..7
    const bool is_k = (dq & 2) == 0;
    const int grp = dq >> 2, key = 32 * (dq & 1) + lane;
    const uint8_t* codes = is_k ? a.k_codes : a.v_codes;
    const uint8_t* scales = is_k ? a.k_scales : a.v_scales;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* free_ = is_k ? k_free : v_free;
    uint8_t* tiles = is_k ? Kb : Vb;
    const uint32_t L = (uint32_t)a.L_f, t_stop = (uint32_t)t_end;
    const uint32_t t_first = (uint32_t)(t_begin + grp * kPfKTile + key);
    uint32_t f = t_first / L, rr = t_first - f * L;  // frame and offset of the key in the group's first tile
    uint4 kc[4];
    uint2 ks;
    int kvs;  // view slot of the loaded key, -1 past the view
    auto load_key = [&](uint32_t t) {
#pragma unroll
      for (int i = 0; i < 4; ++i) kc[i] = make_uint4(0u, 0u, 0u, 0u);
      ks = make_uint2(0u, 0u);
      kvs = -1;
      if (t < t_stop) {
        const int64_t base = (view.row[f] + (int64_t)rr) * a.H + h;
        const uint4* src = reinterpret_cast<const uint4*>(codes + base * (kPfD / 2));
#pragma unroll
        for (int i = 0; i < 4; ++i) kc[i] = src[i];
        ks = *reinterpret_cast<const uint2*>(scales + base * (kPfD / 16));
        kvs = view.vslot[f];
      }
    };
    load_key(t_first);
    for (int j = grp; j < n_tiles; j += 2) {
      const int b = j % kPfBufs, use = j / kPfBufs, tb = j % kPfKeyBufs;
      uint8_t* buf = tiles + b * kTileKV;
      // tile j into buffer j % 4, once the MMAs of tile j - 4 have read it
      if (j >= kPfBufs && !pf_wait_warp(&free_[b], (use - 1) & 1)) break;
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // block k: code bytes 8 k .. 8 k + 7, scale byte k
        const uint4 c4 = kc[k >> 1];
        const uint32_t E2 = scale_bf16x2(((k < 4 ? ks.x : ks.y) >> (8 * (k & 3))) & 0xFFu);
        uint32_t w[8];
        decode_word_bf16((k & 1) ? c4.z : c4.x, E2, w);
        decode_word_bf16((k & 1) ? c4.w : c4.y, E2, w + 4);
        *reinterpret_cast<uint4*>(buf + core_off(key, 2 * k, kLboStd, kSboStd)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(buf + core_off(key, 2 * k + 1, kLboStd, kSboStd)) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      if (is_k) {  // the key's factors, for the softmax
        key_a[tb * kPfKTile + key] = kvs >= 0 ? slot_a[kvs] : 0.0f;
        key_gv[tb * kPfKTile + key] = kvs >= 0 ? slot_gv[kvs] : 0.0f;
        key_off[tb * kPfKTile + key] = kvs >= 0 ? kvs * kPfRows : -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&key_ready[tb]);
      }
      if (j + 2 < n_tiles) {  // the same key of tile j + 2
        rr += 2 * kPfKTile;
        while (rr >= L) {
          rr -= L;
          ++f;
        }
        load_key((uint32_t)(t_begin + (j + 2) * kPfKTile + key));
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[b]);
      if (__any_sync(0xffffffffu, *vfailed != 0)) break;
    }
  } else if (lane == 0) {
    // ================= MMA issue, one thread per half =================
    // S is one tile ahead: S_hh(j + 2) goes into S buffer j % 2 as soon as P'_hh(j) V'(j) has
    // read P'_hh(j) from it, so the softmax finds S_hh(j + 1) ready.
    const int hh = warp - 14;  // warps 14, 15: sub-partitions 2 and 3
    const uint32_t idesc_s = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kPfKTile >> 3) << 17) |
                             ((uint32_t)(kPfQTile >> 4) << 24);  // bf16 x bf16 -> fp32, K-major, N = 64 keys
    const uint32_t idesc_o = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(kPfD >> 3) << 17) |
                             ((uint32_t)(kPfQTile >> 4) << 24);  // B = V' MN-major, N = d = 128
    const uint32_t t_half = tmem + hh * 256, q_smem = smem_u32(Qs + hh * kTileQ);
    bool ok = true;
    auto issue_s = [&](int j) {  // S_hh(j) = Q_hh K'(j)^T into S buffer j % 2
      const int b = j % kPfBufs;
      if (!mbar_wait(&k_full[b], (j / kPfBufs) & 1)) return false;
      if (j >= 2 && !mbar_wait(&o_done[2 * hh + (j & 1)], ((j - 2) >> 1) & 1)) return false;  // P'_hh(j - 2) read
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      pf_mma_tile(t_half + 64 * (j & 1), q_smem, kLboStd, kSboStd, smem_u32(Kb + b * kTileKV), kLboStd, kSboStd,
                  idesc_s, false);
      pf_commit(&s_full[2 * hh + (j & 1)]);
      pf_commit(&k_free[b]);
      return true;
    };
    for (int j = 0; j < 2 && j < n_tiles && ok; ++j) ok = issue_s(j);
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int b = j % kPfBufs;
      if (!mbar_wait(&v_full[b], (j / kPfBufs) & 1)) { ok = false; break; }
      if (!mbar_wait(&p_full[2 * hh + (j & 1)], (j >> 1) & 1)) { ok = false; break; }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      pf_mma_tile_ta(t_half + 128, t_half + 64 * (j & 1), smem_u32(Vb + b * kTileKV), kLboV, kSboV, idesc_o, j > 0);
      pf_commit(&o_done[2 * hh + (j & 1)]);  // O_hh (+)= P'_hh(j) V'(j)
      pf_commit(&v_free[b]);
      if (j + 2 < n_tiles) ok = issue_s(j + 2);
      if (*vfailed) ok = false;
    }
    if (!ok) atomicExch(failed, 1);
    pf_commit(drain);
    if (!mbar_wait(drain, 0)) atomicExch(failed, 1);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (tid == 0 && *vfailed && a.dev_status) atomicOr(a.dev_status, NVFP4_DEV_TIMEOUT);
  if (warp == kPfMmaWarp) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

// The two halves of each split unit: out = (o_0 w_0 + o_1 w_1) / (w_0 + w_1) with
// w_i = l_i 2^(m_i - max(m_0, m_1)) (o_i = G O_i / l_i over the half's keys).  One thread per
// row and 4 channels.
__global__ void __launch_bounds__(256) prefill_merge_kernel(const float* __restrict__ part, float* __restrict__ out,
                                                            int64_t n_split, int64_t n_full, int64_t q_tiles,
                                                            int64_t n_q, int H) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_split * kPfRows * (kPfD / 4)) return;
  const int c4 = (int)(i % (kPfD / 4));
  const int r = (int)((i / (kPfD / 4)) % kPfRows);
  const int64_t s = i / ((int64_t)kPfRows * (kPfD / 4));
  const int64_t unit = n_full + s;
  const int h = (int)(unit / q_tiles);
  const int64_t row = (unit - (int64_t)h * q_tiles) * kPfRows + r;
  if (row >= n_q) return;
  const float* P0 = part + 2 * s * kPfPartFloats;
  const float* P1 = P0 + kPfPartFloats;
  const float m0 = P0[kPfRows * kPfD + r], m1 = P1[kPfRows * kPfD + r];
  const float l0 = P0[kPfRows * kPfD + kPfRows + r], l1 = P1[kPfRows * kPfD + kPfRows + r];
  const float mm = fmaxf(m0, m1);
  const float w0 = __fmul_rn(l0, ex2_approx(m0 - mm)), w1 = __fmul_rn(l1, ex2_approx(m1 - mm));
  const float inv = __frcp_rn(__fadd_rn(w0, w1));
  const float4 o0 = reinterpret_cast<const float4*>(P0 + (int64_t)r * kPfD)[c4];
  const float4 o1 = reinterpret_cast<const float4*>(P1 + (int64_t)r * kPfD)[c4];
  float4 v;
  v.x = __fmul_rn(__fmaf_rn(o0.x, w0, __fmul_rn(o1.x, w1)), inv);
  v.y = __fmul_rn(__fmaf_rn(o0.y, w0, __fmul_rn(o1.y, w1)), inv);
  v.z = __fmul_rn(__fmaf_rn(o0.z, w0, __fmul_rn(o1.z, w1)), inv);
  v.w = __fmul_rn(__fmaf_rn(o0.w, w0, __fmul_rn(o1.w, w1)), inv);
  reinterpret_cast<float4*>(out + (row * H + h) * kPfD)[c4] = v;
}

bool pf_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int pf_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

// The units of the last, partial wave of CTAs are split along keys when they fill at most half
// of the SMs (the wave then ends after about half a unit's time): how many.
int64_t pf_split_units(int64_t n_q, int H, int64_t n_keys, int sms) {
  const int64_t units = (n_q + kPfRows - 1) / kPfRows * H;
  const int64_t r = sms > 0 ? units % sms : 0;
  return ((n_keys + kPfKTile - 1) / kPfKTile >= 2 && r > 0 && 2 * r <= sms) ? r : 0;
}

}  // namespace
}  // namespace nvfp4

extern "C" {

size_t nvfp4_kv_attention_prefill_workspace_bytes(int64_t n_q, int H, int n_frames, int64_t tokens_per_frame) {
  if (n_q < 1 || H < 1 || n_frames < 1 || tokens_per_frame < 1 || n_frames > NVFP4_MAX_VIEW_FRAMES ||
      tokens_per_frame > ((int64_t)1 << 40) / NVFP4_MAX_VIEW_FRAMES)
    return 0;
  const int64_t split = nvfp4::pf_split_units(n_q, H, (int64_t)n_frames * tokens_per_frame, nvfp4::pf_sm_count());
  return (size_t)split * 2 * nvfp4::kPfPartFloats * sizeof(float);
}

nvfp4_status nvfp4_kv_attention_prefill(const void* q_bf16, int64_t n_q, const uint8_t* k_codes,
                                        const uint8_t* k_scales, const float* k_g, const float* k_mean,
                                        const uint8_t* v_codes, const uint8_t* v_scales, const float* v_g,
                                        int64_t pool_rows, int n_meta, const int64_t* frame_row,
                                        const int* frame_meta, int n_frames, int64_t tokens_per_frame, int H, int D,
                                        float scale, float* out, void* workspace, size_t workspace_bytes,
                                        int* dev_status, void* stream) {
  if (D != nvfp4::kPfD || H < 1 || H > 65535) return NVFP4_ESHAPE;
  if (n_q < 1 || (n_q + nvfp4::kPfRows - 1) / nvfp4::kPfRows * H > ((int64_t)1 << 30)) return NVFP4_ESHAPE;
  if (n_frames < 1 || n_frames > NVFP4_MAX_VIEW_FRAMES || tokens_per_frame < 1 || pool_rows < 1 || n_meta < 1)
    return NVFP4_ESHAPE;
  if (tokens_per_frame > ((int64_t)1 << 40) / NVFP4_MAX_VIEW_FRAMES) return NVFP4_ESHAPE;
  if ((int64_t)n_frames * tokens_per_frame > INT32_MAX) return NVFP4_ESHAPE;  // key indices in 32 bits
  if ((int64_t)H * D > ((int64_t)1 << 46) / pool_rows || (int64_t)H * D > ((int64_t)1 << 46) / n_q)
    return NVFP4_ESHAPE;
  if (!q_bf16 || !k_codes || !k_scales || !k_g || !v_codes || !v_scales || !v_g || !frame_row || !frame_meta || !out)
    return NVFP4_EINVAL;
  if (!nvfp4::pf_aligned(q_bf16, 16) || !nvfp4::pf_aligned(workspace, 16) || !nvfp4::pf_aligned(k_codes, 16) || !nvfp4::pf_aligned(k_scales, 8) ||
      !nvfp4::pf_aligned(v_codes, 16) || !nvfp4::pf_aligned(v_scales, 8) ||
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
  static std::atomic<unsigned long long> smem_set{0};
  if (nvfp4::smem_limit_once(nvfp4::attn_prefill_kernel, nvfp4::kPfSmem, smem_set) != cudaSuccess) return NVFP4_ECUDA;
  a.q_tiles = (n_q + nvfp4::kPfRows - 1) / nvfp4::kPfRows;
  const int64_t units = a.q_tiles * H;
  int64_t split = 0;
  if (workspace) {
    split = nvfp4::pf_split_units(n_q, H, a.n_keys, nvfp4::pf_sm_count());
    if (workspace_bytes < (size_t)split * 2 * nvfp4::kPfPartFloats * sizeof(float)) return NVFP4_EINVAL;
  }
  a.part = static_cast<float*>(workspace);
  a.n_full = units - split;
  a.t_mid = (a.n_keys + nvfp4::kPfKTile - 1) / nvfp4::kPfKTile / 2 * nvfp4::kPfKTile;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  nvfp4::attn_prefill_kernel<<<(unsigned)(units + split), nvfp4::kPfThreads, nvfp4::kPfSmem, st>>>(view, a);
  if (split > 0) {
    const int64_t threads = split * nvfp4::kPfRows * (nvfp4::kPfD / 4);
    nvfp4::prefill_merge_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(a.part, out, split, a.n_full,
                                                                                   a.q_tiles, n_q, H);
  }
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

}  // extern "C"
