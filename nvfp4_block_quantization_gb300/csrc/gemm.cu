// gemm.cu -- the W4A4 NVFP4 GEMM path (sm_103a): Y = X W^T with X quantized by
// the 1-D quantizer (one E4M3 scale per 16 elements of a row) and W by the 2-D
// quantizer (one E4M3 scale per 16x16 tile), each with its fp32 tensor scale.
//
// "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video Generation"
// (summary page): training step 4 runs the GEMMs in NVFP4 with 2-D block
// scales for weights and 1-D block scales for activations; inference step 6
// merges the weights into a W4A4 model.
//
// The contraction is a dense block-scaled FP4 GEMM on the 5th-generation
// tensor cores, written here directly (tcgen05.mma kind::mxf4nvf4, one UE4M3
// scale per 16 elements of K on each operand, fp32 accumulation in TMEM), in a
// persistent kernel, one CTA per SM walking 128 x 256 tiles of Y (when the last
// wave would leave more than half of the SMs idle, each of its tiles runs as two
// 128 x 128 halves on two CTAs):
//   - a TMA thread streams 128-byte-swizzled K slices of 256 elements of X and
//     W codes, with the matching scale tiles (plain bulk copies, issued first on
//     a barrier of their own), into a 4-stage shared-memory ring that runs on
//     across tiles;
//   - four scale warps move each slice's scales from shared memory into TMEM
//     (tcgen05.st), so the tensor-pipe queue holds MMAs only;
//   - one MMA thread issues the slice's four 128 x 256 x 64 MMAs;
//     tcgen05.commit frees the stage;
//   - eight epilogue warps read the accumulator, scale it by
//     alpha = fl(gX * gW), round to bf16, hand TMEM back to the MMA thread and
//     write Y through a swizzled shared-memory buffer in whole 32-byte sectors.
// The block scales sit in the tensor cores' scale layout: tiles of 128 rows x
// 4 blocks (512 bytes, rows r % 32 at 16-byte steps, r / 32 at 4-byte steps,
// the block within the tile at 1-byte steps), K tiles fastest, zeros in the
// padding; a weight tile's scale is repeated for its 16 rows.  In TMEM the
// MMA reads a K step's scales of row r from lane r % 32 of every 32-lane
// quadrant, column r / 32 of that step's 4 columns: one 512-byte tile, lane l
// taking bytes 16 l .. 16 l + 15, written to all four quadrants.
#include <cstring>
#include <new>

#include <cuda.h>  // CUtensorMap and its enums; the encoder comes through the runtime's driver entry point

#include "nvfp4.h"
#include "bulk.cuh"
#include "common.cuh"
#include "rht16.cuh"

typedef CUresult (*TensorMapEncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                         const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                         CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct nvfp4_gemm_plan {
  int64_t M, N, K;
  int sms;  // persistent grid: one CTA per SM
  TensorMapEncodeTiled encode;
};

namespace nvfp4 {
namespace {

// ---- the tcgen05 GEMM's tile and pipeline ---------------------------------
constexpr int kBM = 128;                     // rows of X (and of Y) per CTA
constexpr int kBN = 256;                     // rows of W (columns of Y) per CTA
constexpr int kBK = 256;                     // K elements per pipeline stage: 128 bytes of codes per row
constexpr int kStages = 4;
constexpr int kMmaK = 64;                    // K elements per tcgen05.mma (kind::mxf4nvf4)
constexpr int kABytes = kBM * kBK / 2;       // 16 KB of X codes per stage
constexpr int kBBytes = kBN * kBK / 2;       // 32 KB of W codes per stage
constexpr int kSfaBytes = kBM * kBK / 16;    // 2 KB: 4 scale tiles of 512 bytes
constexpr int kSfbBytes = kBN * kBK / 16;    // 4 KB: 2 row tiles x 4 scale tiles
constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
constexpr int kEpiWarps = 8;                 // two per TMEM lane quadrant, 128 columns each
constexpr int kEpiStageBytes = 32 * 32;      // per epilogue warp: 32 rows x 16 bf16 columns
constexpr int kGemmSmem = kStages * kStageBytes + kEpiWarps * kEpiStageBytes + 1024 + 256;  // + alignment + barriers
constexpr int kTmemCols = 512;
constexpr int kTmemSf = 256;                 // scale columns follow the 256 accumulator columns
constexpr int kSfColsPerMma = 16;            // W's two row tiles at +0 (8 columns), X's tile at +8 (4), 4 spare
constexpr int kSfColsPerStage = (kBK / kMmaK) * kSfColsPerMma;
static_assert(kTmemSf + kStages * kSfColsPerStage <= kTmemCols, "TMEM columns");
static_assert(kGemmSmem <= 232448, "shared memory per CTA");
static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte alignment of 128-byte swizzling");

constexpr size_t kScalarBytes = 256;         // the workspace: word 0 is the bounded-wait error flag

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

// Shared-memory matrix descriptor of tcgen05 (start address, leading and
// stride byte offsets in 16-byte units, version 1, layout type in bits 61-63).
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)layout << 61);
}
constexpr uint32_t kLayoutSw128 = 2;

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

struct GemmArgs {
  const uint8_t* sfa;   // X scales, tensor-core layout
  const uint8_t* sfb;   // W scales, tensor-core layout
  const float* gx;
  const float* gw;
  uint16_t* y;          // bf16 [M][N]
  int M, N, K;
  int kbt;              // scale tiles along K: ceil(K / 64)
  int* err;
  int n_full;           // tiles [0, n_full) run whole; each later tile as two 128-column halves
};

// Work unit u of the persistent walk: a whole 128 x 256 tile of Y (W tiles
// fastest) or one 128-column half of a tile of the last wave.
struct GemmUnit {
  int m0, n0;  // first row and column of Y
  int width;   // columns: up to 256 (a whole tile) or 128 (a half)
  bool half;
};

__device__ __forceinline__ GemmUnit gemm_unit(int u, int n_full, int tiles_n, int N) {
  const bool half = u >= n_full;
  const int t = half ? n_full + ((u - n_full) >> 1) : u;
  const int n0 = (t % tiles_n) * kBN + (half ? ((u - n_full) & 1) * 128 : 0);
  return GemmUnit{(t / tiles_n) * kBM, n0, min(half ? 128 : kBN, N - n0), half};
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t v[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_st12(uint32_t taddr, const uint32_t r[12]) {  // columns 0-7 and 8-11
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr + 8), "r"(r[8]),
               "r"(r[9]), "r"(r[10]), "r"(r[11])
               : "memory");
}


// Persistent: one CTA per SM walks the work units (u = blockIdx.x + i gridDim.x): the
// 128 x 256 tiles of Y, W tiles fastest, the last wave's as 128 x 128 halves (a half
// loads 128 rows of W through its own tensor map and issues N = 128 MMAs; the
// epilogue warps of columns 128..255 then have nothing to store).  Fourteen warps:
//   warp 0, one lane   loads: the stage ring runs on across tiles, so the next
//                      tile's first stages arrive while the epilogue drains;
//   warp 1, one lane   issues each stage's four MMAs once its scales are in
//                      TMEM; waits for the epilogue to hand the accumulator back
//                      before a new tile's first MMA;
//   warps 2..5         scales: warp w writes TMEM lane quadrant w % 4 with
//                      tcgen05.st -- for K step j of stage s, the columns at
//                      256 + 64 s + 16 j hold W's row tiles 0 and 1 (4 columns
//                      each) and X's tile (4 columns, then 4 unused), lane l of every quadrant
//                      holding rows l, l + 32, l + 64, l + 96 of a tile in
//                      consecutive columns; the tensor-pipe queue then carries
//                      MMAs only;
//   warps 6..13        the epilogue: warp w reads lane quadrant w % 4 (its 32
//                      rows) and one half of the 256 columns, rounds alpha * acc
//                      to bf16 in registers, frees the accumulator, then writes
//                      the rows through a swizzled shared-memory buffer (16
//                      columns at a time) so that each store instruction covers
//                      whole 32-byte sectors of 16 rows.
// A stage's TMEM scale slot is rewritten only after its smem stage was
// refilled, which waits for the MMAs that read the slot.  Every wait is bounded;
// on a timeout the CTA records it, stops issuing work, waits (bounded) for what
// it issued and frees TMEM.
constexpr int kScaleWarps = 4;
constexpr int kGemmThreads = 32 * (2 + kScaleWarps + kEpiWarps);

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_w4a4_kernel(const __grid_constant__ CUtensorMap map_x,
                                                                    const __grid_constant__ CUtensorMap map_w,
                                                                    const __grid_constant__ CUtensorMap map_w_half,
                                                                    GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi_stage = smem + kStages * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(epi_stage + kEpiWarps * kEpiStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* sf_ready = empty + kStages;
  uint64_t* sf_full = sf_ready + kStages;  // a stage's scale bytes landed (ahead of its codes)
  uint64_t* acc_full = sf_full + kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* failed = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* vfailed = failed;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_n = (a.N + kBN - 1) / kBN;
  const int tiles = tiles_n * ((a.M + kBM - 1) / kBM);
  const int nkb = (a.K + kBK - 1) / kBK;
  const int units = a.n_full + 2 * (tiles - a.n_full);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_ready[s], kScaleWarps);
      mbar_init(&sf_full[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    mbar_init(drain, 1);
    *failed = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---- loads ----
      uint32_t g = 0;  // stages issued so far (all tiles)
      for (int u = blockIdx.x; u < units && !*vfailed; u += gridDim.x) {
        const GemmUnit un = gemm_unit(u, a.n_full, tiles_n, a.N);
        const int m0 = un.m0, n0 = un.n0;
        const int n_rt = un.width > 128 ? 2 : 1;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = g % kStages;
          if (g >= kStages && !mbar_wait(&empty[s], ((g / kStages) - 1) & 1)) { atomicExch(failed, 1); break; }
          uint8_t* st = smem + s * kStageBytes;
          const int kt0 = kb * (kBK / kMmaK);
          const int nkt = min(kBK / kMmaK, a.kbt - kt0);
          // the scales first, on their own barrier: the scale warps move them into TMEM while the
          // codes are still landing
          mbar_expect_tx(&sf_full[s], 512u * nkt * (1 + n_rt));
          bulk_load(st + kABytes + kBBytes, a.sfa + ((size_t)(m0 / 128) * a.kbt + kt0) * 512, 512u * nkt, &sf_full[s]);
          for (int rt = 0; rt < n_rt; ++rt)
            bulk_load(st + kABytes + kBBytes + kSfaBytes + rt * (kSfbBytes / 2),
                      a.sfb + ((size_t)(n0 / 128 + rt) * a.kbt + kt0) * 512, 512u * nkt, &sf_full[s]);
          mbar_expect_tx(&full[s], kABytes + (un.half ? kBBytes / 2 : kBBytes));
          tma_load_2d(st, &map_x, kb * (kBK / 2), m0, &full[s]);
          tma_load_2d(st + kABytes, un.half ? &map_w_half : &map_w, kb * (kBK / 2), n0, &full[s]);
        }
      }
      // copies still in flight land before the CTA leaves
      for (uint32_t q = g > (uint32_t)kStages ? g - kStages : 0; q < g; ++q)
        if (!mbar_wait(&full[q % kStages], (q / kStages) & 1) || !mbar_wait(&sf_full[q % kStages], (q / kStages) & 1))
          atomicExch(failed, 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMAs ----
      uint32_t g = 0;
      int i = 0;
      for (int u = blockIdx.x; u < units && !*vfailed; u += gridDim.x, ++i) {
        const int n_tile = gemm_unit(u, a.n_full, tiles_n, a.N).width;
        const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(((n_tile + 15) & ~15) >> 3) << 17) |
                               ((uint32_t)(kBM >> 4) << 24);  // E2M1 x E2M1, UE4M3 scales, K-major, fp32 D
        if (i > 0 && !mbar_wait(acc_empty, (i - 1) & 1)) { atomicExch(failed, 1); break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = g % kStages;
          if (!mbar_wait(&sf_ready[s], (g / kStages) & 1) || !mbar_wait(&full[s], (g / kStages) & 1)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t st = smem_u32(smem + s * kStageBytes);
          const int nkt = min(kBK / kMmaK, a.kbt - kb * (kBK / kMmaK));
          for (int j = 0; j < nkt; ++j) {
            const uint32_t sfb_col = tmem + kTmemSf + s * kSfColsPerStage + j * kSfColsPerMma, sfa_col = sfb_col + 8;
            const uint64_t da = umma_desc(st + j * (kMmaK / 2), 16, 1024, kLayoutSw128);
            const uint64_t db = umma_desc(st + kABytes + j * (kMmaK / 2), 16, 1024, kLayoutSw128);
            const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
                ::"r"(tmem), "l"(da), "l"(db), "r"(idesc), "r"(sfa_col), "r"(sfb_col), "r"(acc) : "memory");
          }
          umma_commit(&empty[s]);
        }
        if (!ok) { atomicExch(failed, 1); break; }
        umma_commit(acc_full);
      }
      // every MMA issued above has finished before TMEM is freed
      umma_commit(drain);
      if (!mbar_wait(drain, 0)) atomicExch(failed, 1);
    }
  } else if (warp < 2 + kScaleWarps) {
    // ---- scales: shared memory -> registers -> TMEM ----
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t g = 0;
    for (int u = blockIdx.x; u < units && !*vfailed; u += gridDim.x) {
      const int n_rt = gemm_unit(u, a.n_full, tiles_n, a.N).width > 128 ? 2 : 1;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb, ++g) {
        const int s = g % kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&sf_full[s], (g / kStages) & 1));  // warp-uniform: tcgen05.st is .aligned
        if (!ok) break;
        const uint8_t* sf = smem + s * kStageBytes + kABytes + kBBytes;
        const int nkt = min(kBK / kMmaK, a.kbt - kb * (kBK / kMmaK));
        for (int j = 0; j < nkt; ++j) {
          uint32_t r[12];
          const uint4 b0 = *reinterpret_cast<const uint4*>(sf + kSfaBytes + j * 512 + lane * 16);
          const uint4 b1 = n_rt == 2 ? *reinterpret_cast<const uint4*>(sf + kSfaBytes + kSfbBytes / 2 + j * 512 + lane * 16)
                                     : make_uint4(0u, 0u, 0u, 0u);
          const uint4 a0 = *reinterpret_cast<const uint4*>(sf + j * 512 + lane * 16);
          r[0] = b0.x; r[1] = b0.y; r[2] = b0.z; r[3] = b0.w;
          r[4] = b1.x; r[5] = b1.y; r[6] = b1.z; r[7] = b1.w;
          r[8] = a0.x; r[9] = a0.y; r[10] = a0.z; r[11] = a0.w;
          tmem_st12(lane_base + kTmemSf + s * kSfColsPerStage + j * kSfColsPerMma, r);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[s]);
      }
      if (!ok) { atomicExch(failed, 1); break; }
    }
  } else {
    // ---- epilogue: TMEM -> alpha * acc -> bf16 registers -> shared -> Y ----
    const int e = warp - 2 - kScaleWarps;
    const int quad = warp & 3, half = e >> 2;  // half 0: columns 0..127, half 1: columns 128..255
    uint8_t* stg = epi_stage + e * kEpiStageBytes;
    const float alpha = __fmul_rn(*a.gx, *a.gw);
    int i = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, i & 1));  // warp-uniform: tcgen05.ld is .aligned
      if (!ok) { atomicExch(failed, 1); break; }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const GemmUnit un = gemm_unit(u, a.n_full, tiles_n, a.N);
      const int m0 = un.m0, n0 = un.n0;
      const int cols = min(128, un.width - half * 128);  // this warp's valid columns (a multiple of 16, maybe <= 0)
      uint32_t o[64];  // row `lane`, 128 columns as bf16 pairs
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * 128);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t v[32];
        tmem_ld32(taddr + 32 * c4, v);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const __nv_bfloat162 h = __float22bfloat162_rn(make_float2(__fmul_rn(alpha, __uint_as_float(v[2 * q])),
                                                                     __fmul_rn(alpha, __uint_as_float(v[2 * q + 1]))));
          o[16 * c4 + q] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);  // the MMAs of the next tile may overwrite TMEM now
#pragma unroll
      for (int h8 = 0; h8 < 8; ++h8) {
        if (h8 * 16 >= cols) break;
        // row `lane` of this warp's 32 rows: 2 chunks of 16 bytes, chunk c at (c ^ ((lane / 4) % 2)) * 16
#pragma unroll
        for (int c = 0; c < 2; ++c)
          *reinterpret_cast<uint4*>(stg + lane * 32 + ((c ^ ((lane >> 2) & 1)) << 4)) =
              make_uint4(o[8 * h8 + 4 * c], o[8 * h8 + 4 * c + 1], o[8 * h8 + 4 * c + 2], o[8 * h8 + 4 * c + 3]);
        __syncwarp();
        // sixteen rows per store instruction: lanes 2 j, 2 j + 1 write the two chunks of row 16 r + j
        const int c = lane & 1;
        const int col = n0 + half * 128 + h8 * 16 + c * 8;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int rr = 16 * r + (lane >> 1);
          const int row = m0 + quad * 32 + rr;
          const uint4 val = *reinterpret_cast<const uint4*>(stg + rr * 32 + ((c ^ ((rr >> 2) & 1)) << 4));
          if (row < a.M) *reinterpret_cast<uint4*>(a.y + (size_t)row * a.N + col) = val;
        }
        __syncwarp();
      }
    }
  }
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0 && *vfailed) atomicExch(a.err, 1);
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
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

// A K-major code matrix [rows][K/2] bytes as a TMA tensor: boxes of 128 bytes
// (256 elements of K) x box_rows rows, 128-byte swizzled, zeros outside.
bool encode_codes(TensorMapEncodeTiled enc, CUtensorMap* map, const uint8_t* codes, int64_t rows, int64_t K,
                  uint32_t box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  const cuuint32_t box[2] = {(cuuint32_t)(kBK / 2), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

size_t nvfp4_gemm_workspace_bytes(void) { return nvfp4::kScalarBytes; }

nvfp4_status nvfp4_gemm_plan_create(int64_t M, int64_t N, int64_t K, nvfp4_gemm_plan** plan) {
  if (!plan) return NVFP4_EINVAL;
  *plan = nullptr;
  if (M < 1 || N < 16 || (N % 16) != 0 || K < 32 || (K % 32) != 0) return NVFP4_ESHAPE;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return NVFP4_ESHAPE;
  if (((M + nvfp4::kBM - 1) / nvfp4::kBM) * ((N + nvfp4::kBN - 1) / nvfp4::kBN) > INT32_MAX) return NVFP4_ESHAPE;
  if (M * N > ((int64_t)1 << 46)) return NVFP4_ESHAPE;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return NVFP4_ECUDA;
  if (cudaFuncSetAttribute(nvfp4::gemm_w4a4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, nvfp4::kGemmSmem) !=
      cudaSuccess)
    return NVFP4_ECUDA;
  const int sms = nvfp4::sm_count();
  if (sms <= 0) return NVFP4_ECUDA;
  nvfp4_gemm_plan* p = new (std::nothrow) nvfp4_gemm_plan;
  if (!p) return NVFP4_ECUDA;
  p->M = M;
  p->N = N;
  p->K = K;
  p->encode = reinterpret_cast<TensorMapEncodeTiled>(fn);
  p->sms = sms;
  *plan = p;
  return NVFP4_OK;
}

void nvfp4_gemm_plan_destroy(nvfp4_gemm_plan* plan) { delete plan; }

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
  CUtensorMap mx, mw, mwh;
  if (!nvfp4::encode_codes(plan->encode, &mx, x_codes, plan->M, plan->K, nvfp4::kBM) ||
      !nvfp4::encode_codes(plan->encode, &mw, w_codes, plan->N, plan->K, nvfp4::kBN) ||
      !nvfp4::encode_codes(plan->encode, &mwh, w_codes, plan->N, plan->K, nvfp4::kBN / 2))
    return NVFP4_ECUDA;
  nvfp4::GemmArgs a;
  a.sfa = x_scales_mma;
  a.sfb = w_scales_mma;
  a.gx = x_tensor_scale;
  a.gw = w_tensor_scale;
  a.y = static_cast<uint16_t*>(y_bf16);
  a.M = (int)plan->M;
  a.N = (int)plan->N;
  a.K = (int)plan->K;
  a.kbt = (int)((plan->K + 63) / 64);
  a.err = static_cast<int*>(workspace);
  const int64_t tiles = ((plan->N + nvfp4::kBN - 1) / nvfp4::kBN) * ((plan->M + nvfp4::kBM - 1) / nvfp4::kBM);
  // a last wave on at most half of the SMs runs as 128-column halves (every tile wider than 128)
  const int64_t r = tiles % plan->sms;
  const bool split = r > 0 && 2 * r <= plan->sms && (plan->N % nvfp4::kBN == 0 || plan->N % nvfp4::kBN > 128);
  a.n_full = (int)(split ? tiles - r : tiles);
  const int64_t units = a.n_full + 2 * (tiles - a.n_full);
  const unsigned grid = (unsigned)(units < plan->sms ? units : plan->sms);
  nvfp4::gemm_w4a4_kernel<<<grid, nvfp4::kGemmThreads, nvfp4::kGemmSmem, static_cast<cudaStream_t>(stream)>>>(mx, mw,
                                                                                                          mwh, a);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ECUDA;
}

}  // extern "C"
