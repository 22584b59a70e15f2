/*
 * nvfp4_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, single-threaded CPU statement of what the NVFP4 KV-cache
 * quantizer computes: per-chunk K-smoothing followed by Four-Over-Six (4/6)
 * adaptive block scaling into packed NVFP4, the matching dequantize, and the
 * same quantizer over 16x16 weight tiles.  Only the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg may load this file's
 * library.  It shares no code with the CUDA kernels.
 *
 * Sources (page titles; the pages print no code for any of this):
 *   "LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video
 *    Generation" (summary page, paper.rainbus.top/paper/2605.18739):
 *     - inference pipeline, step 7: every chunk of F_c = 8 frames
 *       (T_c = F_c * L_f tokens) is K-smoothed, K <- K - mean(K), and then
 *       quantized into the NVFP4 KV cache with 4/6 adaptive block scales;
 *     - "full-stack NVFP4" paragraph: Four-Over-Six picks, per block, the
 *       one of two candidate FP8 block scales with the lower MSE, keeping
 *       the +-6 range or switching to +-4 for finer steps near 75% of the
 *       block maximum;
 *     - training pipeline, step 4: weights use 2-D block scales,
 *       activations 1-D block scales.
 *   The NVFP4 format itself (E2M1 element values {0, .5, 1, 1.5, 2, 3, 4, 6}
 *   with sign, 16-element blocks, an E4M3 block scale and an fp32 per-tensor
 *   scale; E4M3 cast round-to-nearest-even with saturation; ties of the 4/6
 *   comparison going to 6) is the standard NVFP4 definition this library uses.
 *
 * Where the pages are silent the readings below are used (each one is listed
 * with its reason in the design notes):
 *   R1  bf16 inputs are widened to fp32 exactly.
 *   R2  mean[c] = (float)((sum over t of (double)X[t,c]) / (double)T), the sum
 *       taken in binary64 in token order, rounded once to fp32.
 *   R3  Z = fl(X - mean) in fp32; V and activations are not smoothed (Z = X).
 *   R4  amax = max |Z| over the tensor; g = fl(amax / 2688), 2688 = 6 * 448.
 *       H1 (headroom variant, separate entry points): g = fl(amax / 1792), 1792 = 4 * 448.
 *       A non-finite Z makes the call report NONFINITE with filler outputs.
 *   R5  per-tensor candidate factors k_M = fl(1 / fl(M * g)), M in {6, 4};
 *       block candidate scale s_M = fl(a_b * k_M) with a_b = max |Z| over the
 *       block; e_M = E4M3_rne_sat(s_M); S_M = fl(E_M * g).
 *   R6  a candidate is usable iff E_M > 0, S_M > 0 and inv_M = fl(1/S_M) is
 *       finite (correctly rounded reciprocal).
 *   R7  y_i = fl(Z_i * inv_M); q_i = E2M1_rne_sat(y_i) (ties to the even code,
 *       sign kept, |y| beyond 6 saturates); d_i = fl(y_i - Q_i).
 *   R8  sum_M accumulates d_i^2 in element order with one fused multiply-add
 *       per element (acc = fma(d_i, d_i, acc), acc starting at +0); for a
 *       16x16 tile the element order is row-major within the tile.
 *       err_M = fl(fl(E_M * E_M) * sum_M), the block MSE up to the common
 *       factor g^2 / n.
 *   R9  choose M = 4 iff it is usable and (6 is unusable or err_4 < err_6);
 *       ties go to 6.  A block with a_b == 0, or with neither candidate
 *       usable, or a tensor with g == 0, gets scale byte 0x00 and codes 0.
 *   R10 packing: byte j of a row holds element 2j in its low nibble and
 *       element 2j+1 in its high nibble; scales are one E4M3 byte per block,
 *       row-major; the 4/6 choice is folded into the scale byte.
 *   R11 dequant: Xhat = bf16_rne(fl(fl(Q * fl(E * g)) + mean)), the mean term
 *       only when a mean is supplied.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -pthread (no
 * contraction of a*b+c into FMA except the explicit fmaf() of R8).
 *
 * oracle_kv_smooth_quant_threads runs the same statement on several host
 * threads, for timing the baseline on all cores: each thread takes a range of
 * channels (each channel's mean is still one binary64 sum in token order), of
 * elements (amax is a maximum, so the order of the partial maxima does not
 * matter) or of blocks (blocks are independent).  Its results are bit for bit
 * those of the single-threaded function, which stays the statement of record.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_NONFINITE 1
#define ORACLE_EINVAL 2

/* ------------------------------------------------------------------------ */
/* Minifloat formats, written out from their definitions.                    */
/* A format with ebits exponent bits, mbits mantissa bits and bias b has     */
/* normal values (1 + m/2^mbits) * 2^(e-b) for e >= 1 and subnormal values   */
/* m * 2^(1-b-mbits) for e == 0.  maxcode is the largest finite magnitude    */
/* code (E2M1: 0x7 = 6.0; E4M3 "fn": 0x7E = 448, 0x7F being NaN).            */
/* ------------------------------------------------------------------------ */

static double mf_decode_mag(unsigned code, int mbits, int bias) {
  unsigned e = code >> mbits;
  unsigned m = code & ((1u << mbits) - 1u);
  if (e == 0) return ldexp((double)m, 1 - bias - mbits);
  return ldexp(1.0 + ldexp((double)m, -mbits), (int)e - bias);
}

/* Round-to-nearest-even of a finite non-negative value onto the format's   */
/* grid, saturating at the largest finite value.                             */
static unsigned mf_encode_mag(double a, int mbits, int bias, unsigned maxcode) {
  double maxval = mf_decode_mag(maxcode, mbits, bias);
  if (a >= maxval) return maxcode;
  int emin = 1 - bias; /* exponent of the smallest normal */
  if (a < ldexp(1.0, emin)) {
    /* subnormal range: multiples of 2^(emin - mbits); the result m may be  */
    /* 2^mbits, which is exactly the code of the smallest normal.           */
    double m = nearbyint(ldexp(a, -(emin - mbits)));
    return (unsigned)m;
  }
  int e2 = 0;
  (void)frexp(a, &e2);  /* a = f * 2^e2, f in [0.5, 1) */
  int e = e2 - 1;       /* a in [2^e, 2^(e+1)) */
  double q = nearbyint(ldexp(a, mbits - e)); /* in [2^mbits, 2^(mbits+1)] */
  if (q >= ldexp(1.0, mbits + 1)) { q = ldexp(1.0, mbits); e += 1; }
  unsigned code = ((unsigned)(e + bias) << mbits) | ((unsigned)q - (1u << mbits));
  if (code > maxcode) code = maxcode;
  return code;
}

/* E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit. 4-bit code.      */
unsigned oracle_e2m1_encode(float y) {
  unsigned sign = signbit(y) ? 0x8u : 0x0u;
  return sign | mf_encode_mag(fabs((double)y), 1, 1, 0x7u);
}
float oracle_e2m1_decode(unsigned code) {
  double v = mf_decode_mag(code & 0x7u, 1, 1);
  return (float)((code & 0x8u) ? -v : v);
}

/* E4M3 ("fn" variant, no infinities, 0x7F/0xFF = NaN): 4 exponent bits     */
/* (bias 7), 3 mantissa bits.  Encoding saturates at 448.                    */
unsigned oracle_e4m3_encode(float s) {
  unsigned sign = signbit(s) ? 0x80u : 0x0u;
  return sign | mf_encode_mag(fabs((double)s), 3, 7, 0x7Eu);
}
float oracle_e4m3_decode(unsigned code) {
  if ((code & 0x7Fu) == 0x7Fu) return NAN;
  double v = mf_decode_mag(code & 0x7Fu, 3, 7);
  return (float)((code & 0x80u) ? -v : v);
}

/* Array forms of the two encoders (element by element, same arithmetic). */
void oracle_e2m1_encode_n(const float* y, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_e2m1_encode(y[i]);
}
void oracle_e4m3_encode_n(const float* s, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_e4m3_encode(s[i]);
}

/* bfloat16 = the upper 16 bits of an fp32; rounding keeps 8 significant    */
/* bits with round-to-nearest-even, done here on the value with nearbyint.  */
uint16_t oracle_bf16_rne(float x) {
  uint32_t bits;
  if (isnan(x)) return 0x7FC0u;
  if (isinf(x) || x == 0.0f) { memcpy(&bits, &x, 4); return (uint16_t)(bits >> 16); }
  double a = fabs((double)x);
  int e2 = 0;
  (void)frexp(a, &e2);
  int e = e2 - 1; /* a in [2^e, 2^(e+1)) */
  if (e < -126) e = -126; /* bf16 subnormals share fp32's exponent floor */
  double q = nearbyint(ldexp(a, 7 - e)); /* 8 significant bits */
  double r = ldexp(q, e - 7);
  float rf = (float)r; /* exact: r has at most 8 significant bits, or overflows to inf */
  if (signbit(x)) rf = -rf;
  memcpy(&bits, &rf, 4);
  return (uint16_t)(bits >> 16);
}

float oracle_bf16_widen(uint16_t b) {
  uint32_t bits = (uint32_t)b << 16;
  float f;
  memcpy(&f, &bits, 4);
  return f;
}

/* ------------------------------------------------------------------------ */
/* Per-tensor constants (R4, R5).                                            */
/* ------------------------------------------------------------------------ */

float oracle_tensor_scale(float amax) { return amax / 2688.0f; }

/* Headroom variant of R4 (reading H1): g = fl(amax / 1792), 1792 = 4 * 448, the largest
 * denominator under which the 4-candidate of the block that holds the tensor's amax maps
 * to 448 and so never saturates in E4M3.  Everything after g is unchanged. */
float oracle_tensor_scale_headroom(float amax) { return amax / 1792.0f; }

static void candidate_factors(float g, float* k6, float* k4) {
  float m6 = 6.0f * g;
  float m4 = 4.0f * g;
  *k6 = 1.0f / m6;
  *k4 = 1.0f / m4;
}

/* ------------------------------------------------------------------------ */
/* One block, Four-Over-Six (R5..R9).  z holds the block's n values in the   */
/* order of R8 (n = 16 for 1-D blocks, 256 for 16x16 tiles; n <= 256).       */
/* ------------------------------------------------------------------------ */

typedef struct {
  unsigned scale;      /* chosen E4M3 scale byte */
  int chose4;          /* 1 when the 4-candidate was kept */
  unsigned e6, e4;     /* candidate E4M3 codes */
  int ok6, ok4;        /* candidate usable (R6) */
  float err6, err4;    /* candidate errors (R8) */
  float sum6, sum4;    /* candidate sums of squared scaled errors */
} block_result;

static void quantize_candidate(const float* z, int n, float E, float g, unsigned* codes,
                               int* ok, float* sum, float* err) {
  float S = E * g;
  float inv = 1.0f / S;
  *ok = (E > 0.0f) && (S > 0.0f) && isfinite(inv);
  if (!*ok) { *sum = INFINITY; *err = INFINITY; return; }
  float acc = 0.0f;
  for (int i = 0; i < n; ++i) {
    float y = z[i] * inv;
    unsigned q = oracle_e2m1_encode(y);
    float Q = oracle_e2m1_decode(q);
    float d = y - Q;
    acc = fmaf(d, d, acc);
    codes[i] = q;
  }
  *sum = acc;
  *err = (E * E) * acc;
}

static block_result quantize_block(const float* z, int n, float g, float k6, float k4,
                                   unsigned* codes_out) {
  block_result r;
  memset(&r, 0, sizeof(r));
  float ab = 0.0f;
  for (int i = 0; i < n; ++i) ab = fmaxf(ab, fabsf(z[i]));
  for (int i = 0; i < n; ++i) codes_out[i] = 0;
  if (g == 0.0f || ab == 0.0f) { r.scale = 0; r.err6 = r.err4 = 0.0f; return r; }

  float s6 = ab * k6;
  float s4 = ab * k4;
  r.e6 = oracle_e4m3_encode(s6);
  r.e4 = oracle_e4m3_encode(s4);
  float E6 = oracle_e4m3_decode(r.e6);
  float E4 = oracle_e4m3_decode(r.e4);

  unsigned c6[256], c4[256];
  quantize_candidate(z, n, E6, g, c6, &r.ok6, &r.sum6, &r.err6);
  quantize_candidate(z, n, E4, g, c4, &r.ok4, &r.sum4, &r.err4);

  r.chose4 = r.ok4 && (!r.ok6 || r.err4 < r.err6);
  if (r.chose4) {
    r.scale = r.e4;
    memcpy(codes_out, c4, sizeof(unsigned) * (size_t)n);
  } else if (r.ok6) {
    r.scale = r.e6;
    memcpy(codes_out, c6, sizeof(unsigned) * (size_t)n);
  } else {
    r.scale = 0;
  }
  return r;
}

/* Inspect one block: exported so the tests can check candidates directly. */
int oracle_block_detail(const float* z, int n, float g, unsigned* codes_out, unsigned* scale,
                        int* chose4, unsigned* e6, unsigned* e4, int* ok6, int* ok4, float* err6,
                        float* err4, float* sum6, float* sum4) {
  if (n <= 0 || n > 256) return ORACLE_EINVAL;
  float k6, k4;
  candidate_factors(g, &k6, &k4);
  block_result r = quantize_block(z, n, g, k6, k4, codes_out);
  *scale = r.scale; *chose4 = r.chose4; *e6 = r.e6; *e4 = r.e4; *ok6 = r.ok6; *ok4 = r.ok4;
  *err6 = r.err6; *err4 = r.err4; *sum6 = r.sum6; *sum4 = r.sum4;
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Input widening (R1).  dtype 0 = bf16 bit patterns, 1 = fp32.              */
/* ------------------------------------------------------------------------ */

static float load_elem(const void* x, int dtype, size_t i) {
  if (dtype == 0) return oracle_bf16_widen(((const uint16_t*)x)[i]);
  return ((const float*)x)[i];
}

/* Token mean per channel (R2).  x is [T][C]. */
void oracle_channel_mean(const void* x, int dtype, int64_t T, int64_t C, float* mean) {
  for (int64_t c = 0; c < C; ++c) {
    double s = 0.0;
    for (int64_t t = 0; t < T; ++t) s += (double)load_elem(x, dtype, (size_t)(t * C + c));
    mean[c] = (float)(s / (double)T);
  }
}

/* ------------------------------------------------------------------------ */
/* KV chunk quantizer: x is [T][H][D] (D % 16 == 0), blocks of 16 along D.   */
/*   smooth   1 for K (subtract the per-(h,d) token mean), 0 for V/acts     */
/*   mean_in  optional [H*D]; used as the mean instead of computing it      */
/*   mean_out optional [H*D]; receives the mean actually used               */
/*   codes    [T*H*D/2] packed nibbles (R10); scales [T*H*D/16] E4M3 bytes   */
/*   g        per-tensor scale;  chose4 optional [T*H*D/16] decision bytes  */
/* Returns ORACLE_OK, ORACLE_NONFINITE (filler: codes 0, scales 0x7F,        */
/* g = NaN) or ORACLE_EINVAL.                                                */
/* ------------------------------------------------------------------------ */
static int kv_smooth_quant_impl(const void* x, int dtype, int64_t T, int64_t H, int64_t D, int smooth,
                                const float* mean_in, float* mean_out, uint8_t* codes, uint8_t* scales,
                                float* g_out, uint8_t* chose4, int headroom) {
  if (T < 0 || H <= 0 || D <= 0 || (D % 16) != 0 || (dtype != 0 && dtype != 1)) return ORACLE_EINVAL;
  if (!smooth && (mean_in || mean_out)) return ORACLE_EINVAL;
  const int64_t C = H * D;
  const size_t N = (size_t)(T * C);
  const size_t NB = N / 16;

  float* mean = (float*)calloc((size_t)C, sizeof(float));
  if (smooth) {
    if (mean_in) memcpy(mean, mean_in, sizeof(float) * (size_t)C);
    else if (T > 0) oracle_channel_mean(x, dtype, T, C, mean);
    if (mean_out) memcpy(mean_out, mean, sizeof(float) * (size_t)C);
  }

  /* R3 + R4 */
  float* z = (float*)malloc(sizeof(float) * (N ? N : 1));
  int finite = 1;
  float amax = 0.0f;
  for (size_t i = 0; i < N; ++i) {
    float xi = load_elem(x, dtype, i);
    float zi = smooth ? xi - mean[i % (size_t)C] : xi;
    z[i] = zi;
    if (!isfinite(zi)) finite = 0;
    else amax = fmaxf(amax, fabsf(zi));
  }
  if (!finite) {
    memset(codes, 0, N / 2);
    memset(scales, 0x7F, NB);
    if (chose4) memset(chose4, 0, NB);
    *g_out = NAN;
    free(z); free(mean);
    return ORACLE_NONFINITE;
  }
  float g = headroom ? oracle_tensor_scale_headroom(amax) : oracle_tensor_scale(amax);
  *g_out = g;
  float k6 = 0.0f, k4 = 0.0f;
  if (g != 0.0f) candidate_factors(g, &k6, &k4);

  unsigned blk[16];
  for (size_t b = 0; b < NB; ++b) {
    block_result r = quantize_block(z + 16 * b, 16, g, k6, k4, blk);
    scales[b] = (uint8_t)r.scale;
    if (chose4) chose4[b] = (uint8_t)r.chose4;
    for (int j = 0; j < 8; ++j)
      codes[8 * b + (size_t)j] = (uint8_t)(blk[2 * j] | (blk[2 * j + 1] << 4));
  }
  free(z); free(mean);
  return ORACLE_OK;
}

int oracle_kv_smooth_quant(const void* x, int dtype, int64_t T, int64_t H, int64_t D, int smooth,
                           const float* mean_in, float* mean_out, uint8_t* codes, uint8_t* scales,
                           float* g_out, uint8_t* chose4) {
  return kv_smooth_quant_impl(x, dtype, T, H, D, smooth, mean_in, mean_out, codes, scales, g_out, chose4, 0);
}

/* The same with the headroom tensor scale (H1). */
int oracle_kv_smooth_quant_headroom(const void* x, int dtype, int64_t T, int64_t H, int64_t D, int smooth,
                                    const float* mean_in, float* mean_out, uint8_t* codes, uint8_t* scales,
                                    float* g_out, uint8_t* chose4) {
  return kv_smooth_quant_impl(x, dtype, T, H, D, smooth, mean_in, mean_out, codes, scales, g_out, chose4, 1);
}

/* ------------------------------------------------------------------------ */
/* The same quantizer on several host threads (see the header).              */
/* ------------------------------------------------------------------------ */
#define ORACLE_MAX_THREADS 256

typedef struct {
  const void* x;
  int dtype, smooth, phase;
  int64_t T, C;
  float* mean;
  float* z;
  float g, k6, k4;
  uint8_t* codes;
  uint8_t* scales;
  int64_t lo, hi; /* this thread's range of channels, elements or blocks */
  float amax;     /* phase 2: the range's max |Z| */
  int finite;     /* phase 2: every Z of the range finite */
} mt_range;

static void* mt_range_run(void* arg) {
  mt_range* w = (mt_range*)arg;
  if (w->phase == 1) { /* channel means, as oracle_channel_mean */
    for (int64_t c = w->lo; c < w->hi; ++c) {
      double s = 0.0;
      for (int64_t t = 0; t < w->T; ++t) s += (double)load_elem(w->x, w->dtype, (size_t)(t * w->C + c));
      w->mean[c] = (float)(s / (double)w->T);
    }
  } else if (w->phase == 2) { /* Z and amax (R3, R4) */
    for (int64_t i = w->lo; i < w->hi; ++i) {
      float xi = load_elem(w->x, w->dtype, (size_t)i);
      float zi = w->smooth ? xi - w->mean[i % w->C] : xi;
      w->z[i] = zi;
      if (!isfinite(zi)) w->finite = 0;
      else w->amax = fmaxf(w->amax, fabsf(zi));
    }
  } else { /* blocks (R5-R10) */
    unsigned blk[16];
    for (int64_t b = w->lo; b < w->hi; ++b) {
      block_result r = quantize_block(w->z + 16 * b, 16, w->g, w->k6, w->k4, blk);
      w->scales[b] = (uint8_t)r.scale;
      for (int j = 0; j < 8; ++j) w->codes[8 * b + j] = (uint8_t)(blk[2 * j] | (blk[2 * j + 1] << 4));
    }
  }
  return NULL;
}

/* Splits [0, n) into nthreads ranges of `phase` and runs them; a range whose
 * thread cannot be started runs on the calling thread. */
static void mt_phase(const mt_range* base, int phase, int64_t n, int nthreads, mt_range* w) {
  pthread_t th[ORACLE_MAX_THREADS];
  int started[ORACLE_MAX_THREADS];
  for (int i = 0; i < nthreads; ++i) {
    w[i] = *base;
    w[i].phase = phase;
    w[i].lo = n * i / nthreads;
    w[i].hi = n * (i + 1) / nthreads;
    w[i].amax = 0.0f;
    w[i].finite = 1;
  }
  for (int i = 1; i < nthreads; ++i) started[i] = pthread_create(&th[i], NULL, mt_range_run, &w[i]) == 0;
  mt_range_run(&w[0]);
  for (int i = 1; i < nthreads; ++i) {
    if (started[i]) pthread_join(th[i], NULL);
    else mt_range_run(&w[i]);
  }
}

/* oracle_kv_smooth_quant without mean_in / chose4, on nthreads (1..256) host
 * threads.  mean_out optional.  Same returns and filler as the single-threaded
 * function. */
int oracle_kv_smooth_quant_threads(const void* x, int dtype, int64_t T, int64_t H, int64_t D, int smooth,
                                   float* mean_out, uint8_t* codes, uint8_t* scales, float* g_out, int nthreads) {
  if (T < 0 || H <= 0 || D <= 0 || (D % 16) != 0 || (dtype != 0 && dtype != 1)) return ORACLE_EINVAL;
  if (nthreads < 1 || nthreads > ORACLE_MAX_THREADS || (!smooth && mean_out)) return ORACLE_EINVAL;
  const int64_t C = H * D;
  const int64_t N = T * C;
  const int64_t NB = N / 16;
  mt_range base, w[ORACLE_MAX_THREADS];
  memset(&base, 0, sizeof(base));
  base.x = x;
  base.dtype = dtype;
  base.smooth = smooth;
  base.T = T;
  base.C = C;
  base.mean = (float*)calloc((size_t)C, sizeof(float));
  base.z = (float*)malloc(sizeof(float) * (size_t)(N ? N : 1));
  base.codes = codes;
  base.scales = scales;
  if (smooth) {
    if (T > 0) mt_phase(&base, 1, C, nthreads, w);
    if (mean_out) memcpy(mean_out, base.mean, sizeof(float) * (size_t)C);
  }
  mt_phase(&base, 2, N, nthreads, w);
  float amax = 0.0f;
  int finite = 1;
  for (int i = 0; i < nthreads; ++i) {
    amax = fmaxf(amax, w[i].amax);
    finite = finite && w[i].finite;
  }
  if (!finite) {
    memset(codes, 0, (size_t)N / 2);
    memset(scales, 0x7F, (size_t)NB);
    *g_out = NAN;
    free(base.z); free(base.mean);
    return ORACLE_NONFINITE;
  }
  base.g = oracle_tensor_scale(amax);
  *g_out = base.g;
  if (base.g != 0.0f) candidate_factors(base.g, &base.k6, &base.k4);
  mt_phase(&base, 3, NB, nthreads, w);
  free(base.z); free(base.mean);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Dequantize (R11).  codes [T*H*D/2], scales [T*H*D/16]; token t belongs to */
/* group t / tokens_per_group, whose per-tensor scale is g[group] and whose  */
/* mean (optional) is mean[group*H*D + c].  out: bf16 bit patterns.          */
/* ------------------------------------------------------------------------ */
int oracle_kv_dequant(const uint8_t* codes, const uint8_t* scales, const float* g,
                      const float* mean, int64_t tokens_per_group, int64_t T, int64_t H, int64_t D,
                      uint16_t* out) {
  if (T < 0 || H <= 0 || D <= 0 || (D % 16) != 0 || tokens_per_group <= 0) return ORACLE_EINVAL;
  const int64_t C = H * D;
  for (int64_t t = 0; t < T; ++t) {
    int64_t grp = t / tokens_per_group;
    float gg = g[grp];
    for (int64_t c = 0; c < C; ++c) {
      size_t i = (size_t)(t * C + c);
      unsigned byte = codes[i / 2];
      unsigned q = (i % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
      float Q = oracle_e2m1_decode(q);
      float E = oracle_e4m3_decode(scales[i / 16]);
      float S = E * gg;
      float v = Q * S;
      if (mean) v = v + mean[grp * C + c];
      out[i] = oracle_bf16_rne(v);
    }
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Weights, 16x16 tiles.  w is [M][N] (M, N multiples of 16).  codes use the */
/* same row-major nibble packing as above ([M][N/2]); scales [M/16][N/16].   */
/* ------------------------------------------------------------------------ */
int oracle_weight_quant_2d(const void* w, int dtype, int64_t M, int64_t N, uint8_t* codes,
                           uint8_t* scales, float* g_out, uint8_t* chose4) {
  if (M < 0 || N <= 0 || (M % 16) != 0 || (N % 16) != 0 || (dtype != 0 && dtype != 1)) return ORACLE_EINVAL;
  const size_t total = (size_t)(M * N);
  const int64_t TM = M / 16, TN = N / 16;
  int finite = 1;
  float amax = 0.0f;
  for (size_t i = 0; i < total; ++i) {
    float v = load_elem(w, dtype, i);
    if (!isfinite(v)) finite = 0;
    else amax = fmaxf(amax, fabsf(v));
  }
  if (!finite) {
    memset(codes, 0, total / 2);
    memset(scales, 0x7F, (size_t)(TM * TN));
    if (chose4) memset(chose4, 0, (size_t)(TM * TN));
    *g_out = NAN;
    return ORACLE_NONFINITE;
  }
  float g = oracle_tensor_scale(amax);
  *g_out = g;
  float k6 = 0.0f, k4 = 0.0f;
  if (g != 0.0f) candidate_factors(g, &k6, &k4);

  float tile[256];
  unsigned tc[256];
  for (int64_t ti = 0; ti < TM; ++ti) {
    for (int64_t tj = 0; tj < TN; ++tj) {
      for (int r = 0; r < 16; ++r)
        for (int c = 0; c < 16; ++c)
          tile[r * 16 + c] = load_elem(w, dtype, (size_t)((ti * 16 + r) * N + tj * 16 + c));
      block_result br = quantize_block(tile, 256, g, k6, k4, tc);
      scales[ti * TN + tj] = (uint8_t)br.scale;
      if (chose4) chose4[ti * TN + tj] = (uint8_t)br.chose4;
      for (int r = 0; r < 16; ++r) {
        for (int c = 0; c < 16; c += 2) {
          size_t i = (size_t)((ti * 16 + r) * N + tj * 16 + c);
          codes[i / 2] = (uint8_t)(tc[r * 16 + c] | (tc[r * 16 + c + 1] << 4));
        }
      }
    }
  }
  return ORACLE_OK;
}

/* Dequantize 16x16-tiled weights back to bf16 (R11 without a mean). */
int oracle_weight_dequant_2d(const uint8_t* codes, const uint8_t* scales, float g, int64_t M,
                             int64_t N, uint16_t* out) {
  if (M < 0 || N <= 0 || (M % 16) != 0 || (N % 16) != 0) return ORACLE_EINVAL;
  const int64_t TN = N / 16;
  for (int64_t r = 0; r < M; ++r) {
    for (int64_t c = 0; c < N; ++c) {
      size_t i = (size_t)(r * N + c);
      unsigned byte = codes[i / 2];
      unsigned q = (i % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
      float Q = oracle_e2m1_decode(q);
      float E = oracle_e4m3_decode(scales[(r / 16) * TN + c / 16]);
      float S = E * g;
      out[i] = oracle_bf16_rne(Q * S);
    }
  }
  return ORACLE_OK;
}
