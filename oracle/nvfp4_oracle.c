/*
 * nvfp4_oracle.c -- plain, single-threaded CPU oracle for NVFP4 block-scaled
 * quantization of bf16 tensors and for the scale-learning STE backward.
 *
 * The loops over independent blocks, rows or elements carry OpenMP pragmas.
 * The default build ignores them and runs on one thread; a second build
 * (-fopenmp) runs the same loops on all host cores, only to time the oracle
 * as an all-core CPU baseline. Every parallel iteration writes outputs that
 * no other iteration touches (4/6 bitmaps are built one 32-block word per
 * iteration), and status bits are OR-reduced, so both builds give the same
 * bytes.
 *
 * TEST INFRASTRUCTURE. This file is the yardstick the CUDA library is checked
 * against; it is not part of the product. Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg load it. It shares no source, header, table
 * or constant generator with the CUDA library, and it includes nothing of it.
 *
 * Arithmetic: IEEE binary32 with round-to-nearest-even. The file is compiled
 * with -ffp-contract=off, so every product and every sum rounds by itself; the
 * only fused operations are the explicit fmaf() calls. Distances used to find
 * the nearest representable value are taken in binary64, where they are exact
 * for every case that can decide a tie.
 *
 * Sources (page title, then section):
 *  [SL]  "Scale Learning: Training NVFP4 Block Scales to Recover Accuracy",
 *        section "How Scale Learning Works" (fake-quant forward, STE
 *        derivatives, dual pre/post scales).
 *  [UE]  "UE5M3: ..." (hankli.space), sections on the math derivation
 *        (block scale = quant(amax / Qmax), Qmax = 6), current vs periodic
 *        tensor scaling, selective stochastic rounding, and the E2M1 grid.
 *  [E2E] "End-to-End 4-Bit Training", sections "Low-precision formats on
 *        Blackwell" (E2M1 grid, E4M3 block scale, FP32 outer scale, the
 *        -54 -> -6 @ scale 9 example), "Block-scaled backward passes" (row vs
 *        column blocks) and "Re-quantization with stochastic rounding" (the
 *        5.4 and 4.5 examples).
 *  [46]  "Four Over Six: More Accurate NVFP4 Quantization with Adaptive Block
 *        Scaling" (both summaries): method (quantize each block with its max
 *        scaled to 6 and to 4, keep the lower-MSE one), implementation details
 *        (tensor scale computed with an FP8 maximum of 256 instead of 448).
 *
 * Readings of points the pages leave open (each is a definition both sides
 * obey):
 *  R1 E2M1 rounding is nearest-value with ties to the even code; |y| >= 6
 *     saturates to 6; the sign bit is copied from y (so -0 -> 0x8).
 *  R2 E4M3: bias 7, subnormals, max 448, no NaN produced, RNE, saturating.
 *     UE5M3: unsigned, bias 15, exponent field 0 subnormal (m/8 * 2^-14),
 *     all 256 codes finite, max 1.875 * 2^16 = 122880, RNE, saturating.
 *  R3 Global decode scale g = gamax / (6 M) (M = 448, or 256 with 4/6);
 *     g = 1 when gamax == 0.
 *  R4 Block scale for a target k (6, or 4 under 4/6): den = k g,
 *     rden = 1/den (per slice, clamped to FLT_MAX), t = amax_b * rden, code = Q(t),
 *     d = dec(code) * g, inv = 1/d (clamped to FLT_MAX; 0 when d == 0),
 *     y_i = x_i * inv. Every step is one fp32 operation rounded to nearest.
 *  R5 Stochastic rounding: a = |y|; lo <= a < hi are the grid neighbours,
 *     p = (a - lo) / (hi - lo) (exact), u = V * 2^-16 with V the element's
 *     16 random bits; round up iff u < p.
 *     V comes from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
 *     random numbers: as easy as 1, 2, 3", SC'11), key = (seed, step),
 *     counter = (j mod 2^32, j / 2^32, direction, 0) with j = idx / 8, where
 *     idx is the element's flat index in the encoded layout; element idx
 *     takes the 16-bit half (idx % 2) of output word (idx % 8) / 2.
 *  R6 4/6 compares the block sums of squared errors (the MSE denominator is
 *     the same for both): e_i = fma(-q_i, d, x_i); the sum uses the fixed
 *     order of block_sum() below; pick 4 iff sse4 < sse6 (ties keep 6).
 *     The other two rules the 4/6 pages evaluate: MAE (sum of |e_i| with
 *     plain adds in the same order) and max error (max |e_i|); same tie rule.
 *  R7 Dequantised value = bf16_rne(q_i * d) with the product rounded to fp32.
 *  R8 Column (16x1) blocks: the encoding of slice X is the row (1x16)
 *     encoding of X^T, with direction 1 in the random counter.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- status bits returned by the oracle (meaning mirrors the C-ABI) ----- */
#define ORC_ST_NONFINITE_INPUT 1 /* a NaN or Inf element in x            */
#define ORC_ST_BAD_SCALE 2       /* an STE scale that is not usable      */
#define ORC_ST_BAD_AMAX 4        /* a global amax that is NaN/Inf/< 0    */

/* Threads of the OpenMP build (n > 0 sets them); returns the count in use,
 * 1 for the default build. */
int orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/* ---------------------------------------------------------------- bits -- */
static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

float orc_bf16_to_f32(uint16_t h) { return u2f((uint32_t)h << 16); }

/* Round a binary32 value to the nearest bfloat16, ties to even. */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u = f2u(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

void orc_f32_to_bf16_array(const float* f, int64_t n, uint16_t* out);

/* ------------------------------------------------------ value tables ---- */
/* E2M1 magnitudes for codes 0..7: 1 sign, 2 exponent (bias 1), 1 mantissa
 * bit; exponent field 0 is subnormal. [UE] / [E2E]: {0,.5,1,1.5,2,3,4,6}. */
static double e2m1_mag(int m) {
  int e = (m >> 1) & 3, f = m & 1;
  if (e == 0) return f * 0.5;
  return (1.0 + f / 2.0) * ldexp(1.0, e - 1);
}
/* E4M3 (bias 7) for codes 0..126; 127 is NaN and never produced. */
static double e4m3_mag(int c) {
  int e = (c >> 3) & 15, f = c & 7;
  if (e == 0) return f / 8.0 * ldexp(1.0, -6);
  return (1.0 + f / 8.0) * ldexp(1.0, e - 7);
}
/* UE5M3 (unsigned, bias 15) for codes 0..255, all finite (reading R2). */
static double ue5m3_mag(int c) {
  int e = (c >> 3) & 31, f = c & 7;
  if (e == 0) return f / 8.0 * ldexp(1.0, -14);
  return (1.0 + f / 8.0) * ldexp(1.0, e - 15);
}

float orc_e2m1_value(uint8_t code) {
  double v = e2m1_mag(code & 7);
  return (float)((code & 8) ? -v : v);
}
float orc_e4m3_value(uint8_t code) { return (float)e4m3_mag(code & 0x7F); }
float orc_ue5m3_value(uint8_t code) { return (float)ue5m3_mag(code); }

/* Index of the value nearest to a in an ascending table of n values, ties
 * to the even index, a above the top -> top. This is the plain definition
 * of round-to-nearest-even into a small float format (R1, R2). */
static int nearest_index(double a, double (*val)(int), int n) {
  if (!(a < val(n - 1))) return n - 1; /* saturate (also catches NaN) */
  int lo = 0, hi = n - 1;              /* val(lo) <= a < val(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (val(mid) <= a) lo = mid; else hi = mid;
  }
  double dlo = a - val(lo), dhi = val(hi) - a;
  if (dlo < dhi) return lo;
  if (dhi < dlo) return hi;
  return (lo % 2 == 0) ? lo : hi;
}

/* R1: E2M1 round-to-nearest-even, saturating, sign copied from y. */
uint8_t orc_e2m1_rne(float y) {
  uint8_t s = signbit(y) ? 8 : 0;
  return (uint8_t)(s | nearest_index(fabs((double)y), e2m1_mag, 8));
}

/* R2: encode a non-negative block-scale target t. fmt 0 = E4M3, 1 = UE5M3. */
uint8_t orc_scale_encode(int fmt, float t) {
  if (fmt == 0) return (uint8_t)nearest_index((double)t, e4m3_mag, 127);
  return (uint8_t)nearest_index((double)t, ue5m3_mag, 256);
}
float orc_scale_value(int fmt, uint8_t code) {
  return fmt == 0 ? orc_e4m3_value(code) : orc_ue5m3_value(code);
}

/* ------------------------------------------------------------ Philox ---- */
/* Philox4x32-10 exactly as published (SC'11): ten rounds of two 32x32->64
 * multiplies with the Weyl key schedule. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)p0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* R5: the 16 random bits of element idx of an encoding. */
uint32_t orc_sr_bits(uint32_t seed, uint32_t step, uint32_t dir, uint64_t idx) {
  uint64_t j = idx >> 3;
  uint32_t ctr[4] = {(uint32_t)j, (uint32_t)(j >> 32), dir, 0u};
  uint32_t key[2] = {seed, step};
  uint32_t w[4];
  orc_philox4x32_10(ctr, key, w);
  uint32_t word = w[(idx & 7) >> 1];
  return (idx & 1) ? (word >> 16) : (word & 0xFFFFu);
}

/* R5: stochastic rounding of y onto the E2M1 grid with random bits v16. */
uint8_t orc_e2m1_sr(float y, uint32_t v16) {
  uint8_t s = signbit(y) ? 8 : 0;
  double a = fabs((double)y);
  if (!(a < 6.0)) return (uint8_t)(s | 7);
  int lo = 0;
  while (lo < 7 && e2m1_mag(lo + 1) <= a) ++lo;
  double p = (a - e2m1_mag(lo)) / (e2m1_mag(lo + 1) - e2m1_mag(lo));
  double u = (double)(v16 & 0xFFFFu) / 65536.0;
  return (uint8_t)(s | (u < p ? lo + 1 : lo));
}

/* Array forms, used by the exhaustive codec tests. */
void orc_e2m1_rne_array(const float* y, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_rne(y[i]);
}
void orc_scale_encode_array(int fmt, const float* t, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_scale_encode(fmt, t[i]);
}
void orc_e2m1_sr_array(const float* y, const uint32_t* v16, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_sr(y[i], v16[i]);
}
void orc_sr_bits_array(uint32_t seed, uint32_t step, uint32_t dir, uint64_t idx0,
                       int64_t n, uint32_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_sr_bits(seed, step, dir, idx0 + (uint64_t)i);
}

void orc_f32_to_bf16_array(const float* f, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(f[i]);
}

/* ---------------------------------------------------------- block sums -- */
/* The fixed in-block reduction order shared by the 4/6 error sums and the
 * STE scale gradients: the block's 16 terms a_i * b_i are split into halves
 * 0..7 and 8..15; inside a half, even and odd positions accumulate separately
 * from +0 with fma in increasing index; half = even + odd; block = half0 +
 * half1. */
static float block_sum(const float* a, const float* b) {
  float half[2];
  for (int h = 0; h < 2; ++h) {
    float acc[2] = {0.0f, 0.0f};
    for (int p = 0; p < 2; ++p)
      for (int j = 0; j < 4; ++j) {
        int i = 8 * h + p + 2 * j;
        acc[p] = fmaf(a[i], b[i], acc[p]);
      }
    half[h] = acc[0] + acc[1];
  }
  return half[0] + half[1];
}

/* The MAE form of block_sum(): |e_i| added (no fma) in the same order. */
static float block_abs_sum(const float* e) {
  float half[2];
  for (int h = 0; h < 2; ++h) {
    float acc[2] = {0.0f, 0.0f};
    for (int p = 0; p < 2; ++p)
      for (int j = 0; j < 4; ++j) acc[p] = acc[p] + fabsf(e[8 * h + p + 2 * j]);
    half[h] = acc[0] + acc[1];
  }
  return half[0] + half[1];
}
static float block_abs_max(const float* e) {
  float m = 0.0f;
  for (int i = 0; i < 16; ++i)
    if (fabsf(e[i]) > m) m = fabsf(e[i]);
  return m;
}

/* ----------------------------------------------------- scale policy ----- */
/* R3: the global decode scale of a slice. Returns the status bit for a bad
 * amax (and uses g = 1 then, so the result stays defined). */
static int global_decode_scale(float gamax, float M, float* g) {
  if (!(gamax >= 0.0f) || isinf(gamax)) { *g = 1.0f; return ORC_ST_BAD_AMAX; }
  if (gamax == 0.0f) { *g = 1.0f; return 0; }
  float den = 6.0f * M;
  *g = gamax / den;
  return 0;
}

/* R3 as a value: the decode scale g of a slice with global amax gamax and
 * FP8 maximum M (for tests that encode single blocks of a larger tensor). */
float orc_decode_scale(float gamax, float M) {
  float g;
  global_decode_scale(gamax, M, &g);
  return g;
}

/* One candidate encoding of a 16-value block for target k (R4, R1/R5). */
typedef struct {
  uint8_t scale;     /* block-scale code                    */
  float d;           /* decoded block scale times g         */
  uint8_t q[16];     /* E2M1 codes                          */
  float qv[16];      /* their values                        */
  float sse;         /* block sum of squared errors (R6)    */
  float sae;         /* block sum of |errors|               */
  float emax;        /* largest |error|                     */
} cand_t;

static void encode_candidate(const float* x, float amax, float g, float k, int fmt,
                             int rounding, const uint32_t* v16, cand_t* c) {
  float den = k * g;
  float rden = 1.0f / den;
  if (rden > FLT_MAX) rden = FLT_MAX; /* g so small that 1/(k g) overflows */
  float t = amax * rden;
  c->scale = orc_scale_encode(fmt, t);
  c->d = orc_scale_value(fmt, c->scale) * g;
  float inv = 0.0f;
  if (c->d > 0.0f) {
    inv = 1.0f / c->d;
    if (inv > FLT_MAX) inv = FLT_MAX;
  }
  for (int i = 0; i < 16; ++i) {
    float y = x[i] * inv;
    c->q[i] = rounding ? orc_e2m1_sr(y, v16[i]) : orc_e2m1_rne(y);
    c->qv[i] = orc_e2m1_value(c->q[i]);
  }
  float e[16];
  for (int i = 0; i < 16; ++i) e[i] = fmaf(-c->qv[i], c->d, x[i]);
  c->sse = block_sum(e, e);
  c->sae = block_abs_sum(e);
  c->emax = block_abs_max(e);
}

/* The 4/6 selection metric: 0 = sum of squares (MSE), 1 = sum of |e| (MAE),
 * 2 = max |e|. */
static float fos_metric(const cand_t* c, int rule) {
  return rule == 1 ? c->sae : (rule == 2 ? c->emax : c->sse);
}

/* Encode one block of 16 fp32 values (the steps of one block, in the pages'
 * order: block amax -> scale -> element rounding -> 4/6 choice -> dequant).
 * idx0 is the flat encoded-layout index of element 0 (for the random bits).
 * Outputs: codes[16] (one code per byte), *scale, *choice (1 = target 4),
 * dq[16] (bf16 bits), dqf[16] (fp32 q*d), sse[2] = the 4/6 metric of the two
 * candidates {k=6, k=4} under `rule`. */
void orc_encode_block(const float* x, float g, int fmt, int rounding, int fos, int rule,
                      uint32_t seed, uint32_t step, uint32_t dir, uint64_t idx0,
                      uint8_t* codes, uint8_t* scale, uint8_t* choice,
                      uint16_t* dq, float* dqf, float* sse) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  uint32_t v16[16] = {0};
  if (rounding)
    for (int i = 0; i < 16; ++i) v16[i] = orc_sr_bits(seed, step, dir, idx0 + (uint64_t)i);
  cand_t c6, c4;
  encode_candidate(x, amax, g, 6.0f, fmt, rounding, v16, &c6);
  const cand_t* pick = &c6;
  sse[0] = fos_metric(&c6, rule);
  sse[1] = 0.0f;
  *choice = 0;
  if (fos) {
    encode_candidate(x, amax, g, 4.0f, fmt, rounding, v16, &c4);
    sse[1] = fos_metric(&c4, rule);
    if (sse[1] < sse[0]) { pick = &c4; *choice = 1; }
  }
  *scale = pick->scale;
  for (int i = 0; i < 16; ++i) {
    codes[i] = pick->q[i];
    dqf[i] = pick->qv[i] * pick->d;
    dq[i] = orc_f32_to_bf16(dqf[i]);
  }
}

/* Row (1x16) encoding of a stack of S matrices [S][Rm][Cm] (Cm % 16 == 0).
 * Outputs (any may be NULL): codes [S][Rm][Cm/2] (element c in the low nibble
 * when c is even), scales [S][Rm][Cm/16], choice bitmap [S][ceil(B/32)]
 * 32-bit words (bit b % 32 of word b / 32 for block b of the slice, B =
 * Rm*Cm/16), dequant bf16 [S][Rm][Cm]. */
static int encode_rows(const float* xs, int64_t S, int64_t Rm, int64_t Cm,
                       const float* g, int fmt, int rounding, int fos, int rule,
                       uint32_t seed, uint32_t step, uint32_t dir,
                       uint8_t* codes, uint8_t* scales, uint32_t* choice, uint16_t* dq) {
  int64_t B = Rm * Cm / 16, W = (B + 31) / 32;
  if (choice) memset(choice, 0, (size_t)(S * W) * sizeof(uint32_t));
  for (int64_t s = 0; s < S; ++s) {
#pragma omp parallel for schedule(static)
    for (int64_t w = 0; w < W; ++w)
    for (int64_t b = 32 * w; b < B && b < 32 * w + 32; ++b) {
      int64_t e0 = s * Rm * Cm + b * 16;
      uint8_t q[16], sc, ch;
      uint16_t d16[16];
      float df[16], sse[2];
      orc_encode_block(xs + e0, g[s], fmt, rounding, fos, rule, seed, step, dir,
                       (uint64_t)e0, q, &sc, &ch, d16, df, sse);
      if (codes)
        for (int i = 0; i < 16; i += 2)
          codes[(e0 + i) / 2] = (uint8_t)((q[i] & 15) | ((q[i + 1] & 15) << 4));
      if (scales) scales[s * B + b] = sc;
      if (choice && ch) choice[s * W + b / 32] |= 1u << (b % 32);
      if (dq) memcpy(dq + e0, d16, sizeof d16);
    }
  }
  return 0;
}

/* ------------------------------------------------------- entry points ---- */

/* Per-slice global amax: max |x| over each slice of n elements (a1). */
int orc_global_amax(const uint16_t* x, int64_t S, int64_t n, float* amax) {
  int st = 0;
  for (int64_t s = 0; s < S; ++s) {
    uint16_t m = 0;
#pragma omp parallel for schedule(static) reduction(max : m) reduction(| : st)
    for (int64_t i = 0; i < n; ++i) {
      uint16_t a = x[s * n + i] & 0x7FFFu;
      if (a >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;
      if (a > m) m = a;
    }
    amax[s] = orc_bf16_to_f32(m);
  }
  return st;
}

/* Full quantisation (a2..a7). blocks: 1 = rows, 2 = columns, 3 = both.
 * scale_max 0 selects 256 with 4/6 and 448 without (R3). */
int orc_quantize(int blocks, int fmt, int rounding, int fos, int rule, float scale_max,
                 uint32_t seed, uint32_t step,
                 const uint16_t* x, int64_t S, int64_t R, int64_t C, const float* gamax,
                 uint8_t* r_codes, uint8_t* r_scales, uint32_t* r_choice, uint16_t* r_dq,
                 uint8_t* c_codes, uint8_t* c_scales, uint32_t* c_choice, uint16_t* c_dq) {
  int st = 0;
  int64_t N = S * R * C;
  float M = scale_max > 0.0f ? scale_max : (fos ? 256.0f : 448.0f);
  float* g = (float*)malloc((size_t)(S > 0 ? S : 1) * sizeof(float));
  float* xf = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
  for (int64_t s = 0; s < S; ++s) st |= global_decode_scale(gamax[s], M, &g[s]);
#pragma omp parallel for schedule(static) reduction(| : st)
  for (int64_t i = 0; i < N; ++i) {
    if ((x[i] & 0x7FFFu) >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;
    xf[i] = orc_bf16_to_f32(x[i]);
  }
  if (blocks & 1)
    encode_rows(xf, S, R, C, g, fmt, rounding, fos, rule, seed, step, 0,
                r_codes, r_scales, r_choice, r_dq);
  if (blocks & 2) {
    float* xt = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
    for (int64_t s = 0; s < S; ++s)
#pragma omp parallel for schedule(static)
      for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
          xt[s * R * C + c * R + r] = xf[s * R * C + r * C + c];
    encode_rows(xt, S, C, R, g, fmt, rounding, fos, rule, seed, step, 1,
                c_codes, c_scales, c_choice, c_dq);
    free(xt);
  }
  free(xf);
  free(g);
  return st;
}

/* ----------------------------------------------------- scale learning ---- */
/* [SL] fake quantisation: x~ = s_post * clamp(round(x / s_pre), -6, 6), with
 * round the E2M1 rounding (R1) and x / s_pre taken as x * (1 / s_pre). A NULL
 * s_post means a single (tied) scale. x is [R][C], scales [R][C/16]. */
static int scale_ok(float s_pre, float s_post) {
  if (!(s_pre >= FLT_MIN) || !(s_pre <= FLT_MAX)) return 0;
  if (!(fabsf(s_post) <= FLT_MAX)) return 0;
  return 1;
}

int orc_fakequant_fwd(const uint16_t* x, int64_t R, int64_t C, const float* s_pre,
                      const float* s_post, uint16_t* xq) {
  int st = 0;
  int64_t nb = R * C / 16;
#pragma omp parallel for schedule(static) reduction(| : st)
  for (int64_t b = 0; b < nb; ++b) {
    float sp = s_pre[b], so = s_post ? s_post[b] : s_pre[b];
    if (!scale_ok(sp, so)) st |= ORC_ST_BAD_SCALE;
    float inv = 1.0f / sp;
    for (int i = 0; i < 16; ++i) {
      int64_t e = b * 16 + i;
      if ((x[e] & 0x7FFFu) >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;
      float r = orc_bf16_to_f32(x[e]) * inv;
      float q = orc_e2m1_value(orc_e2m1_rne(r));
      xq[e] = orc_f32_to_bf16(so * q);
    }
  }
  return st;
}

/* [SL] STE backward. gq = dL/dx~ (bf16 [R][C]).
 *   r = x * (1/s_pre), q = clamp(round(r)), in = (-6 <= r <= 6)
 *   dL/dx = in ? g * (s_post/s_pre) : 0, with s_post/s_pre taken as
 *           a = s_post * (1/s_pre) for dual scales and exactly 1 when tied
 *   dual:  dL/ds_post = sum g * q
 *          dL/ds_pre  = -a * sum g * (in ? r : 0)
 *   tied:  dL/ds      = sum g * (in ? q - r : q)      (q = +-6 when clamped)
 * Sums follow block_sum(). gx, gs_post may be NULL; gs_post must be NULL when
 * s_post is NULL (tied), and gs_pre then receives dL/ds. */
int orc_scale_grad_bwd(const uint16_t* x, const uint16_t* gq, int64_t R, int64_t C,
                       const float* s_pre, const float* s_post, uint16_t* gx,
                       float* gs_pre, float* gs_post) {
  int st = 0;
  int64_t nb = R * C / 16;
  int tied = (s_post == NULL);
#pragma omp parallel for schedule(static) reduction(| : st)
  for (int64_t b = 0; b < nb; ++b) {
    float sp = s_pre[b], so = tied ? sp : s_post[b];
    if (!scale_ok(sp, so)) st |= ORC_ST_BAD_SCALE;
    float inv = 1.0f / sp;
    float a = tied ? 1.0f : so * inv;
    float g[16], q[16], rin[16], t[16];
    for (int i = 0; i < 16; ++i) {
      int64_t e = b * 16 + i;
      if ((x[e] & 0x7FFFu) >= 0x7F80u || (gq[e] & 0x7FFFu) >= 0x7F80u)
        st |= ORC_ST_NONFINITE_INPUT;
      g[i] = orc_bf16_to_f32(gq[e]);
      float r = orc_bf16_to_f32(x[e]) * inv;
      int in = (r >= -6.0f) && (r <= 6.0f);
      q[i] = orc_e2m1_value(orc_e2m1_rne(r));
      rin[i] = in ? r : 0.0f;
      t[i] = in ? (q[i] - r) : q[i];
      if (gx) gx[e] = orc_f32_to_bf16(in ? g[i] * a : 0.0f);
    }
    if (tied) {
      if (gs_pre) gs_pre[b] = block_sum(g, t);
    } else {
      if (gs_post) gs_post[b] = block_sum(g, q);
      if (gs_pre) gs_pre[b] = -a * block_sum(g, rin);
    }
  }
  return st;
}

/* ------------------------------------------------- re-quantisation -------- */
/* End-to-End 4-Bit Training, "Re-quantization with stochastic rounding" and
 * its quantised-linear-layer figure: the backward pass de-quantises the
 * forward NVFP4 tensor, transposes it in higher precision and re-quantises it
 * with stochastic rounding, to MXFP8 (the pages' choice) or to NVFP4.
 *
 * Readings:
 *  R9  De-quantised value (fp32, no bf16 rounding): q * d with
 *      d = dec(scale) * g exactly as in the forward encoding. A value that
 *      is not finite (scale times g overflowing fp32, possible only for a
 *      global amax near FLT_MAX) is reported as non-finite input.
 *  R10 MXFP8 (the pages name MXFP8: E4M3 values with one E8M0 power-of-two
 *      scale per 32): per block of 32 values along the transposed rows, the
 *      shared exponent e is the smallest integer with amax <= 448 * 2^e
 *      (448 = E4M3's largest normal), i.e. floor(log2(amax)) - 8, plus 1 when
 *      amax's significand exceeds 1.75; clamped to [-127, 127] (amax = 0 gives
 *      -127); scale byte = e + 127. The pages require the re-quantised tensor
 *      to equal the forward one in expectation; the plain floor(log2) - 8
 *      exponent would clip block maxima between 448 and 512 times the scale,
 *      a bias, so the scale is rounded up instead. Element = E4M3 code of
 *      y = v * 2^-e (one fp32 rounding), by RNE or by stochastic rounding onto
 *      the E4M3 grid (R5's rule and bits, direction 2); |y| <= 448 always.
 *  R11 NVFP4 target: the row encoding (R1..R8) of the transposed fp32 values,
 *      with the forward's per-slice global amax and direction 2. */

/* Stochastic rounding of y onto the signed E4M3 grid (sign in bit 7),
 * saturating at 448, with the 16 random bits v16 (R5's rule). */
uint8_t orc_e4m3_sr(float y, uint32_t v16) {
  uint8_t s = signbit(y) ? 0x80 : 0;
  double a = fabs((double)y);
  if (!(a < 448.0)) return (uint8_t)(s | 0x7E);
  int lo = 0;
  while (lo < 126 && e4m3_mag(lo + 1) <= a) ++lo;
  double p = (a - e4m3_mag(lo)) / (e4m3_mag(lo + 1) - e4m3_mag(lo));
  double u = (double)(v16 & 0xFFFFu) / 65536.0;
  return (uint8_t)(s | (u < p ? lo + 1 : lo));
}
/* Round-to-nearest-even of y onto the signed E4M3 grid, saturating. */
uint8_t orc_e4m3_rne(float y) {
  uint8_t s = signbit(y) ? 0x80 : 0;
  return (uint8_t)(s | nearest_index(fabs((double)y), e4m3_mag, 127));
}
float orc_e4m3_signed_value(uint8_t code) {
  float v = orc_e4m3_value(code & 0x7F);
  return (code & 0x80) ? -v : v;
}

/* Array forms, used by the exhaustive codec tests. */
void orc_e4m3_rne_array(const float* y, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_rne(y[i]);
}
void orc_e4m3_sr_array(const float* y, const uint32_t* v16, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_sr(y[i], v16[i]);
}
int orc_mx_shared_exp(float amax);
void orc_mx_shared_exp_array(const float* amax, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)(orc_mx_shared_exp(amax[i]) + 127);
}

/* R10: the MX shared exponent of a block whose largest |value| is amax: the
 * smallest e with amax <= 448 * 2^e, within [-127, 127]. */
int orc_mx_shared_exp(float amax) {
  if (!(amax > 0.0f)) return -127;
  int e2;
  float m = frexpf(amax, &e2); /* amax = m * 2^e2, m in [0.5, 1) */
  int e = (e2 - 1) - 8 + (2.0f * m > 1.75f ? 1 : 0);
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* MXFP8 encoding of n values (n % 32 == 0), blocks of 32 consecutive values;
 * idx0 = flat index of v[0] in the output layout (for the random bits). */
void orc_mx_encode(const float* v, int64_t n, int rounding, uint32_t seed, uint32_t step,
                   uint32_t dir, uint64_t idx0, uint8_t* codes, uint8_t* scales) {
  for (int64_t b = 0; b < n / 32; ++b) {
    const float* vb = v + 32 * b;
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i)
      if (fabsf(vb[i]) > amax) amax = fabsf(vb[i]);
    int e = orc_mx_shared_exp(amax);
    scales[b] = (uint8_t)(e + 127);
    for (int i = 0; i < 32; ++i) {
      float y = ldexpf(vb[i], -e);
      uint64_t idx = idx0 + (uint64_t)(32 * b + i);
      codes[32 * b + i] = rounding ? orc_e4m3_sr(y, orc_sr_bits(seed, step, dir, idx))
                                   : orc_e4m3_rne(y);
    }
  }
}

/* R9: de-quantise a row encoding [S][R][C] (codes two per byte, scale bytes
 * per 16) to fp32. fmt / scale_max / fos describe the forward encoding. */
int orc_dequant(int fmt, float scale_max, int fos, const uint8_t* codes,
                const uint8_t* scales, int64_t S, int64_t R, int64_t C, const float* gamax,
                float* out) {
  int st = 0;
  float M = scale_max > 0.0f ? scale_max : (fos ? 256.0f : 448.0f);
  for (int64_t s = 0; s < S; ++s) {
    float g;
    st |= global_decode_scale(gamax[s], M, &g);
#pragma omp parallel for schedule(static) reduction(| : st)
    for (int64_t i = 0; i < R * C; ++i) {
      int64_t e = s * R * C + i;
      float d = orc_scale_value(fmt, scales[e / 16]) * g;
      uint8_t c = (e & 1) ? (codes[e / 2] >> 4) : (codes[e / 2] & 15);
      out[e] = orc_e2m1_value(c) * d;
      if (!isfinite(out[e])) st |= ORC_ST_NONFINITE_INPUT;
    }
  }
  return st;
}

/* De-quantise -> transpose -> re-quantise. target 0 = MXFP8 (out_codes
 * [S][C][R] E4M3 bytes, out_scales [S][C][R/32] E8M0 bytes; R % 32 == 0),
 * target 1 = NVFP4 (out_codes [S][C][R/2], out_scales [S][C][R/16], 4/6
 * bitmap when dst_fos, selected under dst_rule). */
int orc_requant(int src_fmt, float src_scale_max, int src_fos, const uint8_t* codes,
                const uint8_t* scales, int64_t S, int64_t R, int64_t C, const float* gamax,
                int target, int rounding, uint32_t seed, uint32_t step, int dst_fmt,
                int dst_fos, int dst_rule, float dst_scale_max, uint8_t* out_codes,
                uint8_t* out_scales, uint32_t* out_choice) {
  int64_t N = S * R * C;
  float* xh = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
  float* xt = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
  int st = orc_dequant(src_fmt, src_scale_max, src_fos, codes, scales, S, R, C, gamax, xh);
  for (int64_t s = 0; s < S; ++s)
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
      for (int64_t c = 0; c < C; ++c) xt[s * R * C + c * R + r] = xh[s * R * C + r * C + c];
  if (target == 0) {
    for (int64_t s = 0; s < S; ++s)
#pragma omp parallel for schedule(static)
      for (int64_t c = 0; c < C; ++c) {
        int64_t e0 = s * C * R + c * R;
        orc_mx_encode(xt + e0, R, rounding, seed, step, 2, (uint64_t)e0, out_codes + e0,
                      out_scales + e0 / 32);
      }
  } else {
    float M = dst_scale_max > 0.0f ? dst_scale_max : (dst_fos ? 256.0f : 448.0f);
    float* g = (float*)malloc((size_t)(S > 0 ? S : 1) * sizeof(float));
    for (int64_t s = 0; s < S; ++s) st |= global_decode_scale(gamax[s], M, &g[s]);
    encode_rows(xt, S, C, R, g, dst_fmt, rounding, dst_fos, dst_rule, seed, step, 2, out_codes,
                out_scales, out_choice, NULL);
    free(g);
  }
  free(xh);
  free(xt);
  return st;
}

/* --------------------------------------------- scale learning, FP8 scales - */
/* Scale Learning blog, "How Scale Learning Works" (the block scale is itself
 * quantised to FP8, with a straight-through estimator there as well) and
 * "Using Scale Learning" (MSE scale setting with an FP8 scale sweep; the
 * learned post-scale is what the exported checkpoint carries).
 *
 * Readings:
 *  R12 FP8 scale unit per tensor: g = gamax / (6 * 448) (g = 1 for a zero
 *      amax, as R3 with M = 448), rg = 1/g clamped to FLT_MAX;
 *      Q8(s) = dec(E4M3(s * rg)) * g for s >= 0 (E4M3 by R2).
 *  R13 STE through the FP8 scale: the fake-quant forward and the STE backward
 *      are evaluated at Q8(s_pre), Q8(s_post) (one Q8(s) when tied); their
 *      scale gradients are returned as the gradients of the unquantised
 *      scales (the derivative of Q8 taken as 1). Bad scale: s_pre not a
 *      normal positive number, s_post negative or not finite, or
 *      Q8(s_pre) < FLT_MIN.
 *  R14 MSE scale setting with an FP8 sweep: per 1x16 block, every positive
 *      finite E4M3 code c = 1..126 is a candidate scale s_c = dec(c) * g; its
 *      error is the fake quantisation of the block at s_c: q_i =
 *      clamp(round(x_i * inv_c)), inv_c = 1/s_c (clamped to FLT_MAX, 0 when
 *      s_c = 0), e_i = fma(-q_i, s_c, x_i), summed as block_sum(e, e). The
 *      smallest sum wins; ties keep the smaller code.
 *  R15 Export: the codes are the FP8-scale fake-quant forward's q (rounding
 *      at Q8(s_pre)), the scale byte is E4M3(s_post * rg); de-quantised with
 *      the same g (R9) it reproduces that forward. */

typedef struct {
  float g, rg;
} fp8_unit;

static int fp8_scale_unit(float gamax, fp8_unit* u) {
  int st = global_decode_scale(gamax, 448.0f, &u->g);
  float rg = 1.0f / u->g;
  u->rg = rg > FLT_MAX ? FLT_MAX : rg;
  return st;
}
static uint8_t q8_code(float s, const fp8_unit* u) { return orc_scale_encode(0, s * u->rg); }
static float q8_value(float s, const fp8_unit* u) {
  return orc_scale_value(0, q8_code(s, u)) * u->g;
}

/* R13: bad-scale status of the raw scales and their FP8 roundings. */
static int fp8_scale_status(const float* s_pre, const float* s_post, int64_t nb,
                            const float* sp_q) {
  int st = 0;
  for (int64_t b = 0; b < nb; ++b) {
    float sp = s_pre[b], so = s_post ? s_post[b] : sp;
    if (!(sp >= FLT_MIN && sp <= FLT_MAX) || !(so >= 0.0f && so <= FLT_MAX) ||
        !(sp_q[b] >= FLT_MIN))
      st |= ORC_ST_BAD_SCALE;
  }
  return st;
}

/* R12/R13: Q8 of every scale of an array (NULL in, NULL out). */
static float* q8_array(const float* s, int64_t nb, const fp8_unit* u) {
  if (!s) return NULL;
  float* out = (float*)malloc((size_t)(nb > 0 ? nb : 1) * sizeof(float));
  for (int64_t b = 0; b < nb; ++b) out[b] = s[b] >= 0.0f ? q8_value(s[b], u) : 0.0f;
  return out;
}

int orc_fakequant_fwd_fp8(const uint16_t* x, int64_t R, int64_t C, const float* s_pre,
                          const float* s_post, float gamax, uint16_t* xq) {
  fp8_unit u;
  int64_t nb = R * C / 16;
  int st = fp8_scale_unit(gamax, &u);
  float* sp = q8_array(s_pre, nb, &u);
  float* so = q8_array(s_post, nb, &u);
  st |= fp8_scale_status(s_pre, s_post, nb, sp);
  st |= orc_fakequant_fwd(x, R, C, sp, so, xq);
  free(sp);
  free(so);
  return st;
}

int orc_scale_grad_bwd_fp8(const uint16_t* x, const uint16_t* gq, int64_t R, int64_t C,
                           const float* s_pre, const float* s_post, float gamax, uint16_t* gx,
                           float* gs_pre, float* gs_post) {
  fp8_unit u;
  int64_t nb = R * C / 16;
  int st = fp8_scale_unit(gamax, &u);
  float* sp = q8_array(s_pre, nb, &u);
  float* so = q8_array(s_post, nb, &u);
  st |= fp8_scale_status(s_pre, s_post, nb, sp);
  st |= orc_scale_grad_bwd(x, gq, R, C, sp, so, gx, gs_pre, gs_post);
  free(sp);
  free(so);
  return st;
}

/* R14: the block SSE of fake quantisation at scale s (inv as R14 says). */
static float fakequant_sse(const float* x, float s) {
  float inv = 0.0f;
  if (s > 0.0f) {
    inv = 1.0f / s;
    if (inv > FLT_MAX) inv = FLT_MAX;
  }
  float e[16];
  for (int i = 0; i < 16; ++i) {
    float q = orc_e2m1_value(orc_e2m1_rne(x[i] * inv));
    e[i] = fmaf(-q, s, x[i]);
  }
  return block_sum(e, e);
}

int orc_scale_init_mse(const uint16_t* x, int64_t R, int64_t C, float gamax, uint8_t* codes,
                       float* s_out, float* sse_out) {
  fp8_unit u;
  int st = fp8_scale_unit(gamax, &u);
  int64_t nb = R * C / 16;
#pragma omp parallel for schedule(dynamic, 64) reduction(| : st)
  for (int64_t b = 0; b < nb; ++b) {
    float xb[16];
    for (int i = 0; i < 16; ++i) {
      uint16_t h = x[b * 16 + i];
      if ((h & 0x7FFFu) >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;
      xb[i] = orc_bf16_to_f32(h);
    }
    int best = 1;
    float best_sse = 0.0f;
    for (int c = 1; c <= 126; ++c) {
      float sse = fakequant_sse(xb, orc_scale_value(0, (uint8_t)c) * u.g);
      if (c == 1 || sse < best_sse) {
        best = c;
        best_sse = sse;
      }
    }
    if (codes) codes[b] = (uint8_t)best;
    if (s_out) s_out[b] = orc_scale_value(0, (uint8_t)best) * u.g;
    if (sse_out) sse_out[b] = best_sse;
  }
  return st;
}

/* R15: export of learned scales to an NVFP4 row encoding [R][C]. */
int orc_export_scales(const uint16_t* x, int64_t R, int64_t C, const float* s_pre,
                      const float* s_post, float gamax, uint8_t* codes, uint8_t* scales) {
  fp8_unit u;
  int64_t nb = R * C / 16;
  int st = fp8_scale_unit(gamax, &u);
  float* sp = q8_array(s_pre, nb, &u);
  st |= fp8_scale_status(s_pre, s_post, nb, sp);
#pragma omp parallel for schedule(static) reduction(| : st)
  for (int64_t b = 0; b < nb; ++b) {
    float inv = 1.0f / sp[b];
    float so = s_post ? s_post[b] : s_pre[b];
    scales[b] = so >= 0.0f ? q8_code(so, &u) : 0;
    for (int i = 0; i < 16; i += 2) {
      int64_t e = b * 16 + i;
      if ((x[e] & 0x7FFFu) >= 0x7F80u || (x[e + 1] & 0x7FFFu) >= 0x7F80u)
        st |= ORC_ST_NONFINITE_INPUT;
      uint8_t q0 = orc_e2m1_rne(orc_bf16_to_f32(x[e]) * inv);
      uint8_t q1 = orc_e2m1_rne(orc_bf16_to_f32(x[e + 1]) * inv);
      codes[e / 2] = (uint8_t)((q0 & 15) | ((q1 & 15) << 4));
    }
  }
  free(sp);
  return st;
}

/* --------------------------------------------------- 16x16 tile scale ---- */
/* End-to-End 4-Bit Training, "Block-scaled backward passes": for weights one
 * scale per 16x16 square tile, from the tile's largest value, keeps the
 * scales identical when the tensor is transposed.
 *
 * Reading:
 *  R16 A tile's scale is the 1x16 block scale of R4 with k = 6 computed from
 *      the tile's amax (no 4/6: the pages pair the tile scale with plain
 *      NVFP4); every 1x16 row block inside the tile is encoded with it
 *      (element rounding R1 or R5 with the row layout's indices, direction 0).
 *      The row encoding has the layout of encode_rows, each row block storing
 *      its tile's scale byte; the column encoding is that encoding transposed
 *      (codes, scales, dequant), so the backward operand is bit for bit the
 *      forward one transposed. R % 16 == 0 and C % 16 == 0. */
int orc_quantize_tile16(int fmt, int rounding, float scale_max, uint32_t seed, uint32_t step,
                        const uint16_t* x, int64_t S, int64_t R, int64_t C, const float* gamax,
                        uint8_t* r_codes, uint8_t* r_scales, uint16_t* r_dq,
                        uint8_t* c_codes, uint8_t* c_scales, uint16_t* c_dq) {
  int st = 0;
  float M = scale_max > 0.0f ? scale_max : 448.0f;
  for (int64_t s = 0; s < S; ++s) {
    float g;
    st |= global_decode_scale(gamax[s], M, &g);
#pragma omp parallel for schedule(static) reduction(| : st)
    for (int64_t tr = 0; tr < R / 16; ++tr)
      for (int64_t tc = 0; tc < C / 16; ++tc) {
        float amax = 0.0f;
        for (int rr = 0; rr < 16; ++rr)
          for (int cc = 0; cc < 16; ++cc) {
            uint16_t h = x[s * R * C + (16 * tr + rr) * C + 16 * tc + cc];
            if ((h & 0x7FFFu) >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;
            float a = fabsf(orc_bf16_to_f32(h));
            if (a > amax) amax = a;
          }
        for (int rr = 0; rr < 16; ++rr) {
          int64_t e0 = s * R * C + (16 * tr + rr) * C + 16 * tc;
          float xb[16];
          uint32_t v16[16] = {0};
          for (int i = 0; i < 16; ++i) {
            xb[i] = orc_bf16_to_f32(x[e0 + i]);
            if (rounding) v16[i] = orc_sr_bits(seed, step, 0, (uint64_t)(e0 + i));
          }
          cand_t cd;
          encode_candidate(xb, amax, g, 6.0f, fmt, rounding, v16, &cd);
          if (r_codes)
            for (int i = 0; i < 16; i += 2)
              r_codes[(e0 + i) / 2] = (uint8_t)((cd.q[i] & 15) | ((cd.q[i + 1] & 15) << 4));
          if (r_scales) r_scales[e0 / 16] = cd.scale;
          if (r_dq)
            for (int i = 0; i < 16; ++i) r_dq[e0 + i] = orc_f32_to_bf16(cd.qv[i] * cd.d);
        }
      }
  }
  /* the column encoding: the row encoding transposed */
  for (int64_t s = 0; s < S; ++s)
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < C; ++c)
      for (int64_t r = 0; r < R; ++r) {
        int64_t e = s * R * C + r * C + c, t = s * R * C + c * R + r;
        if (c_codes) {
          uint8_t q = (e & 1) ? (r_codes[e / 2] >> 4) : (r_codes[e / 2] & 15);
          if (t & 1) c_codes[t / 2] = (uint8_t)((c_codes[t / 2] & 0x0F) | (q << 4));
          else c_codes[t / 2] = (uint8_t)((c_codes[t / 2] & 0xF0) | q);
        }
        if (c_scales && r % 16 == 0) c_scales[t / 16] = r_scales[e / 16];
        if (c_dq) c_dq[t] = r_dq[e];
      }
  return st;
}

/* ------------------------------------------ MXFP8 quantisation of bf16 ---- */
/* End-to-End 4-Bit Training, the quantised-linear-layer figure: the bf16
 * output gradient is quantised to MXFP8 with stochastic rounding for the
 * DGRAD GEMM and, transposed, again for the WGRAD GEMM.
 *
 * Reading:
 *  R17 Row encoding: per 32 consecutive values along C, the MX encoding of
 *      R10 (E8M0 shared exponent rounded up, E4M3 elements by RNE or by the
 *      stochastic rule with direction 0 and the row layout's flat indices);
 *      codes [S][R][C], scales [S][R][C/32]. Column encoding: the row
 *      encoding of X^T with direction 1 (codes [S][C][R], scales
 *      [S][C][R/32]). C % 32 == 0 for rows, R % 32 == 0 for columns. */
int orc_mx_quantize(int blocks, int rounding, uint32_t seed, uint32_t step, const uint16_t* x,
                    int64_t S, int64_t R, int64_t C, uint8_t* r_codes, uint8_t* r_scales,
                    uint8_t* c_codes, uint8_t* c_scales) {
  int st = 0;
  int64_t N = S * R * C;
  float* xf = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
#pragma omp parallel for schedule(static) reduction(| : st)
  for (int64_t i = 0; i < N; ++i) {
    if ((x[i] & 0x7FFFu) >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;
    xf[i] = orc_bf16_to_f32(x[i]);
  }
  if (blocks & 1)
    for (int64_t s = 0; s < S; ++s)
#pragma omp parallel for schedule(static)
      for (int64_t r = 0; r < R; ++r) {
        int64_t e0 = s * R * C + r * C;
        orc_mx_encode(xf + e0, C, rounding, seed, step, 0, (uint64_t)e0, r_codes + e0,
                      r_scales + e0 / 32);
      }
  if (blocks & 2) {
    float* xt = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
    for (int64_t s = 0; s < S; ++s)
#pragma omp parallel for schedule(static)
      for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) xt[s * R * C + c * R + r] = xf[s * R * C + r * C + c];
    for (int64_t s = 0; s < S; ++s)
#pragma omp parallel for schedule(static)
      for (int64_t c = 0; c < C; ++c) {
        int64_t e0 = s * C * R + c * R;
        orc_mx_encode(xt + e0, R, rounding, seed, step, 1, (uint64_t)e0, c_codes + e0,
                      c_scales + e0 / 32);
      }
    free(xt);
  }
  free(xf);
  return st;
}
