// scale_init.cu -- MSE scale setting with an FP8 scale sweep (Scale Learning
// blog, "Using Scale Learning": the MSE scale algorithm with fp8_scale_sweep
// initialises the learnable scales).
//
// Per 1x16 block every positive finite E4M3 scale s_c = dec(c) * g
// (c = 1..126, g = gamax / (6 * 448)) is a candidate: the block is
// fake-quantised at s_c (q = clamp(round(x * (1/s_c))), E2M1 RNE) and its
// error e = fma(-q, s_c, x) summed in the fixed block order (per half of 8,
// even and odd positions accumulated separately with fma from +0). The
// smallest sum wins, ties keep the smaller code. One lane per block holds its
// 16 values in registers; d and 1/d of every code come from a per-CTA table.
//
// Only the candidates that can win are evaluated, and the result is that of
// the full sweep. With A the block's largest |x| (finite blocks):
//  * below: for s_c < A / 6 every q has |q s_c| <= 6 s_c, so the largest
//    value's error is at least m = A - 6 s_c > 0; its fp32 square is a term
//    of the computed sum, and the sum of non-negative terms rounded to
//    nearest never drops below any of them, so the computed sum is at least
//    RN(m)^2 (1 - 2^-24). A code whose RN(m)^2 (1 - 2^-18) already exceeds a
//    computed sum of another code cannot win, and m falls as c grows, so
//    neither can any code below it;
//  * above: from the first code with s_c >= 4.00002 A on, every x * (1/s_c)
//    rounds to at most 1/4 and encodes to 0, so every such code has the same
//    sum (that of the values themselves): only the first of them can win.
// The sweep starts at the amax-derived code c0 (the E4M3 code of A / (6 g)),
// walks down while the bound lets a code beat the best sum so far (a tie
// moves to the smaller code), then up to the first all-zero code (a tie stays
// with the smaller code), so the smallest code with the smallest sum wins as
// in the full sweep. Blocks with a NaN or Inf are swept whole.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;

// E2M1 codes of 8 values (RNE) decoded back to fp32 pairs: the conversions'
// byte results feed the decode directly, with no packed word in between (the
// sweep needs only the decoded values: 278 vs 289 us per sweep of a
// 14336x4096 weight against rounding to a word and splitting it again).
__device__ __forceinline__ void e2m1x8_rn_q(const f2 (&y)[4], f2 (&q)[4]) {
  uint32_t h0, h1, h2, h3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %5, %4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %7, %6;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %9, %8;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %11, %10;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "f"(y[0].x), "f"(y[0].y), "f"(y[1].x), "f"(y[1].y), "f"(y[2].x), "f"(y[2].y),
        "f"(y[3].x), "f"(y[3].y));
  q[0] = __half22float2(*reinterpret_cast<__half2*>(&h0));
  q[1] = __half22float2(*reinterpret_cast<__half2*>(&h1));
  q[2] = __half22float2(*reinterpret_cast<__half2*>(&h2));
  q[3] = __half22float2(*reinterpret_cast<__half2*>(&h3));
}

// The block's error sum at scale d (1/d = inv), in the fixed order.
__device__ __forceinline__ float candidate_sse(const f2 (&lo)[4], const f2 (&hi)[4], float2 di) {
  const f2 iv = make_float2(di.y, di.y);
  f2 y[4], q[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) y[k] = f2_mul(lo[k], iv);
  e2m1x8_rn_q(y, q);
  const float s_lo = half_metric_q(lo, q, di.x, 0);
#pragma unroll
  for (int k = 0; k < 4; ++k) y[k] = f2_mul(hi[k], iv);
  e2m1x8_rn_q(y, q);
  return __fadd_rn(s_lo, half_metric_q(hi, q, di.x, 0));
}

// First c in [lo, hi] where pred(c) is false, pred being true on a prefix of
// [lo, hi]; hi + 1 when it holds everywhere. lo >= 1.
template <class Pred>
__device__ __forceinline__ uint32_t first_false(uint32_t lo, uint32_t hi, Pred pred) {
  while (lo <= hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (pred(mid)) lo = mid + 1;
    else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads) scale_init_mse_kernel(const ScaleInitParams p) {
  pdl_begin();
  __shared__ float2 s_tab[128];  // (d, 1/d) of code c
  const SliceScale ss = slice_scale(*p.gamax, 448.0f);
  if (threadIdx.x < 128) {
    float d, inv;
    scale_entry<0>((uint32_t)threadIdx.x, ss.g, d, inv);
    s_tab[threadIdx.x] = make_float2(d, inv);
  }
  if (ss.bad && blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
  __syncthreads();
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x; b < p.nblocks; b += stride) {
    const uint4 v0 = __ldcs(p.x + 2 * b), v1 = __ldcs(p.x + 2 * b + 1);
    const uint32_t abits = max(absmax_bits4(v0), absmax_bits4(v1));
    f2 lo[4], hi[4];
    unpack8(v0, lo);
    unpack8(v1, hi);
    uint32_t best = 1;
    float best_sse = 0.0f;
    if (abits >= 0x7F80u) {
      flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
      for (uint32_t c = 1; c <= 126; ++c) {
        const float sse = candidate_sse(lo, hi, s_tab[c]);
        if (c == 1 || sse < best_sse) {
          best = c;
          best_sse = sse;
        }
      }
    } else {
      const float A = __uint_as_float(abits << 16);
      const uint32_t c0 = min(max(e4m3_encode(__fmul_rn(A, ss.rden6)), 1u), 126u);
      const float T = __fmul_rn(A, 4.00002f);
      const uint32_t c_last =
          max(min(first_false(1u, 126u, [&](uint32_t c) { return s_tab[c].x < T; }), 126u), c0);
      best = c0;
      best_sse = candidate_sse(lo, hi, s_tab[c0]);
#pragma unroll 1
      for (uint32_t c = c0 - 1; c >= 1; --c) {  // down: stop where the bound rules c out
        const float2 di = s_tab[c];
        const float m = __fmaf_rn(-6.0f, di.x, A);
        if (m > 0.0f && __fmul_rn(__fmul_rn(m, m), 0.999996185302734375f) > best_sse) break;
        const float sse = candidate_sse(lo, hi, di);
        if (sse <= best_sse) {
          best = c;
          best_sse = sse;
        }
      }
#pragma unroll 2
      for (uint32_t c = c0 + 1; c <= c_last; ++c) {  // up to the first all-zero code
        const float sse = candidate_sse(lo, hi, s_tab[c]);
        if (sse < best_sse) {
          best = c;
          best_sse = sse;
        }
      }
    }
    if (p.codes) p.codes[b] = (uint8_t)best;
    if (p.s) p.s[b] = s_tab[best].x;
  }
}

}  // namespace

cudaError_t launch_scale_init_mse(const ScaleInitParams& p, cudaStream_t st) {
  const int64_t want = (p.nblocks + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)sm_count() * resident_ctas(scale_init_mse_kernel, kThreads);
  const unsigned grid = (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
  return launch_pdl(scale_init_mse_kernel, dim3(grid), dim3(kThreads), st, p);
}

}  // namespace nvfp4
