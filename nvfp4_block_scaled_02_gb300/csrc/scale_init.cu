// scale_init.cu -- MSE scale setting with an FP8 scale sweep (Scale Learning
// blog, "Using Scale Learning": the MSE scale algorithm with fp8_scale_sweep
// initialises the learnable scales).
//
// Per 1x16 block every positive finite E4M3 scale s_c = dec(c) * g
// (c = 1..126, g = gamax / (6 * 448)) is tried: the block is fake-quantised at
// s_c (q = clamp(round(x * (1/s_c))), E2M1 RNE) and its error
// e = fma(-q, s_c, x) summed in the fixed block order (per half of 8, even
// and odd positions accumulated separately with fma from +0). The smallest sum
// wins, ties keep the smaller code. One lane per block holds its 16 values in
// registers for the whole sweep; d and 1/d of every code come from a per-CTA
// shared table.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) scale_init_mse_kernel(const ScaleInitParams p) {
  pdl_begin();
  __shared__ float s_d[128], s_inv[128];
  const SliceScale ss = slice_scale(*p.gamax, 448.0f);
  if (threadIdx.x < 128) scale_entry<0>((uint32_t)threadIdx.x, ss.g, s_d[threadIdx.x],
                                        s_inv[threadIdx.x]);
  if (ss.bad && blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
  __syncthreads();
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x; b < p.nblocks; b += stride) {
    const uint4 v0 = __ldcs(p.x + 2 * b), v1 = __ldcs(p.x + 2 * b + 1);
    if (max(absmax_bits4(v0), absmax_bits4(v1)) >= 0x7F80u)
      flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
    f2 lo[4], hi[4];
    unpack8(v0, lo);
    unpack8(v1, hi);
    uint32_t best = 1;
    float best_sse = 0.0f;
#pragma unroll 2
    for (uint32_t c = 1; c <= 126; ++c) {
      const float d = s_d[c], inv = s_inv[c];
      const uint4 none = make_uint4(0, 0, 0, 0);
      f2 q[4];
      const float sse = __fadd_rn(half_sse(lo, round8<false>(lo, inv, none), d, q),
                                  half_sse(hi, round8<false>(hi, inv, none), d, q));
      if (c == 1 || sse < best_sse) {
        best = c;
        best_sse = sse;
      }
    }
    if (p.codes) p.codes[b] = (uint8_t)best;
    if (p.s) p.s[b] = s_d[best];
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
