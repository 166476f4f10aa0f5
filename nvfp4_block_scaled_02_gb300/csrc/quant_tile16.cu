// quant_tile16.cu -- NVFP4 with one block scale per 16x16 tile (End-to-End
// 4-Bit Training, "Block-scaled backward passes": a single scale from the
// largest value of each 16x16 tile keeps the scales identical when the
// tensor is transposed).
//
// One warp per tile, persistent over tiles (column tiles fastest, the warps
// of a CTA on consecutive tiles so a CTA reads 8 x 32 B of every row). Lane
// (r, h) = (lane >> 1, lane & 1) loads the 8 values of tile row r, columns
// 8h .. 8h+7 (one 16-byte load); the tile amax is a warp max-reduction of
// bf16 bit patterns; the scale is the 1x16 block scale of that amax (target
// 6); each lane encodes its 8 values (RNE, or stochastic with the row
// layout's random bits) and writes them to the row encoding. The column
// encoding is the same codes transposed: lane (c, h) = (lane >> 1, lane & 1)
// gathers column c's codes of rows 8h .. 8h+7 from eight lanes by shuffles.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Tile cursor of one warp: slice, row tile, column tile (fastest); advanced by
// the number of warps of the grid, split into whole row bands and a remainder.
struct WarpTileCursor {
  int64_t s, rt, ct;
  __device__ __forceinline__ void start(int64_t t, int64_t tiles_r, int64_t tiles_c) {
    const int64_t per = tiles_r * tiles_c;
    s = t / per;
    const int64_t rem = t - s * per;
    rt = rem / tiles_c;
    ct = rem - rt * tiles_c;
  }
  __device__ __forceinline__ void next(int64_t g_rows, int64_t g_cols, int64_t tiles_r,
                                       int64_t tiles_c) {
    ct += g_cols;
    rt += g_rows;
    if (ct >= tiles_c) {
      ct -= tiles_c;
      ++rt;
    }
    if (rt >= tiles_r) {
      const int64_t k = rt / tiles_r;
      s += k;
      rt -= k * tiles_r;
    }
  }
};

template <int FMT, bool SR>
__global__ void __launch_bounds__(kThreads) quant_tile16_kernel(const Tile16Params p,
                                                                int64_t tiles_r, int64_t tiles_c) {
  pdl_begin();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 1, h = lane & 1;
  const int64_t R = p.R, C = p.C;
  const int64_t total = p.S * tiles_r * tiles_c;
  const int64_t G = (int64_t)gridDim.x * kWarps;
  const int64_t t0 = (int64_t)blockIdx.x * kWarps + warp;
  if (t0 >= total) return;  // warp-uniform
  const int64_t ntiles = (total - t0 + G - 1) / G;
  const int64_t g_rows = G / tiles_c, g_cols = G - g_rows * tiles_c;
  const bool want_dq = p.r_dq != nullptr;
  WarpTileCursor cur;
  cur.start(t0, tiles_r, tiles_c);
  for (int64_t it = 0; it < ntiles; ++it, cur.next(g_rows, g_cols, tiles_r, tiles_c)) {
    const int64_t r0 = cur.rt * 16, c0 = cur.ct * 16;
    // this lane's 8 values in the row layout
    const int64_t e = (cur.s * R + r0 + r) * C + c0 + 8 * h;
    const uint4 v = __ldcs(p.x + e / 8);
    uint32_t m = absmax_bits4(v);
    if (m >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const SliceScale ss = slice_scale(p.gamax[cur.s], p.M);
    if (ss.bad && lane == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
    const uint32_t code = scale_encode<FMT>(__fmul_rn(__uint_as_float(m << 16), ss.rden6));
    float d, inv;
    scale_entry<FMT>(code, ss.g, d, inv);
    uint4 rb = make_uint4(0, 0, 0, 0);
    if constexpr (SR) rb = sr_group_bits(p.seed, p.step, 0u, (uint64_t)e);
    f2 x[4];
    unpack8(v, x);
    const uint32_t w = round8<SR>(x, inv, rb);
    p.r_codes[e / 8] = w;
    if (h == 0) p.r_scales[e / 16] = (uint8_t)code;
    if (want_dq) {
      f2 q[4];
      e2m1x8_to_f2(w, q);
      __stcs(p.r_dq + e / 8, dequant8(q, d));
    }
    if (p.c_codes) {  // the column encoding: column c = r of this lane's index, rows 8h..8h+7
      const int c = r;
      uint32_t cw = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t src = __shfl_sync(0xFFFFFFFFu, w, 2 * (8 * h + k) + (c >> 3));
        cw |= ((src >> (4 * (c & 7))) & 15u) << (4 * k);
      }
      const int64_t ce = (cur.s * C + c0 + c) * R + r0 + 8 * h;
      p.c_codes[ce / 8] = cw;
      if (h == 0) p.c_scales[ce / 16] = (uint8_t)code;
      if (want_dq) {
        f2 q[4];
        e2m1x8_to_f2(cw, q);
        __stcs(p.c_dq + ce / 8, dequant8(q, d));
      }
    }
  }
}

template <int FMT, bool SR>
cudaError_t launch_t(const Tile16Params& p, cudaStream_t st) {
  const int64_t tiles_r = p.R / 16, tiles_c = p.C / 16;
  const int64_t total = p.S * tiles_r * tiles_c;
  auto k = quant_tile16_kernel<FMT, SR>;
  const int64_t want = (total + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)sm_count() * resident_ctas(k, kThreads);
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  return launch_pdl(k, dim3(grid), dim3(kThreads), st, p, tiles_r, tiles_c);
}

}  // namespace

cudaError_t launch_quant_tile16(const Tile16Params& p, int fmt, bool sr, cudaStream_t st) {
  if (fmt == 0) return sr ? launch_t<0, true>(p, st) : launch_t<0, false>(p, st);
  return sr ? launch_t<1, true>(p, st) : launch_t<1, false>(p, st);
}

}  // namespace nvfp4
