// mx_quant.cu -- MXFP8 quantisation of a bf16 tensor, rows and/or the
// transpose from one read (End-to-End 4-Bit Training, quantised-linear-layer
// figure: the bf16 output gradient is quantised to MXFP8 with stochastic
// rounding for the DGRAD GEMM and, transposed, for the WGRAD GEMM). Per 32
// values: E8M0 shared exponent e = the smallest integer with
// amax <= 448 * 2^e (mx_shared_exp), elements the E4M3 codes of v * 2^-e by
// RNE or stochastic rounding (Philox bits of the output layout's flat index,
// direction 0 for rows, 1 for columns).
//
// One CTA (256 threads) per 64 (R) x 128 (C) tile of one slice:
//  1. thread t loads chunks k * 256 + t (k = 0..3) of 8 bf16 (a warp reads two
//     whole 256-byte tile rows per load); a 32-value row block is 4
//     consecutive lanes, which combine their amax with two xor shuffles, and
//     each lane encodes its 8 values from registers (one Philox group);
//  2. the chunks go to a 16 KiB shared tile of 32-bit words (two columns
//     each), word w of row r stored at w ^ (((r >> 4) & 3) << 3);
//  3. lane (cp, q) = (lane >> 2, lane & 3) of warp w reads rows 16q .. 16q+15
//     of column pair 8w + cp (one word per row; with the swizzle the 32 lanes
//     hit 32 distinct banks); a 32-row MX block is lanes q, q ^ 1, which
//     combine their amax with one shuffle; each lane writes 16 code bytes per
//     column.
#include "encode.cuh"
#include "launch.h"
#include "mx_quant.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int TR = 64;          // tile rows
constexpr int TC = 128;         // tile columns
constexpr int kWords = TC / 2;  // 32-bit words (column pairs) per tile row
constexpr int kChunksPerRow = TC / 8;

__device__ __forceinline__ int word_of(int r, int w) {
  return r * kWords + (w ^ (((r >> 4) & 3) << 3));
}

// E4M3 codes of 8 scaled values (|y| <= 448), RNE or stochastic with the
// group's random bits rb (value i uses the 16-bit half i % 2 of word i / 2).
template <bool SR>
__device__ __forceinline__ uint2 e4m3x8(const float* y, const uint4& rb) {
  if constexpr (!SR) {
    return make_uint2(e4m3x4_rn(y[0], y[1], y[2], y[3]), e4m3x4_rn(y[4], y[5], y[6], y[7]));
  } else {
    const uint32_t nw[4] = {~rb.x, ~rb.y, ~rb.z, ~rb.w};
    uint32_t x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = e4m3_sr_hi(y[i], e4m3_sr_n8(nw[i >> 1], i & 1));
    // the codes are the top bytes
    return make_uint2(__byte_perm(__byte_perm(x[0], x[1], 0x0073u),
                                  __byte_perm(x[2], x[3], 0x0073u), 0x5410u),
                      __byte_perm(__byte_perm(x[4], x[5], 0x0073u),
                                  __byte_perm(x[6], x[7], 0x0073u), 0x5410u));
  }
}

template <bool SR>
__device__ __forceinline__ uint4 group_bits(const MxParams& p, uint32_t dir, int64_t idx0) {
  if constexpr (SR) return sr_group_bits(p.seed, p.step, dir, (uint64_t)idx0);
  else return make_uint4(0, 0, 0, 0);
}

template <bool SR, bool ROWS, bool COLS>
__global__ void __launch_bounds__(kThreads) mx_quant_kernel(const MxParams p, int64_t tiles_r,
                                                            int64_t tiles_c) {
  pdl_begin();
  __shared__ __align__(16) uint32_t tile[COLS ? TR * kWords : 4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t R = p.R, C = p.C;
  const int64_t bid = blockIdx.x;
  const int64_t tc = bid % tiles_c, tr = (bid / tiles_c) % tiles_r, s = bid / (tiles_c * tiles_r);
  const int64_t r0 = tr * TR, c0 = tc * TC;
  const uint16_t* xs = p.x + s * R * C;
  const bool vec = (C % 8) == 0;

  // ---- 1: load, flag non-finite values, encode the row blocks ------------
  uint4 v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int chunk = k * kThreads + threadIdx.x;
    const int lr = chunk / kChunksPerRow, lc = (chunk % kChunksPerRow) * 8;
    const int64_t r = r0 + lr, c = c0 + lc;
    const bool ok = r < R && c < C;
    v[k] = make_uint4(0, 0, 0, 0);
    if (ok) {
      if (vec) {
        v[k] = __ldcs(reinterpret_cast<const uint4*>(xs + r * C + c));
      } else {  // column-only encoding of a tensor whose rows are not 16 B multiples
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = (c + i < C) ? xs[r * C + c + i] : 0u;
        v[k] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                          h[6] | (h[7] << 16));
      }
    }
    uint32_t m = absmax_bits4(v[k]);
    if (m >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
    if constexpr (ROWS) {  // C % 32 == 0: a block's four chunks are all in range or all out
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      const int ex = mx_shared_exp(__uint_as_float(m << 16));
      const float sc = exp2_neg(ex);
      f2 x[4];
      unpack8(v[k], x);
      float y[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        y[2 * i] = __fmul_rn(x[i].x, sc);
        y[2 * i + 1] = __fmul_rn(x[i].y, sc);
      }
      const int64_t e = (s * R + r) * C + c;  // flat row-layout index
      const uint2 codes = e4m3x8<SR>(y, group_bits<SR>(p, 0u, e));
      if (ok) {
        __stcs(reinterpret_cast<uint2*>(p.r_codes + e), codes);
        if ((lane & 3) == 0) p.r_scales[e / 32] = (uint8_t)(ex + 127);
      }
    }
  }

  if constexpr (COLS) {
    // ---- 2: stage -------------------------------------------------------
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int chunk = k * kThreads + threadIdx.x;
      const int lr = chunk / kChunksPerRow, lw = (chunk % kChunksPerRow) * 4;
      *reinterpret_cast<uint4*>(&tile[word_of(lr, lw)]) = v[k];
    }
    __syncthreads();
    // ---- 3: column blocks -------------------------------------------------
    const int q = lane & 3, cpl = warp * 8 + (lane >> 2);  // column pair within the tile
    const int64_t cg = c0 + 2 * cpl;                        // first of its two columns
    const bool row_ok = r0 + 16 * q < R;                    // R % 32 == 0: whole MX blocks
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = tile[word_of(16 * q + i, cpl)];
    uint32_t mm = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) mm = __vmaxu2(mm, w[i] & 0x7FFF7FFFu);
    mm = __vmaxu2(mm, __shfl_xor_sync(0xFFFFFFFFu, mm, 1));
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // column cg + h
      const int ex = mx_shared_exp(__uint_as_float(h ? (mm & 0xFFFF0000u) : (mm << 16)));
      const float sc = exp2_neg(ex);
      float y[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(h ? bf16_hi(w[i]) : bf16_lo(w[i]), sc);
      const int64_t ce = (s * C + cg + h) * R + r0 + 16 * q;  // flat column-layout index
      const uint2 a = e4m3x8<SR>(y, group_bits<SR>(p, 1u, ce));
      const uint2 b = e4m3x8<SR>(y + 8, group_bits<SR>(p, 1u, ce + 8));
      if (row_ok && cg + h < C) {
        __stcs(reinterpret_cast<uint4*>(p.c_codes + ce), make_uint4(a.x, a.y, b.x, b.y));
        if ((q & 1) == 0) p.c_scales[ce / 32] = (uint8_t)(ex + 127);
      }
    }
  }
}

template <bool SR, bool ROWS, bool COLS>
cudaError_t launch_t(const MxParams& p, cudaStream_t st) {
  const int64_t tiles_r = (p.R + TR - 1) / TR, tiles_c = (p.C + TC - 1) / TC;
  const int64_t n = p.S * tiles_r * tiles_c;
  if (n > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(mx_quant_kernel<SR, ROWS, COLS>, dim3((unsigned)n), dim3(kThreads), st, p,
                    tiles_r, tiles_c);
}

}  // namespace

cudaError_t launch_mx_quant(const MxParams& p, bool rows, bool cols, bool sr, cudaStream_t st) {
  if (rows && cols)
    return sr ? launch_t<true, true, true>(p, st) : launch_t<false, true, true>(p, st);
  if (rows) return sr ? launch_t<true, true, false>(p, st) : launch_t<false, true, false>(p, st);
  return sr ? launch_t<true, false, true>(p, st) : launch_t<false, false, true>(p, st);
}

}  // namespace nvfp4
