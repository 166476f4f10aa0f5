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
//     consecutive lanes, which combine their amax with two xor shuffles;
//     once all four chunks are in, each lane encodes its 8 values per chunk
//     from registers (one Philox group; the stochastic rounder yields
//     magnitudes and the signs are OR-ed in four at a time from the source
//     words with one byte permute);
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

// Stochastic E4M3 rounding of 8 scaled values (|y| <= 448) with the group's
// random bits rb (value i uses the 16-bit half i % 2 of word i / 2): the
// magnitude codes in order (value 0 in the low byte of the first word); the
// caller ORs in the signs, four at a time, from the source bf16 words.
__device__ __forceinline__ uint2 e4m3x8_sr_mag(const float* y, const uint4& rb) {
  const uint32_t nw[4] = {~rb.x, ~rb.y, ~rb.z, ~rb.w};
  uint32_t x[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = e4m3_sr_mag_hi(y[i], e4m3_sr_n8(nw[i >> 1], i & 1));
  // the codes are the top bytes
  return make_uint2(__byte_perm(__byte_perm(x[0], x[1], 0x0073u),
                                __byte_perm(x[2], x[3], 0x0073u), 0x5410u),
                    __byte_perm(__byte_perm(x[4], x[5], 0x0073u),
                                __byte_perm(x[6], x[7], 0x0073u), 0x5410u));
}

// Row blocks: this thread's chunks k (8 values each, v[k]) under shared
// exponents ex[k]; writes codes and (one lane of four) the scale byte.
template <bool SR>
__device__ __forceinline__ void encode_rows(const MxParams& p, const uint4 (&v)[4],
                                            const int (&ex)[4], int64_t e0, int64_t step,
                                            const bool (&ok)[4], int lane) {
  const int64_t e[4] = {e0, e0 + step, e0 + 2 * step, e0 + 3 * step};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const f2 sc = make_float2(exp2_neg(ex[k]), exp2_neg(ex[k]));
    f2 x[4];
    unpack8(v[k], x);
    float y[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const f2 t = f2_mul(x[i], sc);
      y[2 * i] = t.x;
      y[2 * i + 1] = t.y;
    }
    uint2 codes;
    if constexpr (SR) {
      codes = e4m3x8_sr_mag(y, sr_group_bits(make_sr_key(p.seed, p.step), 0u, (uint64_t)e[k]));
      codes.x |= __byte_perm(v[k].x, v[k].y, 0x7531u) & 0x80808080u;  // signs of values 0..3
      codes.y |= __byte_perm(v[k].z, v[k].w, 0x7531u) & 0x80808080u;
    } else {
      codes = make_uint2(e4m3x4_rn(y[0], y[1], y[2], y[3]), e4m3x4_rn(y[4], y[5], y[6], y[7]));
    }
    if (ok[k]) {
      __stcs(reinterpret_cast<uint2*>(p.r_codes + e[k]), codes);
      if ((lane & 3) == 0) p.r_scales[e[k] >> 5] = (uint8_t)(ex[k] + 127);
    }
  }
}

// Column blocks: this lane's 16 rows (w[i] = columns cg, cg + 1 of row i)
// under shared exponents ex[0], ex[1]; ce = flat column-layout index of the
// first value of column cg.
template <bool SR>
__device__ __forceinline__ void encode_cols(const MxParams& p, const uint32_t (&w)[16],
                                            const int (&ex)[2], int64_t ce, bool ok0, bool ok1,
                                            bool write_scale) {
  uint32_t sg[2][4];  // signs of values 4k..4k+3 of each column
  if constexpr (SR) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t a = __byte_perm(w[4 * k], w[4 * k + 1], 0x7351u);
      const uint32_t b = __byte_perm(w[4 * k + 2], w[4 * k + 3], 0x7351u);
      sg[0][k] = __byte_perm(a, b, 0x5410u) & 0x80808080u;
      sg[1][k] = __byte_perm(a, b, 0x7632u) & 0x80808080u;
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // column cg + h
    const f2 sc = make_float2(exp2_neg(ex[h]), exp2_neg(ex[h]));
    float y[16];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const f2 t = f2_mul(h ? make_float2(bf16_hi(w[i]), bf16_hi(w[i + 1]))
                            : make_float2(bf16_lo(w[i]), bf16_lo(w[i + 1])), sc);
      y[i] = t.x;
      y[i + 1] = t.y;
    }
    const int64_t e = ce + h * p.R;
    uint2 a, b;
    if constexpr (SR) {
      a = e4m3x8_sr_mag(y, sr_group_bits(make_sr_key(p.seed, p.step), 1u, (uint64_t)e));
      b = e4m3x8_sr_mag(y + 8, sr_group_bits(make_sr_key(p.seed, p.step), 1u, (uint64_t)e + 8));
      a.x |= sg[h][0];
      a.y |= sg[h][1];
      b.x |= sg[h][2];
      b.y |= sg[h][3];
    } else {
      a = make_uint2(e4m3x4_rn(y[0], y[1], y[2], y[3]), e4m3x4_rn(y[4], y[5], y[6], y[7]));
      b = make_uint2(e4m3x4_rn(y[8], y[9], y[10], y[11]), e4m3x4_rn(y[12], y[13], y[14], y[15]));
    }
    if (h ? ok1 : ok0) {
      __stcs(reinterpret_cast<uint4*>(p.c_codes + e), make_uint4(a.x, a.y, b.x, b.y));
      if (write_scale) p.c_scales[e >> 5] = (uint8_t)(ex[h] + 127);
    }
  }
}

template <bool SR, bool ROWS, bool COLS>
__device__ __forceinline__ void mx_quant_tile(const MxParams& p, const TileGeom& geo) {
  __shared__ __align__(16) uint32_t tile[COLS ? TR * kWords : 4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t R = p.R, C = p.C;
  uint32_t s32, tr32, tc32;
  tile_of(blockIdx.x, geo, s32, tr32, tc32);
  const int64_t s = s32, r0 = (int64_t)tr32 * TR, c0 = (int64_t)tc32 * TC;
  const int64_t slice0 = s * geo.slice_elems;
  const bool vec = (C % 8) == 0;

  // ---- 1: load, flag non-finite values, encode the row blocks ------------
  // chunk k of this thread: row 16 k + t / 16, columns 8 (t % 16) .. of the tile
  const int lr0 = threadIdx.x / kChunksPerRow, lc = (threadIdx.x % kChunksPerRow) * 8;
  const int64_t e0 = slice0 + (r0 + lr0) * C + c0 + lc, step = (int64_t)(kThreads / kChunksPerRow) * C;
  const bool c_ok = c0 + lc < C;
  uint4 v[4];
  bool ok[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ok[k] = r0 + lr0 + 16 * k < R && c_ok;
    const int64_t ek = e0 + k * step;  // flat row-layout index
    v[k] = make_uint4(0, 0, 0, 0);
    if (ok[k]) {
      if (vec) {
        v[k] = __ldcs(reinterpret_cast<const uint4*>(p.x + ek));
      } else {  // column-only encoding of a tensor whose rows are not 16 B multiples
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = (c0 + lc + i < C) ? p.x[ek + i] : 0u;
        v[k] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                          h[6] | (h[7] << 16));
      }
    }
  }
  if constexpr (ROWS) {  // C % 32 == 0: a block's four chunks are all in range or all out
    int ex[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t m = absmax_bits4(v[k]);
      if (m >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      ex[k] = mx_shared_exp(__uint_as_float(m << 16));
    }
    encode_rows<SR>(p, v, ex, e0, step, ok, lane);
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (absmax_bits4(v[k]) >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
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
    int ex[2];
    ex[0] = mx_shared_exp(__uint_as_float(mm << 16));
    ex[1] = mx_shared_exp(__uint_as_float(mm & 0xFFFF0000u));
    const int64_t ce = (int64_t)s32 * geo.slice_elems + cg * R + r0 + 16 * q;  // column layout
    const bool ok0 = row_ok && cg < C, ok1 = row_ok && cg + 1 < C;
    encode_cols<SR>(p, w, ex, ce, ok0, ok1, (q & 1) == 0);
  }
}

// Two entry points for the register budget: the RNE kernels wait mostly on
// memory and run faster with 6 resident CTAs per SM (registers held to 40);
// the stochastic ones are bound by ALU issue and do best at the 57 registers
// the compiler picks with no bound (4 CTAs; held to 64 it takes 63 and runs
// 4 % slower).
template <bool ROWS, bool COLS>
__global__ void __launch_bounds__(kThreads, 6) mx_quant_rne_kernel(const MxParams p,
                                                                   const TileGeom geo) {
  pdl_begin();
  mx_quant_tile<false, ROWS, COLS>(p, geo);
}
template <bool ROWS, bool COLS>
__global__ void mx_quant_sr_kernel(const MxParams p, const TileGeom geo) {
  pdl_begin();
  mx_quant_tile<true, ROWS, COLS>(p, geo);
}

template <bool SR, bool ROWS, bool COLS>
cudaError_t launch_t(const MxParams& p, cudaStream_t st) {
  const int64_t tiles_r = (p.R + TR - 1) / TR, tiles_c = (p.C + TC - 1) / TC;
  const int64_t n = p.S * tiles_r * tiles_c;
  if (n > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const TileGeom geo = make_tile_geom(p.R, p.C, TR, TC);
  if constexpr (SR)
    return launch_pdl(mx_quant_sr_kernel<ROWS, COLS>, dim3((unsigned)n), dim3(kThreads), st, p,
                      geo);
  else
    return launch_pdl(mx_quant_rne_kernel<ROWS, COLS>, dim3((unsigned)n), dim3(kThreads), st, p,
                      geo);
}

}  // namespace

cudaError_t launch_mx_quant(const MxParams& p, bool rows, bool cols, bool sr, cudaStream_t st) {
  if (rows && cols)
    return sr ? launch_t<true, true, true>(p, st) : launch_t<false, true, true>(p, st);
  if (rows) return sr ? launch_t<true, true, false>(p, st) : launch_t<false, true, false>(p, st);
  return sr ? launch_t<true, false, true>(p, st) : launch_t<false, false, true>(p, st);
}

}  // namespace nvfp4
