// quant_dual.cu -- NVFP4 quantisation with 16x1 column blocks, alone or
// together with the 1x16 row blocks from a single read of the input
// (End-to-End 4-Bit Training, "Block-scaled backward passes": the transposed
// operand groups each value with the 15 values above/below it instead).
//
// One CTA (256 threads) per 64 x 128 tile of one slice:
//  1. every thread loads 4 chunks of 8 bf16 (128-bit loads, a warp covers two
//     full 256 B tile rows) and, in BOTH mode, encodes the row blocks straight
//     from registers (lane pairs hold the two halves of a block);
//  2. the chunks go to a 16 KiB shared tile of 32-bit words (two columns
//     each), word w of row r stored at w ^ (((r >> 4) & 3) << 3);
//  3. lane (cp, q) = (lane >> 2, lane & 3) of warp w takes column pair
//     8w + cp in the 16-row band q: it reads one word per row (with the
//     swizzle the 32 lanes hit 32 distinct banks) and encodes the two column
//     blocks it now holds.
// Column outputs are the row encoding of X^T. The four bands of a column sit
// in four adjacent lanes, so each column's 64 rows go out contiguously from
// one store instruction: 32 code bytes, 4 scale bytes, 128 B of dequant (two
// instructions). Scattering a column's bands over four warps instead costs
// several partial-sector writes per sector.
// 4/6 bits are gathered per tile row (a ballot) and per column (a ballot over
// the four band lanes) and OR-ed into the (pre-zeroed) bitmaps, since a
// tile's bits share words with other tiles.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int TR = 64;    // tile rows
constexpr int TC = 128;   // tile columns
constexpr int kChunksPerRow = TC / 8;
constexpr int kWords = TC / 2;  // 32-bit words (column pairs) per tile row

__device__ __forceinline__ int word_of(int r, int w) {
  return r * kWords + (w ^ (((r >> 4) & 3) << 3));
}

__device__ __forceinline__ void or_bits(uint32_t* words, int64_t bit0, uint32_t bits, int nbits) {
  if (bits == 0) return;
  const int64_t w = bit0 >> 5;
  const int off = (int)(bit0 & 31);
  atomicOr(words + w, bits << off);
  if (off + nbits > 32) atomicOr(words + w + 1, bits >> (32 - off));
}

__device__ __forceinline__ uint32_t even_bits8(uint32_t b) {  // lanes 0,2,..,14 -> 8 bits
  b &= 0x5555u;
  b = (b | (b >> 1)) & 0x3333u;
  b = (b | (b >> 2)) & 0x0F0Fu;
  b = (b | (b >> 4)) & 0x00FFu;
  return b;
}

template <int FMT, bool SR, int FOS, bool ROWS>
__global__ void __launch_bounds__(kThreads) quant_dual_kernel(const DualParams p, int64_t tiles_r,
                                                              int64_t tiles_c) {
  pdl_begin();
  __shared__ __align__(16) uint32_t tile[TR * kWords];
  __shared__ float s_d[256], s_inv[256];

  const int64_t R = p.R, C = p.C;
  const int64_t bid = blockIdx.x;
  const int64_t tc = bid % tiles_c;
  const int64_t tr = (bid / tiles_c) % tiles_r;
  const int64_t s = bid / (tiles_c * tiles_r);
  const int64_t r0 = tr * TR, c0 = tc * TC;
  const int64_t slice_elems = R * C;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  const SliceScale ss = slice_scale(p.gamax[s], p.M);
  if (ss.bad && threadIdx.x == 0 && tr == 0 && tc == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
  build_scale_table<FMT>(s_d, s_inv, ss.g);

  // ---- 1 + 2: load, row-encode, stage ------------------------------------
  const uint16_t* xs = p.x + s * slice_elems;
  const bool vec = (C % 8) == 0;
  uint4 v[4];
  bool ok[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int chunk = k * kThreads + threadIdx.x;
    const int lr = chunk / kChunksPerRow, lc = (chunk % kChunksPerRow) * 8;
    const int64_t r = r0 + lr, c = c0 + lc;
    ok[k] = r < R && c < C;
    v[k] = make_uint4(0, 0, 0, 0);
    if (ok[k]) {
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
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int chunk = k * kThreads + threadIdx.x;
    const int lr = chunk / kChunksPerRow, lw = (chunk % kChunksPerRow) * 4;
    *reinterpret_cast<uint4*>(&tile[word_of(lr, lw)]) = v[k];
  }
  __syncthreads();  // tables and tile ready

  if constexpr (ROWS) {
    const bool want_dq = p.r_dq != nullptr;
    const int64_t Bs = slice_elems / 16, W = (Bs + 31) / 32;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int chunk = k * kThreads + threadIdx.x;
      const int lr = chunk / kChunksPerRow, lc = (chunk % kChunksPerRow) * 8;
      const int64_t r = r0 + lr, c = c0 + lc;
      f2 x[4];
      unpack8(v[k], x);
      uint32_t m = absmax_bits4(v[k]);
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      if (ok[k] && m >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
      const int64_t e = s * slice_elems + r * C + c;  // flat row-layout index
      uint4 rb = make_uint4(0, 0, 0, 0);
      if constexpr (SR) rb = sr_group_bits(p.seed, p.step, 0u, (uint64_t)e);
      const HalfResult hr = encode_half<FMT, SR, FOS != 0>(x, m, ss, s_d, s_inv, rb, want_dq,
                                                              FOS == 2 ? p.rule : 0);
      if (ok[k]) {
        reinterpret_cast<uint32_t*>(p.r_codes)[e / 8] = hr.codes;
        if (want_dq) __stcs(reinterpret_cast<uint4*>(p.r_dq + e), hr.dq);
        if ((lane & 1) == 0) p.r_scales[e / 16] = (uint8_t)hr.scale;
      }
      if constexpr (FOS) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, ok[k] && hr.pick4);
        if ((lane & 15) == 0 && ok[k]) {
          const uint32_t bits = even_bits8(b >> (lane & 16));
          const int64_t blk = (r * C + c) / 16;  // block index within the slice
          const int64_t nb = (C - c) / 16 < 8 ? (C - c) / 16 : 8;
          or_bits(p.r_choice + s * W, blk, bits, (int)nb);
        }
      }
    }
  }

  // ---- 3: column blocks ---------------------------------------------------
  {
    const bool want_dq = p.c_dq != nullptr;
    const int q = lane & 3, cpl = warp * 8 + (lane >> 2);  // band, column pair
    const int64_t c = c0 + 2 * cpl, r = r0 + 16 * q;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = tile[word_of(16 * q + i, cpl)];
    uint32_t mm = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) mm = __vmaxu2(mm, w[i] & 0x7FFF7FFFu);
#pragma unroll
    for (int j = 0; j < 2; ++j) {  // column c + j
      const uint32_t m = j ? (mm >> 16) : (mm & 0xFFFFu);
      f2 lo[4], hi[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        lo[k] = j ? make_float2(bf16_hi(w[2 * k]), bf16_hi(w[2 * k + 1]))
                  : make_float2(bf16_lo(w[2 * k]), bf16_lo(w[2 * k + 1]));
        hi[k] = j ? make_float2(bf16_hi(w[8 + 2 * k]), bf16_hi(w[9 + 2 * k]))
                  : make_float2(bf16_lo(w[8 + 2 * k]), bf16_lo(w[9 + 2 * k]));
      }
      const bool okc = c + j < C && r < R;
      if (okc && m >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
      const int64_t e = s * slice_elems + (c + j) * R + r;  // flat column-layout index
      uint4 rb0 = make_uint4(0, 0, 0, 0), rb1 = rb0;
      if constexpr (SR) {
        rb0 = sr_group_bits(p.seed, p.step, 1u, (uint64_t)e);
        rb1 = sr_group_bits(p.seed, p.step, 1u, (uint64_t)e + 8);
      }
      const BlockResult br =
          encode_block<FMT, SR, FOS != 0>(lo, hi, m, ss, TableScales{s_d, s_inv}, rb0, rb1,
                                          want_dq, FOS == 2 ? p.rule : 0);
      if (okc) {
        *reinterpret_cast<uint2*>(p.c_codes + e / 2) = make_uint2(br.codes[0], br.codes[1]);
        p.c_scales[e / 16] = (uint8_t)br.scale;
        if (want_dq) {
          __stcs(reinterpret_cast<uint4*>(p.c_dq + e), br.dq[0]);
          __stcs(reinterpret_cast<uint4*>(p.c_dq + e) + 1, br.dq[1]);
        }
      }
      if constexpr (FOS) {
        // bands 0..3 of this column are lanes 4cp .. 4cp+3: its 4 bits
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, okc && br.pick4);
        if (q == 0 && c + j < C) {
          const int64_t Bs = slice_elems / 16, W = (Bs + 31) / 32;
          const int64_t nb = (R - r0) / 16 < 4 ? (R - r0) / 16 : 4;
          or_bits(p.c_choice + s * W, (c + j) * (R / 16) + r0 / 16, (b >> (lane & ~3)) & 15u,
                  (int)nb);
        }
      }
    }
  }
}

template <int FMT, bool SR, int FOS, bool ROWS>
cudaError_t launch_t(const DualParams& p, int64_t S, cudaStream_t st) {
  const int64_t tiles_r = (p.R + TR - 1) / TR, tiles_c = (p.C + TC - 1) / TC;
  const int64_t n = S * tiles_r * tiles_c;
  if (n > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(quant_dual_kernel<FMT, SR, FOS, ROWS>, dim3((unsigned)n), dim3(kThreads), st,
                    p, tiles_r, tiles_c);
}

}  // namespace

cudaError_t launch_quant_dual(const DualParams& p, int64_t S, bool rows_too, int fmt, bool sr,
                              int fos, cudaStream_t st) {
#define NVFP4_DUAL(F, R, O, B) \
  if (fmt == F && sr == R && fos == O && rows_too == B) return launch_t<F, R, O, B>(p, S, st);
#define NVFP4_DUAL_FOS(F, R, B) NVFP4_DUAL(F, R, 0, B) NVFP4_DUAL(F, R, 1, B) NVFP4_DUAL(F, R, 2, B)
  NVFP4_DUAL_FOS(0, false, false) NVFP4_DUAL_FOS(0, true, false)
  NVFP4_DUAL_FOS(1, false, false) NVFP4_DUAL_FOS(1, true, false)
  NVFP4_DUAL_FOS(0, false, true) NVFP4_DUAL_FOS(0, true, true)
  NVFP4_DUAL_FOS(1, false, true) NVFP4_DUAL_FOS(1, true, true)
#undef NVFP4_DUAL_FOS
#undef NVFP4_DUAL
  return cudaErrorInvalidValue;
}

}  // namespace nvfp4
