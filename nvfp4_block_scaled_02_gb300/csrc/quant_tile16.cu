// quant_tile16.cu -- NVFP4 with one block scale per 16x16 tile (End-to-End
// 4-Bit Training, "Block-scaled backward passes": a single scale from the
// largest value of each 16x16 tile keeps the scales identical when the
// tensor is transposed).
//
// One CTA (256 threads) per 64 x 128 region of one slice (4 x 8 scale tiles):
//  1. thread t loads chunks k * 256 + t (k = 0..3) of 8 bf16 (a warp reads
//     two whole 256-byte rows per load) and stages them in a 16 KiB shared
//     tile of 32-bit words (two columns each), word w of row r stored at
//     w ^ (((r >> 4) & 3) << 3);
//  2. lane (cp, q) = (lane >> 2, lane & 3) of warp w reads rows 16q .. 16q+15
//     of column pair 8w + cp (conflict-free with the swizzle); the eight
//     lanes of one q cover scale tile (q, w), whose amax three xor shuffles
//     reduce; its scale is the 1x16 block scale of that amax (target 6),
//     published in shared memory with d and 1/d;
//  3. every thread encodes its 8-value chunks from registers with their
//     tile's scale (RNE, or stochastic with the row layout's random bits),
//     writes the row encoding and stages the code words in a shared code
//     tile (chunk index XOR-swizzled by the row's band);
//  4. the column encoding is the same codes transposed: lane (cp, q) gathers
//     the code byte of its column pair from each of its 16 rows (byte
//     permutes), splits the two columns' nibbles, and writes per column 8 code
//     bytes, the scale byte and 32 B of dequant; the four lanes of a column's
//     bands are adjacent, so each column's 64 rows leave contiguously.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int TR = 64;                 // region rows (4 scale tiles)
constexpr int TC = 128;                // region columns (8 scale tiles)
constexpr int kChunksPerRow = TC / 8;  // 16
constexpr int kWords = TC / 2;         // 32-bit words (column pairs) per row

__device__ __forceinline__ int word_of(int r, int w) {
  return r * kWords + (w ^ (((r >> 4) & 3) << 3));
}
__device__ __forceinline__ int code_of(int r, int ch) {
  return r * kChunksPerRow + (ch ^ (((r >> 4) & 3) << 2));
}

// The low (j = 0) or high (j = 1) nibbles of the 4 bytes of B, in order, as
// 16 bits.
__device__ __forceinline__ uint32_t nibbles4(uint32_t B, int j) {
  uint32_t x = (j ? (B >> 4) : B) & 0x0F0F0F0Fu;
  x = (x | (x >> 4)) & 0x00FF00FFu;
  return (x | (x >> 8)) & 0xFFFFu;
}

// Six resident CTAs per SM (registers held to 40, no spills): the kernel
// waits mostly on its loads, and 6 CTAs hide that latency better than the 4
// that an unbounded register count allows (92 vs 105 us on a 14336 x 4096
// weight).
template <int FMT, bool SR>
__global__ void __launch_bounds__(kThreads, 6) quant_tile16_kernel(const Tile16Params p,
                                                                int64_t tiles_r, int64_t tiles_c) {
  pdl_begin();
  __shared__ __align__(16) uint32_t tile[TR * kWords];
  __shared__ uint32_t s_codes[TR * kChunksPerRow];
  __shared__ float s_d[4][8], s_inv[4][8];
  __shared__ uint32_t s_code[4][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t R = p.R, C = p.C;
  const int64_t bid = blockIdx.x;
  const int64_t tc = bid % tiles_c, tr = (bid / tiles_c) % tiles_r, s = bid / (tiles_c * tiles_r);
  const int64_t r0 = tr * TR, c0 = tc * TC;
  const SliceScale ss = slice_scale(p.gamax[s], p.M);
  if (ss.bad && threadIdx.x == 0 && tr == 0 && tc == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);

  // ---- 1: load and stage (R, C are multiples of 16: a chunk is in or out) --
  uint4 v[4];
  bool ok[4];
  int64_t e[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int chunk = k * kThreads + threadIdx.x;
    const int lr = chunk / kChunksPerRow, lc = (chunk % kChunksPerRow) * 8;
    const int64_t r = r0 + lr, c = c0 + lc;
    ok[k] = r < R && c < C;
    e[k] = (s * R + r) * C + c;  // flat row-layout index
    v[k] = ok[k] ? __ldcs(p.x + e[k] / 8) : make_uint4(0, 0, 0, 0);
    if (absmax_bits4(v[k]) >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
    *reinterpret_cast<uint4*>(&tile[word_of(lr, (chunk % kChunksPerRow) * 4)]) = v[k];
  }
  __syncthreads();

  // ---- 2: tile amax and scale -----------------------------------------------
  const int q = lane & 3, cpl = warp * 8 + (lane >> 2);  // band, column pair
  {
    uint32_t mm = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) mm = __vmaxu2(mm, tile[word_of(16 * q + i, cpl)] & 0x7FFF7FFFu);
    uint32_t m = max(mm & 0xFFFFu, mm >> 16);
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
    if ((lane >> 2) == 0) {
      const uint32_t code = scale_encode<FMT>(__fmul_rn(__uint_as_float(m << 16), ss.rden6));
      float d, inv;
      scale_entry<FMT>(code, ss.g, d, inv);
      s_code[q][warp] = code;
      s_d[q][warp] = d;
      s_inv[q][warp] = inv;
    }
  }
  __syncthreads();

  // ---- 3: row encoding --------------------------------------------------------
  const bool want_dq = p.r_dq != nullptr, want_cols = p.c_codes != nullptr;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int chunk = k * kThreads + threadIdx.x;
    const int lr = chunk / kChunksPerRow, c16 = chunk % kChunksPerRow;
    const int tb = lr >> 4, tcol = c16 >> 1;
    uint4 rb = make_uint4(0, 0, 0, 0);
    if constexpr (SR) rb = sr_group_bits(p.seed, p.step, 0u, (uint64_t)e[k]);
    f2 x[4];
    unpack8(v[k], x);
    const uint32_t w = round8<SR>(x, s_inv[tb][tcol], rb);
    if (ok[k]) {
      p.r_codes[e[k] / 8] = w;
      if ((c16 & 1) == 0) p.r_scales[e[k] / 16] = (uint8_t)s_code[tb][tcol];
      if (want_dq) {
        f2 qv[4];
        e2m1x8_to_f2(w, qv);
        __stcs(p.r_dq + e[k] / 8, dequant8(qv, s_d[tb][tcol]));
      }
    }
    if (want_cols) s_codes[code_of(lr, c16)] = w;
  }
  if (!want_cols) return;  // block-uniform
  __syncthreads();

  // ---- 4: column encoding = the codes transposed -------------------------------
  const int64_t cc = c0 + 2 * cpl, rr = r0 + 16 * q;
  const int ch = cpl >> 2, bsel = cpl & 3;
  const uint32_t sel = (uint32_t)bsel | ((uint32_t)(bsel + 4) << 4);  // that byte of two words
  uint32_t B[4];  // code bytes of the column pair for rows 4g .. 4g+3 of the band
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t w0 = s_codes[code_of(16 * q + 4 * g, ch)];
    const uint32_t w1 = s_codes[code_of(16 * q + 4 * g + 1, ch)];
    const uint32_t w2 = s_codes[code_of(16 * q + 4 * g + 2, ch)];
    const uint32_t w3 = s_codes[code_of(16 * q + 4 * g + 3, ch)];
    B[g] = __byte_perm(__byte_perm(w0, w1, sel), __byte_perm(w2, w3, sel), 0x5410u);
  }
  const float d = s_d[q][warp];
  const uint32_t code = s_code[q][warp];
  const bool col_dq = p.c_dq != nullptr;
#pragma unroll
  for (int j = 0; j < 2; ++j) {  // column cc + j
    const uint32_t cw0 = nibbles4(B[0], j) | (nibbles4(B[1], j) << 16);
    const uint32_t cw1 = nibbles4(B[2], j) | (nibbles4(B[3], j) << 16);
    const int64_t ce = (s * C + cc + j) * R + rr;  // flat column-layout index
    if (rr < R && cc + j < C) {
      *reinterpret_cast<uint2*>(p.c_codes + ce / 8) = make_uint2(cw0, cw1);
      p.c_scales[ce / 16] = (uint8_t)code;
      if (col_dq) {
        f2 qv[4];
        e2m1x8_to_f2(cw0, qv);
        __stcs(p.c_dq + ce / 8, dequant8(qv, d));
        e2m1x8_to_f2(cw1, qv);
        __stcs(p.c_dq + ce / 8 + 1, dequant8(qv, d));
      }
    }
  }
}

template <int FMT, bool SR>
cudaError_t launch_t(const Tile16Params& p, cudaStream_t st) {
  const int64_t tiles_r = (p.R + TR - 1) / TR, tiles_c = (p.C + TC - 1) / TC;
  const int64_t n = p.S * tiles_r * tiles_c;
  if (n > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(quant_tile16_kernel<FMT, SR>, dim3((unsigned)n), dim3(kThreads), st, p,
                    tiles_r, tiles_c);
}

}  // namespace

cudaError_t launch_quant_tile16(const Tile16Params& p, int fmt, bool sr, cudaStream_t st) {
  if (fmt == 0) return sr ? launch_t<0, true>(p, st) : launch_t<0, false>(p, st);
  return sr ? launch_t<1, true>(p, st) : launch_t<1, false>(p, st);
}

}  // namespace nvfp4
