// quant_tile16.cu -- NVFP4 with one block scale per 16x16 tile (End-to-End
// 4-Bit Training, "Block-scaled backward passes": a single scale from the
// largest value of each 16x16 tile keeps the scales identical when the
// tensor is transposed).
//
// One CTA (256 threads) per 64 x 128 region of one slice (4 x 8 scale tiles):
//  1. thread t loads chunks k * 256 + t (k = 0..3) of 8 bf16 (a warp reads
//     two whole 256-byte rows per load); chunk k of thread t lies in band k
//     and tile column (t % 16) / 2, so within a warp the lanes l, l ^ 1,
//     l ^ 16, l ^ 17 hold that tile column's chunks of the warp's two rows:
//     two xor shuffles combine them and one shared-memory atomic max per
//     tile and warp gives the tile amax;
//  2. after one barrier every thread turns its tiles' amaxes into scales (the
//     1x16 block scale of the amax, target 6), encodes its chunks from
//     registers (RNE, or stochastic with the row layout's random bits),
//     writes the row encoding and stages the code words in a shared code
//     tile (chunk index XOR-swizzled by the row's band);
//  3. the column encoding is the same codes transposed: lane (cp, q) =
//     (lane >> 2, lane & 3) of warp w takes column pair 8w + cp in band q,
//     gathers the code byte of its column pair from each of its 16 rows (byte
//     permutes), splits the two columns' nibbles, and writes per column 8 code
//     bytes, the scale byte and 32 B of dequant; the four lanes of a column's
//     bands are adjacent, so each column's 64 rows leave contiguously.
// (Staging the bf16 region in shared memory to take the tile amaxes in a
// column-mapped pass cost a barrier and 16 KiB per CTA: 92.6 vs 77.4 us.)
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int TR = 64;                 // region rows (4 scale tiles)
constexpr int TC = 128;                // region columns (8 scale tiles)
constexpr int kChunksPerRow = TC / 8;  // 16
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

// Six resident CTAs per SM (registers held to 40): the stochastic and UE5M3
// variants then spill 16 bytes, and still run faster than with 5 CTAs
// (E4M3 with SR: 101.1 vs 103.6 us on a 14336 x 4096 weight).
template <int FMT, bool SR>
__global__ void __launch_bounds__(kThreads, 6) quant_tile16_kernel(const Tile16Params p,
                                                                const TileGeom geo) {
  pdl_begin();
  __shared__ uint32_t s_codes[TR * kChunksPerRow];
  __shared__ uint32_t s_tmax[4][8];  // bf16 bits of each scale tile's amax
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t R = p.R, C = p.C;
  uint32_t s32, tr32, tc32;
  tile_of(blockIdx.x, geo, s32, tr32, tc32);
  const int64_t s = s32, r0 = (int64_t)tr32 * TR, c0 = (int64_t)tc32 * TC;
  const int64_t slice0 = s * geo.slice_elems;

  // ---- 1: loads (thread t's chunk k lies in band k, tile column (t % 16) / 2)
  // chunk k of thread t: row 16 k + t / 16, columns 8 (t % 16) .. of the region
  const int lr0 = tid / kChunksPerRow, lc = (tid % kChunksPerRow) * 8;
  const int64_t e0 = slice0 + (r0 + lr0) * C + c0 + lc, step = (int64_t)(kThreads / kChunksPerRow) * C;
  uint4 v[4];
  bool ok[4];
  int64_t e[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ok[k] = r0 + lr0 + 16 * k < R && c0 + lc < C;
    e[k] = e0 + k * step;  // flat row-layout index
    v[k] = ok[k] ? __ldcs(p.x + (e[k] >> 3)) : make_uint4(0, 0, 0, 0);
  }
  if (tid < 32) (&s_tmax[0][0])[tid] = 0u;
  const SliceScale ss = slice_scale(p.gamax[s], p.M);
  if (ss.bad && tid == 0 && tr32 == 0 && tc32 == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
  __syncthreads();  // s_tmax zeroed
  const int tcol = (tid % kChunksPerRow) >> 1;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t m = absmax_bits4(v[k]);
    if (m >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
    // lanes l, l ^ 1, l ^ 16, l ^ 17 hold this tile column's chunks of the warp's two rows
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
    if ((lane & 17) == 0) atomicMax(&s_tmax[k][tcol], m);
  }
  __syncthreads();  // tile amaxes complete

  // ---- 2: row encoding with the tile's scale (computed by every thread) ----------
  const bool want_dq = p.r_dq != nullptr, want_cols = p.c_codes != nullptr;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int chunk = k * kThreads + tid;
    const int lr = chunk / kChunksPerRow, c16 = chunk % kChunksPerRow;
    const uint32_t code = scale_encode<FMT>(__fmul_rn(__uint_as_float(s_tmax[k][tcol] << 16), ss.rden6));
    float d, inv;
    scale_entry<FMT>(code, ss.g, d, inv);
    uint4 rb = make_uint4(0, 0, 0, 0);
    if constexpr (SR) rb = sr_group_bits(make_sr_key(p.seed, p.step), 0u, (uint64_t)e[k]);
    f2 x[4];
    unpack8(v[k], x);
    const uint32_t w = round8<SR>(x, inv, rb);
    if (ok[k]) {
      p.r_codes[e[k] >> 3] = w;
      if ((c16 & 1) == 0) p.r_scales[e[k] >> 4] = (uint8_t)code;
      if (want_dq) {
        f2 qv[4];
        e2m1x8_to_f2(w, qv);
        __stcs(p.r_dq + (e[k] >> 3), dequant8(qv, d));
      }
    }
    if (want_cols) s_codes[code_of(lr, c16)] = w;
  }
  if (!want_cols) return;  // block-uniform
  __syncthreads();

  // ---- 3: column encoding = the codes transposed ---------------------------------
  const int q = lane & 3, cpl = warp * 8 + (lane >> 2);  // band, column pair
  const int64_t cc = c0 + 2 * cpl, rr = r0 + 16 * q;
  const int ch = cpl >> 2, bsel = cpl & 3;
  const uint32_t sel = (uint32_t)bsel | ((uint32_t)(bsel + 4) << 4);
  uint32_t B[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t w0 = s_codes[code_of(16 * q + 4 * g, ch)];
    const uint32_t w1 = s_codes[code_of(16 * q + 4 * g + 1, ch)];
    const uint32_t w2 = s_codes[code_of(16 * q + 4 * g + 2, ch)];
    const uint32_t w3 = s_codes[code_of(16 * q + 4 * g + 3, ch)];
    B[g] = __byte_perm(__byte_perm(w0, w1, sel), __byte_perm(w2, w3, sel), 0x5410u);
  }
  const uint32_t code = scale_encode<FMT>(__fmul_rn(__uint_as_float(s_tmax[q][warp] << 16), ss.rden6));
  float d, inv;
  scale_entry<FMT>(code, ss.g, d, inv);
  const bool col_dq = p.c_dq != nullptr;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t cw0 = nibbles4(B[0], j) | (nibbles4(B[1], j) << 16);
    const uint32_t cw1 = nibbles4(B[2], j) | (nibbles4(B[3], j) << 16);
    const int64_t ce = slice0 + (cc + j) * R + rr;
    if (rr < R && cc + j < C) {
      *reinterpret_cast<uint2*>(p.c_codes + (ce >> 3)) = make_uint2(cw0, cw1);
      p.c_scales[ce >> 4] = (uint8_t)code;
      if (col_dq) {
        f2 qv[4];
        e2m1x8_to_f2(cw0, qv);
        __stcs(p.c_dq + (ce >> 3), dequant8(qv, d));
        e2m1x8_to_f2(cw1, qv);
        __stcs(p.c_dq + (ce >> 3) + 1, dequant8(qv, d));
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
                    make_tile_geom(p.R, p.C, TR, TC));
}

}  // namespace

cudaError_t launch_quant_tile16(const Tile16Params& p, int fmt, bool sr, cudaStream_t st) {
  if (fmt == 0) return sr ? launch_t<0, true>(p, st) : launch_t<0, false>(p, st);
  return sr ? launch_t<1, true>(p, st) : launch_t<1, false>(p, st);
}

}  // namespace nvfp4
