// requant.cu -- backward-operand re-quantisation (End-to-End 4-Bit Training,
// "Re-quantization with stochastic rounding" and its quantised-linear-layer
// figure): the forward NVFP4 row encoding of X [S][R][C] is de-quantised to
// fp32, transposed, and re-quantised along the other axis, by stochastic
// rounding (or RNE), either to MXFP8 (E4M3 values, one power-of-two E8M0
// scale per 32) or to NVFP4 (the row encoding of the transposed values).
//
// One CTA (256 threads) per 64 (R) x 128 (C) tile; persistent CTAs walk the
// tiles grid-stride:
//  1. each thread loads two 16-code blocks (8 bytes of codes + 1 scale byte
//     each; a warp reads four 64 B row segments) and de-quantises them into a
//     32 KiB fp32 shared tile;
//  2. each warp re-encodes 16 columns: lane (cp, q) reads rows 16q .. 16q+15
//     of columns 2cp, 2cp + 1 of its group with 8-byte loads and encodes one
//     column after the other (16 values: one NVFP4 block; MX blocks of 32
//     pair lanes q, q^1, which combine their amax with one shuffle). A warp's
//     store then covers 8 columns x 64 contiguous bytes (MX) or 32 bytes
//     (NVFP4) of the transposed output.
// Tile layout in shared memory: row-major fp32, the float4 slot j of row r
// stored at j ^ ((j >> 2) & 7) ^ 2((r >> 4) & 3). The first term spreads the
// eight lanes that store one row's blocks over all banks; the second the four
// lanes (16 rows apart) that read one column pair.
// The next tile's codes are loaded into registers while the current one is
// encoded. The de-quantised value of a code is q * d with d = dec(scale) * g
// from a per-slice 256-entry table; the NVFP4 target takes d and 1/d of its
// own scales from a second table. A column's 4/6 bits of one tile are
// adjacent: they are gathered by a ballot and OR-ed into the pre-zeroed
// bitmap with one atomic per column.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int TR = 64;          // tile rows (the re-quantised axis)
constexpr int TC = 128;         // tile columns
constexpr int kSlots = TC / 4;  // float4 slots per tile row

__device__ __forceinline__ int slot_of(int r, int j) {
  return j ^ ((j >> 2) & 7) ^ (((r >> 4) & 3) << 1);
}
// word offset of element (r, c) of the tile
__device__ __forceinline__ int tile_word(int r, int c) {
  return r * TC + 4 * slot_of(r, c >> 2) + (c & 3);
}

// Per-slice tables: de-quantisation d of every source scale code and, for an
// NVFP4 target, d and 1/d of every target scale code.
template <int DFMT, bool NV>
__device__ __forceinline__ void build_tables(const RequantParams& p, int64_t s, float* s_src,
                                             float* s_d, float* s_inv, SliceScale& ss_dst) {
  const float gam = p.gamax[s];
  const SliceScale src = slice_scale(gam, p.M_src);
  ss_dst = slice_scale(gam, p.M_dst);
  const uint32_t c = threadIdx.x;  // 256 threads, one code each
  s_src[c] = __fmul_rn(p.src_fmt == 0 ? e4m3_value(c) : ue5m3_value(c), src.g);
  if constexpr (NV) scale_entry<DFMT>(c, ss_dst.g, s_d[c], s_inv[c]);
  if (threadIdx.x == 0 && (src.bad || (NV && ss_dst.bad))) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
}

// Tiles are numbered slice-major, then by row tile, with the column tiles
// fastest, and dealt to the CTAs grid-stride: the CTAs running at one time
// hold every column tile of a few row bands, so the DRAM pages of those
// source rows are read in full by neighbouring requests, and each output row
// receives one contiguous run of a few row bands. A CTA advances its tile by
// the grid size with a cursor: one division when it starts, then adds with
// carries (the grid size split once into whole row bands and a remainder).
struct TileCursor {
  int64_t s, rt, ct;
  __device__ __forceinline__ void start(int64_t t, int64_t tiles_r, int64_t tiles_c) {
    const int64_t per = tiles_r * tiles_c;
    s = t / per;
    const int64_t rem = t - s * per;
    rt = rem / tiles_c;
    ct = rem - rt * tiles_c;
  }
  // advance by G = g_rows * tiles_c + g_cols tiles (g_cols < tiles_c)
  __device__ __forceinline__ void next(int64_t g_rows, int64_t g_cols, int64_t tiles_r,
                                       int64_t tiles_c) {
    ct += g_cols;
    rt += g_rows;
    if (ct >= tiles_c) {
      ct -= tiles_c;
      ++rt;
    }
    if (rt >= tiles_r) {  // into a later slice
      const int64_t k = rt / tiles_r;
      s += k;
      rt -= k * tiles_r;
    }
  }
  __device__ __forceinline__ int64_t r0() const { return rt * TR; }
  __device__ __forceinline__ int64_t c0() const { return ct * TC; }
};

// The two source blocks of this thread: blocks tid and tid + 256 of the
// tile's 64 x 8 blocks (block bi: row bi >> 3, column block bi & 7), i.e.
// rows (tid >> 3) and (tid >> 3) + 32 of column block tid & 7. Their element
// offsets from the tile's first element are fixed per thread.
struct SrcRegs {
  uint2 codes[2];
  uint32_t scale[2];
};
struct SrcLayout {
  int64_t off0;   // (tid >> 3) * C + 16 * (tid & 7)
  int row0, col0; // (tid >> 3), 16 * (tid & 7)
};
__device__ __forceinline__ void load_src(const RequantParams& p, bool valid, const TileCursor& ti,
                                         const SrcLayout& L, SrcRegs& v) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    v.codes[k] = make_uint2(0, 0);
    v.scale[k] = 0;
  }
  if (!valid) return;
  const int64_t r0 = ti.r0(), c0 = ti.c0();
  const int64_t base = (ti.s * p.R + r0) * p.C + c0;  // block-uniform
  if (c0 + L.col0 < p.C) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (r0 + L.row0 + 32 * k < p.R) {
        const int64_t e = base + L.off0 + k * 32 * p.C;  // flat element index, e % 16 == 0
        v.codes[k] = __ldcs(reinterpret_cast<const uint2*>(p.codes + (e >> 1)));
        v.scale[k] = __ldcs(p.scales + (e >> 4));
      }
    }
  }
}

template <bool SR>
__device__ __forceinline__ uint4 sr_bits_or_zero(const RequantParams& p, uint64_t idx0) {
  if constexpr (SR) return sr_group_bits(p.key, 2u, idx0);
  else return make_uint4(0, 0, 0, 0);
}

// 8 scaled values -> 8 E4M3 codes by stochastic rounding with the group's
// random bits rb (two words, element 0 in the low byte of the first).
__device__ __forceinline__ uint2 e4m3x8_sr(const float* y, const uint4& rb) {
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

// Resident CTAs per SM the register allocation is held to (the kernel is
// latency-bound below this). At these counts only the NVFP4 target with E4M3
// scales, stochastic rounding and 4/6 off spills (4 bytes); the NVFP4 target
// with stochastic rounding and a runtime 4/6 rule would spill at 3.
constexpr int min_blocks(int target, bool sr, int fos) {
  return target == 0 ? 4 : (sr && fos == 2 ? 2 : 3);
}

// TARGET 0: MXFP8; TARGET 1: NVFP4 with block-scale format DFMT and 4/6 mode
// FOS (0 off, 1 MSE, 2 rule from the params).
template <int TARGET, int DFMT, bool SR, int FOS>
__global__ void __launch_bounds__(kThreads, min_blocks(TARGET, SR, FOS)) requant_kernel(const RequantParams p, int64_t tiles_r,
                                                           int64_t tiles_c) {
  pdl_begin();
  constexpr bool NV = TARGET == 1;
  __shared__ __align__(16) float4 s_x[TR * kSlots];
  __shared__ float s_src[256];
  __shared__ float s_d[NV ? 256 : 1], s_inv[NV ? 256 : 1];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = lane & 3, cp = lane >> 2;  // phase 2: 16-row quarter, column pair
  const int64_t total = p.S * tiles_r * tiles_c;
  const int64_t R = p.R, C = p.C;
  const float* xs = reinterpret_cast<const float*>(s_x);

  // this CTA's tiles: blockIdx.x, + G, + 2G, ...
  const int64_t G = gridDim.x;
  const int64_t ntiles = (total - blockIdx.x + G - 1) / G;
  const int64_t g_rows = G / tiles_c, g_cols = G - g_rows * tiles_c;
  TileCursor ti, tn;
  ti.start(blockIdx.x, tiles_r, tiles_c);
  tn = ti;

  SrcLayout L;
  L.row0 = tid >> 3;
  L.col0 = 16 * (tid & 7);
  L.off0 = (int64_t)L.row0 * C + L.col0;
  // phase 2: this lane's columns cpair, cpair + 1 and the element offset of
  // its first value from the tile's first output element
  const int cpair = 16 * warp + 2 * cp;
  const int64_t out_off0 = (int64_t)cpair * R + 16 * q;

  SrcRegs v;
  load_src(p, ntiles > 0, ti, L, v);
  int64_t cur_slice = -1;
  // 4/6 bitmap of the current slice, and the flat index of its first block
  const int64_t W = (R * C / 16 + 31) / 32;
  uint32_t* words = p.out_choice;
  int64_t slice_b0 = 0;
  SliceScale ss_dst{};
  for (int64_t it = 0; it < ntiles; ++it) {  // block-uniform
    ti = tn;
    tn.next(g_rows, g_cols, tiles_r, tiles_c);
    if (ti.s != cur_slice) {  // block-uniform; the previous tile ended with a barrier
      build_tables<DFMT, NV>(p, ti.s, s_src, s_d, s_inv, ss_dst);
      cur_slice = ti.s;
      if constexpr (NV && FOS != 0) {
        words = p.out_choice + ti.s * W;
        slice_b0 = ti.s * (R * C / 16);
      }
      __syncthreads();
    }
    // ---- 1: de-quantise this thread's two blocks into the tile ---------
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int bi = k * kThreads + tid;
      const int row = bi >> 3, cb = bi & 7;
      const float d = s_src[v.scale[k]];
      f2 qv[4];
      float4* dst = s_x + row * kSlots;
      const f2 dd = make_float2(d, d);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        e2m1x8_to_f2(h ? v.codes[k].y : v.codes[k].x, qv);
        const f2 a = f2_mul(qv[0], dd), b = f2_mul(qv[1], dd), c = f2_mul(qv[2], dd),
                 e = f2_mul(qv[3], dd);
        // q * d overflows only when d > FLT_MAX / 6 (g near FLT_MAX): then
        // look at the products themselves
        if (d > 5.0e37f &&
            !(fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y))),
                    fmaxf(fmaxf(fabsf(c.x), fabsf(c.y)), fmaxf(fabsf(e.x), fabsf(e.y)))) <=
              kFltMax))
          flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
        dst[slot_of(row, 4 * cb + 2 * h)] = make_float4(a.x, a.y, b.x, b.y);
        dst[slot_of(row, 4 * cb + 2 * h + 1)] = make_float4(c.x, c.y, e.x, e.y);
      }
    }
    load_src(p, it + 1 < ntiles, tn, L, v);  // next tile in flight
    __syncthreads();

    // ---- 2: re-encode; lane (cp, q) takes columns cpair, cpair + 1 -----
    const int64_t r0 = ti.r0(), c0 = ti.c0();
    const int64_t out_base = (ti.s * C + c0) * R + r0;  // block-uniform
    const bool row_ok = r0 + 16 * q < R;  // R % 32 (MX) or % 16: whole blocks
    // rows 16q .. 16q+15 share the swizzle term of row 16q: one base address,
    // then fixed offsets of one tile row per value; 8-byte reads of 2 columns
    const float2* xc = reinterpret_cast<const float2*>(xs + tile_word(16 * q, cpair));
    float2 xv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) xv[i] = xc[i * (TC / 2)];
    if constexpr (!NV) {
      // both columns at once: amax, shared exponent, scaling (packed)
      float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        m0 = fmax3(m0, fabsf(xv[i].x), fabsf(xv[i + 1].x));
        m1 = fmax3(m1, fabsf(xv[i].y), fabsf(xv[i + 1].y));
      }
      // MX block of 32 = quarters q and q ^ 1
      m0 = fmaxf(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, 1));
      m1 = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, 1));
      const int ex0 = mx_shared_exp(m0), ex1 = mx_shared_exp(m1);
      const f2 scv = make_float2(exp2_neg(ex0), exp2_neg(ex1));
      f2 y[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = f2_mul(xv[i], scv);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = cpair + h;
        const bool ok = row_ok && c0 + c < C;
        const int64_t e0 = out_base + out_off0 + h * R;  // flat output index of y[0].h
        float yc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) yc[i] = h ? y[i].y : y[i].x;
        uint4 w;
        if constexpr (!SR) {
          w = make_uint4(e4m3x4_rn(yc[0], yc[1], yc[2], yc[3]), e4m3x4_rn(yc[4], yc[5], yc[6], yc[7]),
                         e4m3x4_rn(yc[8], yc[9], yc[10], yc[11]),
                         e4m3x4_rn(yc[12], yc[13], yc[14], yc[15]));
        } else {
          const uint2 a = e4m3x8_sr(yc, sr_group_bits(p.key, 2u, (uint64_t)e0));
          const uint2 b = e4m3x8_sr(yc + 8, sr_group_bits(p.key, 2u, (uint64_t)e0 + 8));
          w = make_uint4(a.x, a.y, b.x, b.y);
        }
        if (ok) {
          __stcs(reinterpret_cast<uint4*>(p.out_codes + e0), w);
          if ((q & 1) == 0) p.out_scales[e0 >> 5] = (uint8_t)((h ? ex1 : ex0) + 127);
        }
      }
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = cpair + h;
        const bool ok = row_ok && c0 + c < C;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = h ? xv[i].y : xv[i].x;
        const int64_t e0 = out_base + out_off0 + h * R;  // flat output index of x[0]
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; i += 2) amax = fmax3(amax, fabsf(x[i]), fabsf(x[i + 1]));
        f2 lo[4], hi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          lo[k] = make_float2(x[2 * k], x[2 * k + 1]);
          hi[k] = make_float2(x[8 + 2 * k], x[8 + 2 * k + 1]);
        }
        const BlockResult r = encode_block_f<DFMT, SR, FOS != 0>(
            lo, hi, amax, ss_dst, TableScales{s_d, s_inv}, sr_bits_or_zero<SR>(p, (uint64_t)e0),
            sr_bits_or_zero<SR>(p, (uint64_t)e0 + 8), false, FOS == 2 ? p.rule : 0);
        if (ok) {
          __stcs(reinterpret_cast<uint2*>(p.out_codes + (e0 >> 1)), make_uint2(r.codes[0], r.codes[1]));
          p.out_scales[e0 >> 4] = (uint8_t)r.scale;
        }
        if constexpr (FOS != 0) {
          // bits of this column's 4 blocks: lanes 4 cp .. 4 cp + 3
          const uint32_t bits =
              (__ballot_sync(0xFFFFFFFFu, ok && r.pick4) >> (4 * cp)) & 0xFu;
          if (q == 0 && bits) {
            const int64_t b0 = (e0 >> 4) - slice_b0;  // block index within the slice
            const int off = (int)(b0 & 31);
            atomicOr(words + (b0 >> 5), bits << off);
            if (off > 28 && (bits >> (32 - off))) atomicOr(words + (b0 >> 5) + 1, bits >> (32 - off));
          }
        }
      }
    }
    __syncthreads();  // tile reads done
  }
}

template <int TARGET, int DFMT, bool SR, int FOS>
cudaError_t launch_t(const RequantParams& p, cudaStream_t st) {
  const int64_t tiles_r = (p.R + TR - 1) / TR, tiles_c = (p.C + TC - 1) / TC;
  const int64_t total = p.S * tiles_r * tiles_c;
  auto k = requant_kernel<TARGET, DFMT, SR, FOS>;
  const int64_t cap = (int64_t)sm_count() * resident_ctas(k, kThreads);
  const unsigned grid = (unsigned)(total < cap ? total : cap);
  return launch_pdl(k, dim3(grid), dim3(kThreads), st, p, tiles_r, tiles_c);
}

template <int DFMT, bool SR>
cudaError_t launch_nv(const RequantParams& p, int fos, cudaStream_t st) {
  if (fos == 0) return launch_t<1, DFMT, SR, 0>(p, st);
  if (fos == 1) return launch_t<1, DFMT, SR, 1>(p, st);
  return launch_t<1, DFMT, SR, 2>(p, st);
}

}  // namespace

cudaError_t launch_requant(const RequantParams& p, int target, int dst_fmt, bool sr, int fos,
                           cudaStream_t st) {
  if (target == 0) return sr ? launch_t<0, 0, true, 0>(p, st) : launch_t<0, 0, false, 0>(p, st);
  if (dst_fmt == 0) return sr ? launch_nv<0, true>(p, fos, st) : launch_nv<0, false>(p, fos, st);
  return sr ? launch_nv<1, true>(p, fos, st) : launch_nv<1, false>(p, fos, st);
}

}  // namespace nvfp4
