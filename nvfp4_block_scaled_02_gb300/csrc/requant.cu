// requant.cu -- backward-operand re-quantisation (End-to-End 4-Bit Training,
// "Re-quantization with stochastic rounding" and its quantised-linear-layer
// figure): the forward NVFP4 row encoding of X [S][R][C] is de-quantised to
// fp32, transposed, and re-quantised along the other axis, by stochastic
// rounding (or RNE), either to MXFP8 (E4M3 values, one power-of-two E8M0
// scale per 32) or to NVFP4 (the row encoding of the transposed values).
//
// One CTA (256 threads) per 64 (R) x 128 (C) tile, persistent over tiles:
//  1. each thread loads two 16-code blocks (8 bytes of codes + 1 scale byte
//     each; a warp reads four 64 B row segments) and de-quantises them into a
//     32 KiB fp32 shared tile. The tile is stored row-major with the float4
//     slots of each row XOR-swizzled (slot j at j ^ ((j >> 2) & 7)), so the
//     eight lanes that store one row's blocks hit distinct banks.
//  2. each warp takes 32 consecutive columns of one 32-row band: lane l reads
//     its column (one fp32 per row, 32 consecutive words: conflict-free) and
//     encodes it -- one MX block of 32, or two NVFP4 blocks of 16 -- straight
//     into 32 B (MX) or 16 B (NVFP4) of the transposed output.
// The next tile's codes are loaded into registers while the current one is
// encoded. The de-quantised value of a code is q * d with d = dec(scale) * g
// from a per-slice 256-entry table; the NVFP4 target takes d and 1/d of its
// own scales from a second table. 4/6 bits are gathered per column in shared
// memory and OR-ed into the pre-zeroed bitmap, a column's bits of one tile
// being adjacent.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int TR = 64;   // tile rows (the re-quantised axis)
constexpr int TC = 128;  // tile columns
constexpr int kSlots = TC / 4;  // float4 slots per tile row

__device__ __forceinline__ int swz(int j) { return j ^ ((j >> 2) & 7); }
// word offset of element (r, c) of the swizzled tile
__device__ __forceinline__ int tile_word(int r, int c) {
  return r * TC + 4 * swz(c >> 2) + (c & 3);
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

// Tile t of the grid's tile order: slice, then column tiles, with the row
// tiles fastest (consecutive tiles extend the same output rows).
struct TileIdx {
  int64_t s, r0, c0;
};
__device__ __forceinline__ TileIdx tile_of(int64_t t, int64_t tiles_r, int64_t tiles_c) {
  TileIdx ti;
  const int64_t per = tiles_r * tiles_c;
  ti.s = t / per;
  const int64_t rem = t - ti.s * per;
  ti.c0 = (rem / tiles_r) * TC;
  ti.r0 = (rem % tiles_r) * TR;
  return ti;
}

// The two source blocks of this thread: blocks tid and tid + 256 of the
// tile's 64 x 8 blocks (block bi: row bi >> 3, column block bi & 7).
struct SrcRegs {
  uint2 codes[2];
  uint32_t scale[2];
};
__device__ __forceinline__ void load_src(const RequantParams& p, int64_t t, int64_t total,
                                         int64_t tiles_r, int64_t tiles_c, SrcRegs& v) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    v.codes[k] = make_uint2(0, 0);
    v.scale[k] = 0;
  }
  if (t >= total) return;
  const TileIdx ti = tile_of(t, tiles_r, tiles_c);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int bi = k * kThreads + threadIdx.x;
    const int64_t r = ti.r0 + (bi >> 3), c = ti.c0 + 16 * (bi & 7);
    if (r < p.R && c < p.C) {
      const int64_t e = (ti.s * p.R + r) * p.C + c;  // flat element index, e % 16 == 0
      v.codes[k] = __ldcs(reinterpret_cast<const uint2*>(p.codes + e / 2));
      v.scale[k] = __ldcs(p.scales + e / 16);
    }
  }
}

template <bool SR>
__device__ __forceinline__ uint4 sr_bits_or_zero(const RequantParams& p, uint64_t idx0) {
  if constexpr (SR) return sr_group_bits(p.seed, p.step, 2u, idx0);
  else return make_uint4(0, 0, 0, 0);
}

// MX block of 32 values of one column -> 32 E4M3 codes + the scale byte.
template <bool SR>
__device__ __forceinline__ void mx_block(const RequantParams& p, const float (&v)[32],
                                         uint64_t idx0, uint4 (&out)[2], uint32_t& sbyte) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int e = mx_shared_exp(amax);
  sbyte = (uint32_t)(e + 127);
  const float sc = exp2_neg(e);
  uint32_t w[8];
#pragma unroll
  for (int g = 0; g < 4; ++g) {  // groups of 8 elements: one Philox call each
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(v[8 * g + i], sc);
    if constexpr (!SR) {
      w[2 * g] = e4m3x4_rn(y[0], y[1], y[2], y[3]);
      w[2 * g + 1] = e4m3x4_rn(y[4], y[5], y[6], y[7]);
    } else {
      const uint4 rb = sr_group_bits(p.seed, p.step, 2u, idx0 + 8 * g);
      const uint32_t nw[4] = {~rb.x, ~rb.y, ~rb.z, ~rb.w};  // 0xFFFF - v in each half
      uint32_t c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        c[i] = e4m3_sr(y[i], (i & 1) ? (nw[i >> 1] >> 16) : (nw[i >> 1] & 0xFFFFu));
      w[2 * g] = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
      w[2 * g + 1] = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
    }
  }
  out[0] = make_uint4(w[0], w[1], w[2], w[3]);
  out[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// TARGET 0: MXFP8; TARGET 1: NVFP4 with block-scale format DFMT and 4/6 mode
// FOS (0 off, 1 MSE, 2 rule from the params).
template <int TARGET, int DFMT, bool SR, int FOS>
__global__ void __launch_bounds__(kThreads) requant_kernel(const RequantParams p, int64_t tiles_r,
                                                           int64_t tiles_c) {
  constexpr bool NV = TARGET == 1;
  __shared__ __align__(16) float4 s_x[TR * kSlots];
  __shared__ float s_src[256];
  __shared__ float s_d[NV ? 256 : 1], s_inv[NV ? 256 : 1];
  __shared__ uint32_t s_bits[TC];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t total = p.S * tiles_r * tiles_c;
  const int64_t R = p.R, C = p.C;
  float* xs = reinterpret_cast<float*>(s_x);

  SrcRegs v;
  load_src(p, blockIdx.x, total, tiles_r, tiles_c, v);
  int64_t cur_slice = -1;
  SliceScale ss_dst{};
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {  // block-uniform
    const TileIdx ti = tile_of(t, tiles_r, tiles_c);
    if (ti.s != cur_slice) {  // block-uniform; the previous tile ended with a barrier
      build_tables<DFMT, NV>(p, ti.s, s_src, s_d, s_inv, ss_dst);
      cur_slice = ti.s;
      __syncthreads();
    }
    // ---- 1: de-quantise this thread's two blocks into the tile ---------
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int bi = k * kThreads + tid;
      const int row = bi >> 3, cb = bi & 7;
      const float d = s_src[v.scale[k]];
      f2 q[4];
      float4* dst = s_x + row * kSlots;
      e2m1x8_to_f2(v.codes[k].x, q);
      const f2 dd = make_float2(d, d);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h == 1) e2m1x8_to_f2(v.codes[k].y, q);
        const f2 a = f2_mul(q[0], dd), b = f2_mul(q[1], dd), c = f2_mul(q[2], dd),
                 e = f2_mul(q[3], dd);
        // q * d overflows only when d > FLT_MAX / 6 (g near FLT_MAX): then
        // look at the products themselves
        if (d > 5.0e37f && !(fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y))),
                                  fmaxf(fmaxf(fabsf(c.x), fabsf(c.y)), fmaxf(fabsf(e.x), fabsf(e.y)))) <= kFltMax))
          flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
        dst[swz(4 * cb + 2 * h)] = make_float4(a.x, a.y, b.x, b.y);
        dst[swz(4 * cb + 2 * h + 1)] = make_float4(c.x, c.y, e.x, e.y);
      }
    }
    if (NV && FOS && tid < TC) s_bits[tid] = 0u;
    load_src(p, t + gridDim.x, total, tiles_r, tiles_c, v);  // next tile in flight
    __syncthreads();

    // ---- 2: encode one column band per warp -----------------------------
    const int c = 32 * (warp & 3) + lane;   // tile column
    const int rb = 32 * (warp >> 2);        // first tile row of the band
    const int64_t cg = ti.c0 + c, rg = ti.r0 + rb;
    const bool ok = cg < C && rg < R;       // R % 32 (MX) or R % 16 (NVFP4): whole blocks
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = xs[tile_word(rb + i, c)];
    const int64_t e0 = (ti.s * C + cg) * R + rg;  // flat output index of x[0]
    if constexpr (!NV) {
      uint4 out[2];
      uint32_t sbyte;
      mx_block<SR>(p, x, (uint64_t)e0, out, sbyte);
      if (ok) {
        uint4* o = reinterpret_cast<uint4*>(p.out_codes + e0);
        __stcs(o, out[0]);
        __stcs(o + 1, out[1]);
        p.out_scales[e0 / 32] = (uint8_t)sbyte;
      }
    } else {
      uint32_t pick = 0;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int64_t eb = e0 + 16 * b;
        if (b == 1 && !(rg + 16 < R)) break;  // ragged R: the band's second block is past the end
        f2 lo[4], hi[4];
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          lo[k] = make_float2(x[16 * b + 2 * k], x[16 * b + 2 * k + 1]);
          hi[k] = make_float2(x[16 * b + 8 + 2 * k], x[16 * b + 8 + 2 * k + 1]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[16 * b + i]));
        const uint4 rb0 = sr_bits_or_zero<SR>(p, (uint64_t)eb);
        const uint4 rb1 = sr_bits_or_zero<SR>(p, (uint64_t)eb + 8);
        const BlockResult r = encode_block_f<DFMT, SR, FOS != 0>(
            lo, hi, amax, ss_dst, TableScales{s_d, s_inv}, rb0, rb1, false,
            FOS == 2 ? p.rule : 0);
        if (ok) {
          __stcs(reinterpret_cast<uint2*>(p.out_codes + eb / 2), make_uint2(r.codes[0], r.codes[1]));
          p.out_scales[eb / 16] = (uint8_t)r.scale;
          if (FOS && r.pick4) pick |= 1u << b;
        }
      }
      if constexpr (FOS != 0) {
        if (pick) atomicOr(s_bits + c, pick << (rb / 16));
      }
    }
    __syncthreads();  // tile reads done (and the column bits complete)
    if constexpr (NV && FOS != 0) {
      if (tid < TC) {
        const uint32_t bits = s_bits[tid];
        const int64_t col = ti.c0 + tid;
        if (bits && col < C) {
          // blocks of this column inside the tile: (col * R + r0) / 16 + 0..3
          const int64_t b0 = (col * R + ti.r0) / 16;
          const int64_t W = (R * C / 16 + 31) / 32;
          uint32_t* words = p.out_choice + ti.s * W;
          const int off = (int)(b0 & 31);
          atomicOr(words + (b0 >> 5), bits << off);
          if (off + TR / 16 > 32 && (bits >> (32 - off))) atomicOr(words + (b0 >> 5) + 1, bits >> (32 - off));
        }
      }
    }
  }
}

template <int TARGET, int DFMT, bool SR, int FOS>
cudaError_t launch_t(const RequantParams& p, cudaStream_t st) {
  const int64_t tiles_r = (p.R + TR - 1) / TR, tiles_c = (p.C + TC - 1) / TC;
  const int64_t total = p.S * tiles_r * tiles_c;
  auto k = requant_kernel<TARGET, DFMT, SR, FOS>;
  const int64_t cap = (int64_t)sm_count() * resident_ctas(k, kThreads);
  const unsigned grid = (unsigned)(total < cap ? total : cap);
  k<<<grid, kThreads, 0, st>>>(p, tiles_r, tiles_c);
  return cudaGetLastError();
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
