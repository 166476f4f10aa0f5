// quant_dual.cu -- NVFP4 quantisation with 16x1 column blocks, alone or
// together with the 1x16 row blocks from a single read of the input
// (End-to-End 4-Bit Training, "Block-scaled backward passes": the transposed
// operand groups each value with the 15 values above/below it instead).
//
// A CTA (256 threads) takes a run of consecutive 64 x 128 tiles; for each:
//  1. the tile arrives by cp.async, while the previous one is encoded, into
//     one of two 16 KiB shared buffers of 32-bit words (two columns each),
//     every thread copying 4 chunks of 8 bf16 (a warp covers two full 256 B
//     tile rows); word w of row r is kept at w ^ (((r >> 4) & 3) << 3);
//  2. in BOTH mode the row blocks are read back as 128-bit chunks and
//     encoded with lanes 2m and 2m+1 holding the two halves of a block
//     (encode_half8);
//  3. lane (cp, q) = (lane >> 2, lane & 3) of warp w takes column pair
//     8 w + cp in the 16-row band q: it reads one word per row (with the
//     swizzle the 32 lanes hit 32 distinct banks) and encodes the two column
//     blocks it now holds, one lane per block (encode_block). The four bands
//     of a column are adjacent lanes, so each column's 64 rows of codes
//     (32 B), scales (4 B) and dequant (128 B, two instructions) leave from
//     one store instruction.
// The 4/6 bits of a tile are gathered in shared memory (one ballot per warp
// and half-block) and OR-ed into the pre-zeroed bitmaps during the next tile:
// a tile's bits share words with other tiles. Non-finite inputs are gathered
// per thread and flagged once.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int TR = 64;    // tile rows
constexpr int TC = 128;   // tile columns
constexpr int kWords = TC / 2;  // 32-bit words (column pairs) per tile row

__device__ __forceinline__ int word_of(int r, int w) {
  return r * kWords + (w ^ (((r >> 4) & 3) << 3));
}

// OR `nbits` bits into a bitmap at bit position bit0 (they may straddle two
// words).
__device__ __forceinline__ void or_bits(uint32_t* words, int64_t bit0, uint32_t bits, int nbits) {
  if (bits == 0) return;
  const int64_t w = bit0 >> 5;
  const int off = (int)(bit0 & 31);
  atomicOr(words + w, bits << off);
  if (off + nbits > 32) atomicOr(words + w + 1, bits >> (32 - off));
}

// The bits at even positions 0, 2, .., 2n-2 of b, packed into n bits.
__device__ __forceinline__ uint32_t even_bits(uint32_t b) {
  b &= 0x55555555u;
  b = (b | (b >> 1)) & 0x33333333u;
  b = (b | (b >> 2)) & 0x0F0F0F0Fu;
  b = (b | (b >> 4)) & 0x00FF00FFu;
  return (b | (b >> 8)) & 0x0000FFFFu;
}

// Block amax as bf16 bits from the magnitude maximum m of this lane's half
// (both halves of m) and of its partner's.
__device__ __forceinline__ uint32_t pair_amax(uint32_t m) {
  m = bmax_abs2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  return m;
}

// Launch geometry, computed once on the host. Tiles are numbered slice by
// slice, row of tiles by row of tiles, and CTA b takes the kTilesPerCta
// consecutive tiles from b * kTilesPerCta: while it encodes one the next one
// loads, and since CTAs start in order as earlier ones finish, the tiles in
// flight stay a compact run of neighbours whose rows share DRAM pages. (One
// CTA per SM slot looping over the whole tensor lets the CTAs drift apart,
// and the spread of the tiles in flight slows DRAM down as the tensor grows.)
constexpr uint32_t kTilesPerCta = 8;
struct DualGeom {
  FastDiv by_tiles_c, by_tiles_slice;
  uint32_t tiles_c, tiles_slice;
  uint32_t n_tiles;
  int64_t slice_elems;   // R * C
  int64_t words;         // 4/6 bitmap words per slice
};

template <int FMT, bool SR, int FOS, bool ROWS>
__global__ void __launch_bounds__(kThreads, SR ? (FOS != 0 ? 2 : 3) : (FOS == 2 ? 3 : 4))
    quant_dual_kernel(const DualParams p, const DualGeom geo) {
  pdl_begin();
  __shared__ __align__(16) uint32_t tile[2][TR * kWords];
  // block-scale tables of the current slice and the next one (the two swap
  // when a CTA's run crosses into a new slice) and their 1 / (6 g), 1 / (4 g)
  __shared__ float2 s_tab[2][256];
  __shared__ float s_rden[2][2];
  // 4/6 bits of the tile in each buffer: row ballots (one word per two tile
  // rows) and column ballots (one word per warp and column parity)
  __shared__ uint32_t s_rbits[2][TR / 2], s_cbits[2][16];

  const int64_t R = p.R, C = p.C, R16 = R >> 4, C16 = C >> 4;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int rule = FOS == 2 ? p.rule : 0;
  const bool vec = (C % 8) == 0;
  const int lr0 = t >> 4, lq = t & 15;  // thread t's chunks: rows 16 k + lr0, columns 8 lq ..
  const int cq = lane & 3, cpl = 8 * warp + (lane >> 2);  // column band q, column pair
  constexpr int kTab = FMT == 0 ? 128 : 256;

  // Offsets of this thread's outputs within any tile, fixed for the kernel:
  // row chunk k at (16 k + lr0) C / 8 + lq + 2 C k groups of 8 values from the
  // tile's first; column 2 cpl + j, band q at (2 cpl + j) R / 16 + q groups of
  // 16; the row / column 4/6 bits of tile row t / column t - 128 at
  // t C/16 / (t - 128) R/16 bits from the tile's first.
  const int64_t ro8 = (int64_t)lr0 * (C >> 3) + lq;
  const int64_t co16 = (int64_t)(2 * cpl) * R16 + cq;
  const int64_t rbit_t = (int64_t)t * C16, cbit_t = (int64_t)(t - 128) * R16;
  // thread t's first chunk from the tile origin, and the step of 16 rows
  const int64_t fo = (int64_t)lr0 * C + 8 * lq, C16x16 = 16 * C;

  // Where tile T lies: slice, origin, extent, and the element index of its
  // origin in the row layout (the input's, and the row encoding's) and in the
  // column layout.
  struct Where {
    int64_t s, r0, c0;
    int64_t ro, co;
    int nr, nc;
    bool first;  // the slice's first tile
  };
  auto finish = [&](Where& w) {
    w.nr = (int)(R - w.r0 < TR ? R - w.r0 : TR);
    w.nc = (int)(C - w.c0 < TC ? C - w.c0 : TC);
  };
  auto where = [&](uint32_t T) {
    Where w;
    const uint32_t s = fastdiv(T, geo.by_tiles_slice), u = T - s * geo.tiles_slice;
    const uint32_t tr = fastdiv(u, geo.by_tiles_c), tc = u - tr * geo.tiles_c;
    w.s = s;
    w.r0 = (int64_t)tr * TR;
    w.c0 = (int64_t)tc * TC;
    w.ro = w.s * geo.slice_elems + w.r0 * C + w.c0;
    w.co = w.s * geo.slice_elems + w.c0 * R + w.r0;
    w.first = u == 0;
    finish(w);
    return w;
  };
  // The tile after `w` in the numbering (the next one of this CTA's run):
  // along a row of tiles the origins move by fixed steps.
  auto advance = [&](const Where& w) {
    Where n = w;
    n.first = false;
    n.c0 = w.c0 + TC;
    n.ro = w.ro + TC;
    n.co = w.co + TC * R;
    if (n.c0 >= C) {
      n.c0 = 0;
      n.r0 = w.r0 + TR;
      if (n.r0 >= R) {
        n.r0 = 0;
        n.s = w.s + 1;
        n.first = true;
      }
      n.ro = n.s * geo.slice_elems + n.r0 * C;
      n.co = n.s * geo.slice_elems + n.r0;
    }
    finish(n);
    return n;
  };
  // Copy tile `at` into buffer `buf` (one 16-byte cp.async per chunk; chunks
  // past the tensor's edge are zero-filled).
  auto fetch = [&](const Where& at, int buf) {
    const uint16_t* xt = p.x + at.ro + fo;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int lr = 16 * k + lr0, lc = 8 * lq;
      const bool ok = lr < at.nr && lc < at.nc;
      uint32_t* dst = &tile[buf][word_of(lr, 4 * lq)];
      const uint16_t* src = xt + k * C16x16;
      if (vec) {
        cp_async16_zfill(dst, ok ? src : p.x, ok ? 16u : 0u);
      } else {  // column-only encoding of a tensor whose rows are not 16 B multiples
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = (ok && lc + i < at.nc) ? src[i] : 0u;
        *reinterpret_cast<uint4*>(dst) = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16),
                                                    h[4] | (h[5] << 16), h[6] | (h[7] << 16));
      }
    }
    cp_async_commit();
  };
  // The scale table and outer-scale reciprocals of a slice with global amax
  // gamax into buffer `buf` (threads 0..kTab-1; thread 0 also flags a bad
  // amax, once per slice).
  auto tables = [&](float gamax, bool first, int buf) {
    if (t < kTab) {
      const SliceScale ss = slice_scale(gamax, p.M);
      float d, inv;
      scale_entry<FMT>((uint32_t)t, ss.g, d, inv);
      s_tab[buf][t] = make_float2(d, inv);
      if (t == 0) {
        s_rden[buf][0] = ss.rden6;
        s_rden[buf][1] = ss.rden4;
        if (ss.bad && first) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
      }
    }
  };
  // A finished tile's 4/6 bits (left in s_[rc]bits[buf]) still to be OR-ed
  // into the bitmaps: tile row t's 8 blocks are bits rbit + t C/16 ..,
  // tile column cc's 4 bands bits cbit + cc R/16 ..
  struct Pending {
    uint32_t *rw, *cw;
    int64_t rbit, cbit;
    int nr, nc;
  };
  auto flush = [&](int buf, const Pending& f) {
    if (ROWS && t < f.nr) {  // threads 0..63
      const int nb = f.nc >> 4;
      const uint32_t bits = even_bits(s_rbits[buf][t >> 1] >> (16 * (t & 1)));
      or_bits(f.rw, f.rbit + rbit_t, bits & ((1u << nb) - 1u), nb);
    }
    if (t >= 128 && t - 128 < f.nc) {  // threads 128..255
      const int cc = t - 128, cp = cc >> 1, nb = f.nr >> 4;
      const uint32_t bits = s_cbits[buf][(cc & 1) * 8 + (cp >> 3)] >> (4 * (cp & 7));
      or_bits(f.cw, f.cbit + cbit_t, bits & ((1u << nb) - 1u), nb);
    }
  };

  const uint32_t T0 = blockIdx.x * kTilesPerCta;
  const uint32_t T1 = T0 + kTilesPerCta < geo.n_tiles ? T0 + kTilesPerCta : geo.n_tiles;
  Where cur = where(T0);
  Pending pend{};
  fetch(cur, 0);
  tables(t < kTab ? p.gamax[cur.s] : 0.0f, cur.first, 0);
  uint32_t seen = 0;  // magnitude maximum of every value this thread encodes
  int buf = 0, tb = 0;  // tile buffer, table buffer (flips with the slice)
  for (uint32_t T = T0; T < T1; ++T, buf ^= 1) {
    cp_async_wait<0>();  // this thread's copies of tile T have landed
    __syncthreads();     // everyone's have, and its tables are built; the
                         // previous tile is done with the other buffers
    const bool more = T + 1 < T1;
    const Where nx = more ? advance(cur) : cur;
    if (more) fetch(nx, buf ^ 1);  // in flight while this tile is encoded
    const bool new_slice = more && nx.s != cur.s;
    const float gam_next = new_slice && t < kTab ? p.gamax[nx.s] : 0.0f;
    if (FOS != 0 && T != T0) flush(buf ^ 1, pend);
    SliceScale ss;
    ss.rden6 = s_rden[tb][0];
    ss.rden4 = s_rden[tb][1];
    const float2* tab = s_tab[tb];
    const uint32_t* tl = tile[buf];
    const int nr = cur.nr, nc = cur.nc;

    // ---- row blocks: chunks from the staged tile ----------------------------
    if constexpr (ROWS) {
      const bool want_dq = p.r_dq != nullptr;
      const int64_t g8 = (cur.ro >> 3) + ro8;  // chunk 0, in groups of 8 values
      uint32_t* const rc = reinterpret_cast<uint32_t*>(p.r_codes) + g8;
      uint4* const rd = reinterpret_cast<uint4*>(p.r_dq) + g8;
      uint8_t* const rs = p.r_scales + (g8 >> 1);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int lr = 16 * k + lr0;
        const bool ok = lr < nr && 8 * lq < nc;
        const uint4 v = *reinterpret_cast<const uint4*>(&tl[word_of(lr, 4 * lq)]);
        const uint32_t m = pair_amax(bmax_abs2(bmax_abs2(v.x, v.y), bmax_abs2(v.z, v.w)));
        seen = bmax_abs2(seen, m);
        const uint32_t amax_bits = max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
        f2 x[4];
        unpack8(v, x);
        uint4 rb = make_uint4(0, 0, 0, 0);
        if constexpr (SR)
          rb = sr_group_bits(p.key, 0u, (uint64_t)(8 * (g8 + k * (2 * C))));
        const HalfOut h = encode_half8<FMT, SR, FOS>(x, amax_bits, ss, tab, rb, want_dq, rule);
        if (ok) rc[k * (2 * C)] = h.codes;
        if (ok && want_dq) __stcs(rd + k * (2 * C), h.dq);
        if (ok && (lane & 1) == 0) rs[k * C] = (uint8_t)h.scale;
        if constexpr (FOS != 0) {
          // lanes 0..15: tile row lr (even), lanes 16..31: row lr + 1
          const uint32_t bb = __ballot_sync(0xFFFFFFFFu, ok && h.pick4);
          if (lane == 0) s_rbits[buf][lr >> 1] = bb;
        }
      }
    }

    // ---- column blocks ----------------------------------------------------------
    {
      const bool want_dq = p.c_dq != nullptr;
      const bool rows_ok = 16 * cq < nr;
      const int64_t g16 = (cur.co >> 4) + co16;  // column 2 cpl, in groups of 16 values
      uint2* const ccodes = reinterpret_cast<uint2*>(p.c_codes) + g16;
      uint4* const cdq = reinterpret_cast<uint4*>(p.c_dq) + 2 * g16;
      uint8_t* const cscales = p.c_scales + g16;
      uint32_t w[16];
#pragma unroll
      for (int i2 = 0; i2 < 16; ++i2) w[i2] = tl[word_of(16 * cq + i2, cpl)];
      uint32_t m = 0;
#pragma unroll
      for (int i2 = 0; i2 < 16; ++i2) m = bmax_abs2(m, w[i2]);  // both columns' block amax
      seen = bmax_abs2(seen, m);
#pragma unroll
      for (int j = 0; j < 2; ++j) {  // column 2 cpl + j
        const bool okc = 2 * cpl + j < nc && rows_ok;
        f2 lo[4], hi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          lo[k] = j ? make_float2(bf16_hi(w[2 * k]), bf16_hi(w[2 * k + 1]))
                    : make_float2(bf16_lo(w[2 * k]), bf16_lo(w[2 * k + 1]));
          hi[k] = j ? make_float2(bf16_hi(w[8 + 2 * k]), bf16_hi(w[9 + 2 * k]))
                    : make_float2(bf16_lo(w[8 + 2 * k]), bf16_lo(w[9 + 2 * k]));
        }
        const uint32_t amax_bits = j ? (m >> 16) & 0x7FFFu : m & 0x7FFFu;
        uint4 rb0 = make_uint4(0, 0, 0, 0), rb1 = rb0;
        if constexpr (SR) {
          const uint64_t e = (uint64_t)(16 * (g16 + j * R16));
          rb0 = sr_group_bits(p.key, 1u, e);
          rb1 = sr_group_bits(p.key, 1u, e + 8);
        }
        const BlockResult br = encode_block<FMT, SR, FOS != 0>(
            lo, hi, amax_bits, ss, TableScales2{tab}, rb0, rb1, want_dq, rule);
        if (okc) ccodes[j * R16] = make_uint2(br.codes[0], br.codes[1]);
        if (okc) cscales[j * R16] = (uint8_t)br.scale;
        if (okc && want_dq) {
          __stcs(cdq + 2 * j * R16, br.dq[0]);
          __stcs(cdq + 2 * j * R16 + 1, br.dq[1]);
        }
        if constexpr (FOS != 0) {
          // bit 4 cp + q = band q of the warp's column pair cp, column j
          const uint32_t bb = __ballot_sync(0xFFFFFFFFu, okc && br.pick4);
          if (lane == 0) s_cbits[buf][j * 8 + warp] = bb;
        }
      }
    }
    if constexpr (FOS != 0) {
      pend.rw = p.r_choice + cur.s * geo.words;
      pend.cw = p.c_choice + cur.s * geo.words;
      pend.rbit = cur.r0 * C16 + (cur.c0 >> 4);
      pend.cbit = cur.c0 * R16 + (cur.r0 >> 4);
      pend.nr = nr;
      pend.nc = nc;
    }
    // the next slice's tables in the other table buffer, ready by the next
    // barrier (built after this tile's work, so reading its amax costs no
    // wait; that buffer's last readers finished before this tile's barrier)
    if (new_slice) {
      tables(gam_next, nx.first, tb ^ 1);
      tb ^= 1;
    }
    cur = nx;
  }
  if (FOS != 0) {  // the last tile's bits
    __syncthreads();
    flush(buf ^ 1, pend);
  }
  if (((seen & 0x7FFFu) >= 0x7F80u || ((seen >> 16) & 0x7FFFu) >= 0x7F80u))
    flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
}

template <int FMT, bool SR, int FOS, bool ROWS>
cudaError_t launch_t(const DualParams& p, int64_t S, cudaStream_t st) {
  const int64_t tiles_r = (p.R + TR - 1) / TR, tiles_c = (p.C + TC - 1) / TC;
  const int64_t per_slice = tiles_r * tiles_c, n = S * per_slice;
  if (n > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const int64_t grid = (n + kTilesPerCta - 1) / kTilesPerCta;
  DualGeom geo;
  geo.by_tiles_c = make_fastdiv((uint32_t)tiles_c);
  geo.by_tiles_slice = make_fastdiv((uint32_t)per_slice);
  geo.tiles_c = (uint32_t)tiles_c;
  geo.tiles_slice = (uint32_t)per_slice;
  geo.n_tiles = (uint32_t)n;
  geo.slice_elems = p.R * p.C;
  geo.words = (p.R * p.C / 16 + 31) / 32;
  return launch_pdl(quant_dual_kernel<FMT, SR, FOS, ROWS>, dim3((unsigned)grid), dim3(kThreads),
                    st, p, geo);
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
