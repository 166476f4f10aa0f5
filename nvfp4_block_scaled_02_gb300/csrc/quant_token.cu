// quant_token.cu -- NVFP4 quantisation with per-token (per-row) outer scales
// in a single pass over HBM (End-to-End 4-Bit Training, "Recipe details":
// per-token outer scales when quantising activations).
//
// Every row is its own slice: its outer scale g_r = amax_r / (6 M) comes from
// the row's own amax. Rows up to 16384 values: one CTA (256 threads) per row
// at a time; thread t holds blocks t, t+256, .. of the row in registers (K per
// thread), so the row is read from HBM once and never re-read.
// Wider rows: one warp per row streams the row twice (amax, then encode; the
// second read of the row hits L1/L2). d and 1/d are computed per block from
// g_r instead of a per-slice table. Outputs are those of the row encoding of
// the same tensor taken as `rows` slices of one row each (the 4/6 bitmap has
// ceil(C/512) words per row), plus the per-row amax.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowLoads = 16;  // 16-byte loads per lane in flight in the amax pass

template <int FMT, bool SR, int FOS>
__global__ void __launch_bounds__(kThreads) quant_token_kernel(const TokenParams p) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  const int64_t Bs = p.C / 16, W = (Bs + 31) / 32, nch = p.C / 8;
  const bool want_dq = p.dq != nullptr;
  for (int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); row < p.R;
       row += nwarps) {  // warp-uniform
    const uint4* xr = p.x + row * nch;
    // ---- pass 1: the row's amax ---------------------------------------
    // 16 loads in flight per lane: an 8 KiB row costs one memory round trip
    uint32_t m = 0;
    for (int64_t i = lane; i < nch; i += 32 * kRowLoads) {
      uint4 v[kRowLoads];
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int64_t j = i + 32 * u;
        v[u] = j < nch ? __ldg(xr + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) m = max(m, absmax_bits4(v[u]));
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const float amax_row = __uint_as_float(m << 16);
    const SliceScale ss = slice_scale(amax_row, p.M);
    if (lane == 0) {
      p.row_amax[row] = amax_row;
      if (m >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
      if (ss.bad) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
    }
    const DirectScales<FMT> scales{ss.g};
    // ---- pass 2: encode, 32 blocks per step ----------------------------
    for (int64_t t = 0; t < W; ++t) {
      const int64_t blk = t * 32 + lane;
      const bool ok = blk < Bs;
      const uint4 v0 = ok ? __ldg(xr + 2 * blk) : make_uint4(0, 0, 0, 0);
      const uint4 v1 = ok ? __ldg(xr + 2 * blk + 1) : make_uint4(0, 0, 0, 0);
      const int64_t gblk = row * Bs + blk;
      f2 lo[4], hi[4];
      unpack8(v0, lo);
      unpack8(v1, hi);
      const uint32_t mb = max(absmax_bits4(v0), absmax_bits4(v1));
      uint4 rb0 = make_uint4(0, 0, 0, 0), rb1 = rb0;
      if constexpr (SR) {
        rb0 = sr_group_bits(p.key, 0u, (uint64_t)gblk * 16);
        rb1 = sr_group_bits(p.key, 0u, (uint64_t)gblk * 16 + 8);
      }
      const BlockResult r =
          encode_block<FMT, SR, FOS != 0>(lo, hi, mb, ss, scales, rb0, rb1, want_dq,
                                          FOS == 2 ? p.rule : 0);
      if (ok) {
        __stcs(reinterpret_cast<uint2*>(p.codes) + gblk, make_uint2(r.codes[0], r.codes[1]));
        if (want_dq) {
          __stcs(p.dq + 2 * gblk, r.dq[0]);
          __stcs(p.dq + 2 * gblk + 1, r.dq[1]);
        }
        p.scales[gblk] = (uint8_t)r.scale;
      }
      if constexpr (FOS) {
        const uint32_t word = __ballot_sync(0xFFFFFFFFu, ok && r.pick4);
        if (lane == 0) p.choice[row * W + t] = word;
      }
    }
  }
}

// One CTA per row, K blocks of the row per thread, all held in registers.
// Per row: block amaxes -> warp redux -> barrier -> every thread takes the row
// amax; with RNE it computes the row's outer scale itself and each block's d
// and 1/d directly (one barrier per row: 40.6 -> 29.8 us for 2048 rows of
// 16384); with stochastic rounding every thread builds one entry of the row's
// scale table (d and 1/d of one scale code), warp 0 the two per-row
// reciprocals 1/(k g) -> barrier -> encode with table lookups, as the
// per-slice kernel does.
template <int FMT, bool SR, int FOS, int K>
__global__ void __launch_bounds__(kThreads) quant_token_cta_kernel(const TokenParams p) {
  pdl_begin();
  // RNE: d and 1/d per block from the row's g (no table, one barrier per
  // row); stochastic rounding keeps the per-row table, whose build costs less
  // than two per-block reciprocals in that heavier, issue-bound encoder.
  constexpr bool kDirect = !SR;
  __shared__ uint32_t s_max[2][kWarps];  // by row parity: the next row's partials go to the other
  __shared__ float s_d[kDirect ? 1 : 256], s_inv[kDirect ? 1 : 256];
  __shared__ SliceScale s_ss;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t Bs = p.C / 16, W = (Bs + 31) / 32;
  const bool want_dq = p.dq != nullptr;
  // the thread's blocks of `row` (zeros past the row's end or the last row)
  auto load_row = [&](int64_t row, uint4 (&v)[K][2]) {
    const uint4* xr = p.x + row * (p.C / 8);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int64_t blk = (int64_t)k * kThreads + tid;
      const bool ok = row < p.R && blk < Bs;
      v[k][0] = ok ? __ldcs(xr + 2 * blk) : make_uint4(0, 0, 0, 0);
      v[k][1] = ok ? __ldcs(xr + 2 * blk + 1) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 v[K][2];
  load_row(blockIdx.x, v);
  int par = 0;
  for (int64_t row = blockIdx.x; row < p.R; row += gridDim.x, par ^= 1) {  // block-uniform
    uint4 vn[K][2];
    load_row(row + gridDim.x, vn);  // next row in flight while this one is encoded
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) m = max(m, max(absmax_bits4(v[k][0]), absmax_bits4(v[k][1])));
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) s_max[par][warp] = m;
    __syncthreads();  // A: partial maxima in; the previous row's table reads are done
    uint32_t mr = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mr = max(mr, s_max[par][w]);
    const float amax_row = __uint_as_float(mr << 16);
    SliceScale ss;
    if constexpr (kDirect) {
      ss = slice_scale(amax_row, p.M);
      if (tid == 0) {
        p.row_amax[row] = amax_row;
        if (mr >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
        if (ss.bad) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
      }
    } else {
      // g exactly as slice_scale computes it; then this thread's table entry
      const bool bad = !(amax_row >= 0.0f) || amax_row > kFltMax;
      float g = 1.0f;
      if (!bad && amax_row > 0.0f) g = __fdiv_rn(amax_row, __fmul_rn(6.0f, p.M));
      float d, inv;
      scale_entry<FMT>((uint32_t)tid, g, d, inv);
      s_d[tid] = d;
      s_inv[tid] = inv;
      if (warp == 0) {
        const SliceScale sw = slice_scale(amax_row, p.M);
        if (lane == 0) {
          s_ss = sw;
          p.row_amax[row] = amax_row;
          if (mr >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
          if (sw.bad) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
        }
      }
      __syncthreads();  // B: table and per-row reciprocals ready
      ss = s_ss;
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int64_t blk = (int64_t)k * kThreads + tid;
      const bool ok = blk < Bs;
      const int64_t gblk = row * Bs + blk;
      f2 lo[4], hi[4];
      unpack8(v[k][0], lo);
      unpack8(v[k][1], hi);
      const uint32_t mb = max(absmax_bits4(v[k][0]), absmax_bits4(v[k][1]));
      uint4 rb0 = make_uint4(0, 0, 0, 0), rb1 = rb0;
      if constexpr (SR) {
        rb0 = sr_group_bits(p.key, 0u, (uint64_t)gblk * 16);
        rb1 = sr_group_bits(p.key, 0u, (uint64_t)gblk * 16 + 8);
      }
      BlockResult r;
      if constexpr (kDirect)
        r = encode_block<FMT, SR, FOS != 0>(lo, hi, mb, ss, DirectScales<FMT>{ss.g}, rb0, rb1,
                                            want_dq, FOS == 2 ? p.rule : 0);
      else
        r = encode_block<FMT, SR, FOS != 0>(lo, hi, mb, ss, TableScales{s_d, s_inv}, rb0, rb1,
                                            want_dq, FOS == 2 ? p.rule : 0);
      if (ok) {
        __stcs(reinterpret_cast<uint2*>(p.codes) + gblk, make_uint2(r.codes[0], r.codes[1]));
        if (want_dq) {
          __stcs(p.dq + 2 * gblk, r.dq[0]);
          __stcs(p.dq + 2 * gblk + 1, r.dq[1]);
        }
        p.scales[gblk] = (uint8_t)r.scale;
      }
      if constexpr (FOS) {
        // the warp's 32 blocks are blocks 256k + 32 warp .. + 31: one bitmap word
        const uint32_t word = __ballot_sync(0xFFFFFFFFu, ok && r.pick4);
        const int64_t wi = (int64_t)k * kWarps + warp;
        if (lane == 0 && wi < W) p.choice[row * W + wi] = word;
      }
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      v[k][0] = vn[k][0];
      v[k][1] = vn[k][1];
    }
  }
}

template <int FMT, bool SR, int FOS>
cudaError_t launch_t(const TokenParams& p, cudaStream_t st) {
  const int64_t Bs = p.C / 16;
  auto run_cta = [&](auto kernel) {
    static const int per_sm = resident_ctas(kernel, kThreads);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(p.R, (int64_t)sm_count() * per_sm));
    return launch_pdl(kernel, dim3((unsigned)grid), dim3(kThreads), st, p);
  };
  if (Bs <= kThreads) return run_cta(quant_token_cta_kernel<FMT, SR, FOS, 1>);
  if (Bs <= 2 * kThreads) return run_cta(quant_token_cta_kernel<FMT, SR, FOS, 2>);
  if (Bs <= 4 * kThreads) return run_cta(quant_token_cta_kernel<FMT, SR, FOS, 4>);
  const int64_t want = (p.R + kWarps - 1) / kWarps;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * 8));
  return launch_pdl(quant_token_kernel<FMT, SR, FOS>, dim3((unsigned)grid), dim3(kThreads), st, p);
}

}  // namespace

cudaError_t launch_quant_token(const TokenParams& p, int fmt, bool sr, int fos, cudaStream_t st) {
#define NVFP4_TOK(F, R, O) \
  if (fmt == F && sr == R && fos == O) return launch_t<F, R, O>(p, st);
  NVFP4_TOK(0, false, 0) NVFP4_TOK(0, false, 1) NVFP4_TOK(0, false, 2) NVFP4_TOK(0, true, 0)
  NVFP4_TOK(0, true, 1) NVFP4_TOK(0, true, 2) NVFP4_TOK(1, false, 0) NVFP4_TOK(1, false, 1)
  NVFP4_TOK(1, false, 2) NVFP4_TOK(1, true, 0) NVFP4_TOK(1, true, 1) NVFP4_TOK(1, true, 2)
#undef NVFP4_TOK
  return cudaErrorInvalidValue;
}

}  // namespace nvfp4
