// quant_row.cu -- NVFP4 quantisation with 1x16 row blocks.
//
// Row blocks are 16 consecutive elements of a row, and rows are contiguous
// with C % 16 == 0, so a slice is a flat run of R*C/16 blocks. A warp owns a
// "tile" of 32 consecutive blocks (1 KiB of bf16) and lane l owns block l of
// it, so every per-block step (amax, both scale candidates, the 4/6 sums and
// choice) runs once per block with no shuffles. The tile arrives through a
// cp.async pipeline kStages tiles deep: the warp copies it with two fully
// coalesced 512 B sweeps into shared memory and each lane then reads its own
// 32 B block. Per tile the warp writes 256 B of codes, 32 scale bytes, one
// 32-bit 4/6 word (a ballot) and 1 KiB of dequantised bf16.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 4;  // tiles in flight per warp (cp.async groups)

template <int FMT, bool SR, int FOS>
__global__ void __launch_bounds__(kThreads) quant_row_kernel(const RowParams p) {
  pdl_begin();
  // stage[slot][w][c]: chunk c (0..63) of warp w's tile; chunk c holds values
  // 8c .. 8c+7 of the tile, i.e. half c%2 of block c/2.
  __shared__ __align__(16) uint4 stage[kStages][kWarps][64];
  __shared__ float2 s_tab[256];
  const int64_t s = p.slice0 + blockIdx.y;
  const SliceScale ss = slice_scale(p.gamax[s], p.M);
  if (ss.bad && threadIdx.x == 0 && blockIdx.x == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
  build_scale_table2<FMT>(s_tab, ss.g);
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t ntiles = (p.Bs + 31) / 32;
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  const int64_t blk_base = s * p.Bs;  // first block of the slice
  const bool want_dq = p.dq != nullptr;
  const int64_t t0 = (int64_t)blockIdx.x * kWarps + warp;

  // The warp's two coalesced 512 B copies of `tile` into stage slot `slot`.
  auto issue = [&](int64_t tile, int slot) {
    if (tile < ntiles) {
      const int64_t first = tile * 32;  // first block of the tile
      const int64_t nchunks = 2 * (p.Bs - first);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = h * 32 + lane;
        if (c < nchunks) cp_async16(&stage[slot][warp][c], p.x + (blk_base + first) * 2 + c);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int k = 0; k < kStages - 1; ++k) issue(t0 + k * nwarps, k);

  int slot = 0;
  for (int64_t tile = t0; tile < ntiles; tile += nwarps) {
    issue(tile + (kStages - 1) * nwarps, (slot + kStages - 1) % kStages);
    cp_async_wait<kStages - 1>();  // this lane's copies of the tile have landed
    __syncwarp();                  // ... and every other lane's
    const int64_t blk = tile * 32 + lane;
    const bool ok = blk < p.Bs;
    const uint4 v0 = ok ? stage[slot][warp][2 * lane] : make_uint4(0, 0, 0, 0);
    const uint4 v1 = ok ? stage[slot][warp][2 * lane + 1] : make_uint4(0, 0, 0, 0);
    __syncwarp();  // all reads of this slot done before any lane refills it
    const int64_t gblk = blk_base + blk;
    f2 lo[4], hi[4];
    unpack8(v0, lo);
    unpack8(v1, hi);
    const uint32_t m = max(absmax_bits4(v0), absmax_bits4(v1));
    if (ok && m >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
    uint4 rb0 = make_uint4(0, 0, 0, 0), rb1 = rb0;
    if constexpr (SR) {
      rb0 = sr_group_bits(p.key, 0u, (uint64_t)gblk * 16);
      rb1 = sr_group_bits(p.key, 0u, (uint64_t)gblk * 16 + 8);
    }
    const BlockResult r =
        encode_block<FMT, SR, FOS != 0>(lo, hi, m, ss, TableScales2{s_tab}, rb0, rb1, want_dq,
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
      if (lane == 0) p.choice[s * p.W + tile] = word;
    }
    slot = (slot + 1) % kStages;
  }
  cp_async_wait<0>();
}

template <int FMT, bool SR, int FOS>
cudaError_t launch_t(const RowParams& p, int64_t S, cudaStream_t st) {
  const int64_t ntiles = (p.Bs + 31) / 32;
  const int64_t want = (ntiles + kWarps - 1) / kWarps;
  static const int per_sm = resident_ctas(quant_row_kernel<FMT, SR, FOS>, kThreads);
  const int64_t cap =
      std::max<int64_t>(1, (int64_t)sm_count() * per_sm / std::max<int64_t>(1, S));
  RowParams q = p;
  for (int64_t s0 = 0; s0 < S; s0 += 65535) {
    q.slice0 = s0;
    dim3 grid((unsigned)std::min(want, cap), (unsigned)std::min<int64_t>(S - s0, 65535));
    cudaError_t e = launch_pdl(quant_row_kernel<FMT, SR, FOS>, grid, dim3(kThreads), st, q);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_quant_row(const RowParams& p, int64_t S, int fmt, bool sr, int fos,
                             cudaStream_t st) {
#define NVFP4_ROW(F, R, O) \
  if (fmt == F && sr == R && fos == O) return launch_t<F, R, O>(p, S, st);
  NVFP4_ROW(0, false, 0) NVFP4_ROW(0, false, 1) NVFP4_ROW(0, false, 2) NVFP4_ROW(0, true, 0)
  NVFP4_ROW(0, true, 1) NVFP4_ROW(0, true, 2) NVFP4_ROW(1, false, 0) NVFP4_ROW(1, false, 1)
  NVFP4_ROW(1, false, 2) NVFP4_ROW(1, true, 0) NVFP4_ROW(1, true, 1) NVFP4_ROW(1, true, 2)
#undef NVFP4_ROW
  return cudaErrorInvalidValue;
}

}  // namespace nvfp4
