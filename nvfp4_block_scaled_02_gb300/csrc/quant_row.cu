// quant_row.cu -- NVFP4 quantisation with 1x16 row blocks.
//
// Row blocks are 16 consecutive elements of a row, and rows are contiguous
// with C % 16 == 0, so a slice is a flat run of R*C/16 blocks. A warp owns a
// "tile" of 32 consecutive blocks (1 KiB of bf16): lane l loads chunk l and
// chunk l + 32 of the tile with 128-bit loads (8 values each), so the two
// lanes of a pair (l, l^1) hold the two halves of one block. Per tile the warp
// writes 256 B of codes, 32 scale bytes, one 32-bit 4/6 word (a ballot) and
// 1 KiB of dequantised bf16 -- all coalesced. U tiles are loaded before any is
// processed to keep enough bytes in flight per SM.
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Gather the even bits of a ballot (lanes 0, 2, .., 30) into 16 bits.
__device__ __forceinline__ uint32_t even_bits(uint32_t b) {
  b &= 0x55555555u;
  b = (b | (b >> 1)) & 0x33333333u;
  b = (b | (b >> 2)) & 0x0F0F0F0Fu;
  b = (b | (b >> 4)) & 0x00FF00FFu;
  b = (b | (b >> 8)) & 0x0000FFFFu;
  return b;
}

template <int FMT, bool SR, bool FOS, int U>
__global__ void __launch_bounds__(kThreads) quant_row_kernel(const RowParams p) {
  __shared__ float s_d[256], s_inv[256];
  const int64_t s = p.slice0 + blockIdx.y;
  const SliceScale ss = slice_scale(p.gamax[s], p.M);
  if (ss.bad && threadIdx.x == 0 && blockIdx.x == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
  build_scale_table<FMT>(s_d, s_inv, ss.g);
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (p.Bs + 31) / 32;
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  const int64_t blk_base = s * p.Bs;  // first block of the slice
  const bool want_dq = p.dq != nullptr;

  for (int64_t t0 = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t0 < ntiles;
       t0 += nwarps * U) {
    uint4 v[U][2];
    bool ok[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tile = t0 + (int64_t)u * nwarps;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t blk = tile * 32 + h * 16 + (lane >> 1);  // block within slice
        ok[u][h] = tile < ntiles && blk < p.Bs;
        v[u][h] = ok[u][h] ? __ldcs(p.x + (blk_base + blk) * 2 + (lane & 1))
                           : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tile = t0 + (int64_t)u * nwarps;
      if (tile >= ntiles) break;  // warp-uniform
      uint32_t word = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t blk = tile * 32 + h * 16 + (lane >> 1);
        const int64_t gblk = blk_base + blk;
        f2 x[4];
        unpack8(v[u][h], x);
        uint32_t m = absmax_bits4(v[u][h]);
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        if (ok[u][h] && m >= 0x7F80u) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
        uint4 rb = make_uint4(0, 0, 0, 0);
        if constexpr (SR)
          rb = sr_group_bits(p.seed, p.step, 0u, (uint64_t)(gblk * 16 + (lane & 1) * 8));
        const HalfResult r = encode_half<FMT, SR, FOS>(x, m, ss, s_d, s_inv, rb, want_dq);
        if (ok[u][h]) {
          const int64_t chunk = gblk * 2 + (lane & 1);
          __stcs(p.codes + chunk, r.codes);
          if (want_dq) __stcs(p.dq + chunk, r.dq);
          if ((lane & 1) == 0) p.scales[gblk] = (uint8_t)r.scale;
        }
        if constexpr (FOS) word |= even_bits(__ballot_sync(0xFFFFFFFFu, ok[u][h] && r.pick4)) << (16 * h);
      }
      if constexpr (FOS)
        if (lane == 0) p.choice[s * p.W + tile] = word;
    }
  }
}

template <int FMT, bool SR, bool FOS>
cudaError_t launch_t(const RowParams& p, int64_t S, cudaStream_t st) {
  constexpr int U = FOS ? 1 : 2;
  const int64_t ntiles = (p.Bs + 31) / 32;
  const int64_t want = (ntiles + kWarps * U - 1) / (kWarps * U);
  const int64_t cap = std::max<int64_t>(1, (int64_t)sm_count() * 8 / std::max<int64_t>(1, S));
  RowParams q = p;
  for (int64_t s0 = 0; s0 < S; s0 += 65535) {
    q.slice0 = s0;
    dim3 grid((unsigned)std::min(want, cap), (unsigned)std::min<int64_t>(S - s0, 65535));
    quant_row_kernel<FMT, SR, FOS, U><<<grid, kThreads, 0, st>>>(q);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_quant_row(const RowParams& p, int64_t S, int fmt, bool sr, bool fos,
                             cudaStream_t st) {
#define NVFP4_ROW(F, R, O) \
  if (fmt == F && sr == R && fos == O) return launch_t<F, R, O>(p, S, st);
  NVFP4_ROW(0, false, false) NVFP4_ROW(0, false, true) NVFP4_ROW(0, true, false)
  NVFP4_ROW(0, true, true) NVFP4_ROW(1, false, false) NVFP4_ROW(1, false, true)
  NVFP4_ROW(1, true, false) NVFP4_ROW(1, true, true)
#undef NVFP4_ROW
  return cudaErrorInvalidValue;
}

}  // namespace nvfp4
