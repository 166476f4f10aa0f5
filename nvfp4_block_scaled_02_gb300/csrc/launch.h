// launch.h -- internal host-side interface between the C ABI (api.cu) and the
// kernel translation units. Not installed; the public interface is nvfp4.h.
#pragma once
#include <cstdint>
#include <algorithm>
#include <cuda_runtime.h>

#include "../../include/nvfp4.h"
#include "device.cuh"

#define NVFP4_DEV_NONFINITE_INPUT_BIT NVFP4_DEV_NONFINITE_INPUT
#define NVFP4_DEV_BAD_SCALE_BIT NVFP4_DEV_BAD_SCALE
#define NVFP4_DEV_BAD_AMAX_BIT NVFP4_DEV_BAD_AMAX

namespace nvfp4 {

int sm_count();

// Host side of FastDiv (device.cuh): the constants for divisor d >= 1.
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  FastDiv f;
  f.m = (uint32_t)(((1ull << 32) * ((1ull << l) - d)) / d + 1);
  f.s1 = l < 1 ? l : 1;
  f.s2 = l > 0 ? l - 1 : 0;
  return f;
}

// Where the tile of a one-tile-per-CTA kernel lies: tiles numbered slice by
// slice, row of tiles by row of tiles, column tiles fastest. The divisions by
// the tile counts are FastDiv multiplies (the grid holds < 2^31 tiles), and
// the slice size is precomputed, so no CTA runs a 64-bit division.
struct TileGeom {
  FastDiv by_tiles_c, by_tiles_slice;
  uint32_t tiles_c, tiles_slice;
  int64_t slice_elems;  // R * C
};
inline TileGeom make_tile_geom(int64_t R, int64_t C, int64_t TR, int64_t TC) {
  TileGeom g;
  const int64_t tc = (C + TC - 1) / TC, tr = (R + TR - 1) / TR;
  g.tiles_c = (uint32_t)tc;
  g.tiles_slice = (uint32_t)(tc * tr);
  g.by_tiles_c = make_fastdiv(g.tiles_c);
  g.by_tiles_slice = make_fastdiv(g.tiles_slice);
  g.slice_elems = R * C;
  return g;
}
// Slice, tile row and tile column of tile t.
__device__ __forceinline__ void tile_of(uint32_t t, const TileGeom& g, uint32_t& s, uint32_t& tr,
                                        uint32_t& tc) {
  s = fastdiv(t, g.by_tiles_slice);
  const uint32_t u = t - s * g.tiles_slice;
  tr = fastdiv(u, g.by_tiles_c);
  tc = u - tr * g.tiles_c;
}

// CTAs of `kernel` (with `threads` threads and `smem` dynamic shared memory)
// that fit on one SM at once, at least 1: sizes persistent grids to a single
// wave.
template <class Kernel>
int resident_ctas(Kernel kernel, int threads, size_t smem = 0) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
      n < 1)
    n = 1;
  return n;
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream drains (it calls pdl_begin() before any
// memory access, which waits for that kernel to complete).
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = 0;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, static_cast<Args&&>(args)...);
}

// Row (1x16) quantiser over a stack of S slices of Bs blocks each.
struct RowParams {
  const uint4* x;       // bf16 input, 8 values per uint4
  int64_t Bs;           // blocks per slice = R * C / 16
  int64_t W;            // 4/6 bitmap words per slice = ceil(Bs / 32)
  const float* gamax;   // [S]
  float M;              // outer-scale FP8 maximum
  SrKey key;            // stochastic rounding: Philox round keys of (seed, step)
  uint32_t* codes;      // 8 codes (one uint32) per chunk of 8 values
  uint8_t* scales;      // one byte per block
  uint32_t* choice;     // 4/6 bitmap (may be null when 4/6 is off)
  uint4* dq;            // bf16 dequant, may be null
  int32_t* status;      // may be null
  int64_t slice0;       // first slice of this launch (grids cover <= 65535)
  int rule;             // 4/6 selection metric: 0 MSE, 1 MAE, 2 max error
};
// fos: 0 = 4/6 off, 1 = on with the MSE rule, 2 = on with the rule in the params
cudaError_t launch_quant_row(const RowParams& p, int64_t S, int fmt, bool sr, int fos,
                             cudaStream_t st);

// Column (16x1) and dual (row + column from one read) quantiser.
struct DualParams {
  const uint16_t* x;    // bf16 [S][R][C]
  int64_t S, R, C;
  const float* gamax;
  float M;
  SrKey key;            // Philox round keys of (seed, step)
  // row encoding (used when the kernel writes both)
  uint8_t* r_codes;
  uint8_t* r_scales;
  uint32_t* r_choice;
  uint16_t* r_dq;
  // column encoding
  uint8_t* c_codes;
  uint8_t* c_scales;
  uint32_t* c_choice;
  uint16_t* c_dq;
  int32_t* status;
  int rule;             // 4/6 selection metric
};
cudaError_t launch_quant_dual(const DualParams& p, int64_t S, bool rows_too, int fmt, bool sr,
                              int fos, cudaStream_t st);

// One block scale per 16x16 tile; row encoding and (optionally) its transpose.
struct Tile16Params {
  const uint4* x;       // bf16 [S][R][C], R % 16 == 0, C % 16 == 0
  int64_t S, R, C;
  const float* gamax;   // [S]
  float M;
  uint32_t seed, step;  // stochastic rounding key (round keys derived in the kernel)
  uint32_t* r_codes;    // 8 codes per word, row layout
  uint8_t* r_scales;
  uint4* r_dq;          // may be null
  uint32_t* c_codes;    // column encoding (the transpose), null = not written
  uint8_t* c_scales;
  uint4* c_dq;          // may be null
  int32_t* status;
};
cudaError_t launch_quant_tile16(const Tile16Params& p, int fmt, bool sr, cudaStream_t st);

// Per-token (per-row outer scale) quantiser, amax and encoding in one pass.
struct TokenParams {
  const uint4* x;       // bf16 [R][C], C % 16 == 0
  int64_t R, C;
  float M;
  SrKey key;            // Philox round keys of (seed, step)
  float* row_amax;      // [R], written
  uint32_t* codes;      // as RowParams
  uint8_t* scales;
  uint32_t* choice;     // [R][ceil(C/512)] words (may be null when 4/6 is off)
  uint4* dq;            // may be null
  int32_t* status;
  int rule;             // 4/6 selection metric
};
cudaError_t launch_quant_token(const TokenParams& p, int fmt, bool sr, int fos, cudaStream_t st);

// De-quantise -> transpose -> re-quantise of a row encoding of [S][R][C].
struct RequantParams {
  const uint8_t* codes;   // source codes [S][R][C/2]
  const uint8_t* scales;  // source scale bytes [S][R][C/16]
  int64_t S, R, C;
  const float* gamax;     // [S], the forward encoding's global amax
  int src_fmt;            // source block-scale format
  float M_src, M_dst;     // outer-scale FP8 maxima of the source and target
  SrKey key;            // Philox round keys of (seed, step)
  uint8_t* out_codes;     // MX: [S][C][R] E4M3; NVFP4: [S][C][R/2]
  uint8_t* out_scales;    // MX: [S][C][R/32] E8M0; NVFP4: [S][C][R/16]
  uint32_t* out_choice;   // NVFP4 with 4/6: pre-zeroed bitmap
  int32_t* status;
  int rule;               // 4/6 selection metric
};
// target 0 = MXFP8, 1 = NVFP4 (dst_fmt, fos as launch_quant_row)
cudaError_t launch_requant(const RequantParams& p, int target, int dst_fmt, bool sr, int fos,
                           cudaStream_t st);

// Zero n 32-bit words on the stream (overlaps the previous kernel's tail).
cudaError_t launch_zero_words(uint32_t* p, int64_t n, cudaStream_t st);

// Per-slice global amax.
cudaError_t launch_amax(const uint16_t* x, int64_t S, int64_t n, float* amax, int32_t* status,
                        cudaStream_t st);
// The same in one launch with a workspace of 2 words per slice (zero before,
// zero after).
cudaError_t launch_amax_ticket(const uint16_t* x, int64_t S, int64_t n, float* amax,
                               uint32_t* ws, int32_t* status, cudaStream_t st);
// The same with the library's own fixed scratch array (at most
// kAmaxNoAllocMaxSlices slices): no memory of the caller's beyond x and amax.
constexpr int64_t kAmaxNoAllocMaxSlices = NVFP4_AMAX_NOALLOC_MAX_SLICES;
cudaError_t launch_amax_noalloc(const uint16_t* x, int64_t S, int64_t n, float* amax,
                                int32_t* status, cudaStream_t st);

// Scale-learning fake quantisation and STE backward (row blocks).
struct SteParams {
  const uint4* x;
  const uint4* gq;      // backward only
  int64_t nblocks;      // R * C / 16
  const float* s_pre;
  const float* s_post;  // null = tied
  uint4* out;           // xq (forward) or gx (backward, may be null)
  float* gs_pre;
  float* gs_post;
  int32_t* status;
  const float* gamax;   // [1]: FP8-rounded scales in units of gamax / (6 * 448); null = fp32 scales
  uint8_t* codes;       // export: NVFP4 codes [R][C/2]
  uint8_t* scales;      // export: E4M3 scale bytes [R][C/16]
};
cudaError_t launch_fakequant_fwd(const SteParams& p, cudaStream_t st);
cudaError_t launch_scale_grad_bwd(const SteParams& p, cudaStream_t st);
cudaError_t launch_export_scales(const SteParams& p, cudaStream_t st);

// MSE scale setting over every E4M3 scale of each 1x16 block.
struct ScaleInitParams {
  const uint4* x;       // bf16 [R][C], C % 16 == 0
  int64_t nblocks;
  const float* gamax;   // [1]
  uint8_t* codes;       // [nblocks] or null
  float* s;             // [nblocks] or null
  int32_t* status;
};
cudaError_t launch_scale_init_mse(const ScaleInitParams& p, cudaStream_t st);

// Diagnostics.
cudaError_t launch_codec_probe(int op, const float* in, const uint32_t* aux, int64_t n,
                               uint8_t* out, cudaStream_t st);
cudaError_t launch_sr_bits(uint32_t seed, uint32_t step, uint32_t dir, uint64_t idx0, int64_t n,
                           uint32_t* out, cudaStream_t st);

}  // namespace nvfp4
