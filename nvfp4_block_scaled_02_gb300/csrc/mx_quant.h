// mx_quant.h -- launcher of the MXFP8 quantiser of bf16 tensors (mx_quant.cu).
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

namespace nvfp4 {

struct MxParams {
  const uint16_t* x;      // bf16 [S][R][C]
  int64_t S, R, C;
  uint32_t seed, step;    // stochastic rounding key (round keys derived in the kernel)
  uint8_t* r_codes;       // E4M3 [S][R][C]
  uint8_t* r_scales;      // E8M0 [S][R][C/32]
  uint8_t* c_codes;       // E4M3 [S][C][R]
  uint8_t* c_scales;      // E8M0 [S][C][R/32]
  int32_t* status;
};

// Rows (C % 32 == 0) and/or columns (R % 32 == 0), RNE or stochastic.
cudaError_t launch_mx_quant(const MxParams& p, bool rows, bool cols, bool sr, cudaStream_t st);

}  // namespace nvfp4
