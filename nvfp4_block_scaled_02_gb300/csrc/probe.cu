// probe.cu -- element-by-element access to the device codecs and to the
// stochastic-rounding bit stream, for exhaustive checks of what the kernels
// compute. Not on the quantisation path.
#include "device.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

__global__ void codec_probe_kernel(int op, const float* __restrict__ in,
                                   const uint32_t* __restrict__ aux, int64_t n,
                                   uint8_t* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    if (op == 0) {
      // pairs share one conversion, exactly as in the kernels
      const int64_t e = i & ~(int64_t)1;
      const float a = in[e], b = (e + 1 < n) ? in[e + 1] : 0.0f;
      const uint32_t byte = e2m1x2_rn(a, b);
      out[i] = (uint8_t)((i & 1) ? (byte >> 4) : (byte & 15u));
    } else if (op == 1) {
      out[i] = (uint8_t)e4m3_encode(in[i]);
    } else if (op == 2) {
      out[i] = (uint8_t)ue5m3_encode(in[i]);
    } else {
      out[i] = (uint8_t)e2m1_sr(in[i], aux[i] & 0xFFFFu);
    }
  }
}

__global__ void sr_bits_kernel(uint32_t seed, uint32_t step, uint32_t dir, uint64_t idx0, int64_t n,
                               uint32_t* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t idx = idx0 + (uint64_t)i;
    const uint4 w = sr_group_bits(seed, step, dir, idx & ~(uint64_t)7);
    out[i] = sr_bits_of(w, (int)(idx & 7));
  }
}

unsigned grid_for(int64_t n) {
  return (unsigned)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 16));
}

}  // namespace

cudaError_t launch_codec_probe(int op, const float* in, const uint32_t* aux, int64_t n,
                               uint8_t* out, cudaStream_t st) {
  codec_probe_kernel<<<grid_for(n), 256, 0, st>>>(op, in, aux, n, out);
  return cudaGetLastError();
}

cudaError_t launch_sr_bits(uint32_t seed, uint32_t step, uint32_t dir, uint64_t idx0, int64_t n,
                           uint32_t* out, cudaStream_t st) {
  sr_bits_kernel<<<grid_for(n), 256, 0, st>>>(seed, step, dir, idx0, n, out);
  return cudaGetLastError();
}

}  // namespace nvfp4
