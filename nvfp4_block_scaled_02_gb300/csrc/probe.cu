// probe.cu -- element-by-element access to the device codecs and to the
// stochastic-rounding bit stream, for exhaustive checks of what the kernels
// compute. Not on the quantisation path.
#include "device.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

// Ops 0 and 3 run the kernels' own 8-value helpers (e2m1x8_rn, sr8) on
// groups of 8 consecutive inputs; ops 1 and 2 the block-scale encoders; ops
// 4..7 the MXFP8 element encoders and shared exponent of re-quantisation.
__global__ void codec_probe_kernel(int op, const float* __restrict__ in,
                                   const uint32_t* __restrict__ aux, int64_t n,
                                   uint8_t* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (op == 1 || op == 2) {
    for (int64_t i = t0; i < n; i += stride)
      out[i] = (uint8_t)(op == 1 ? e4m3_encode(in[i]) : ue5m3_encode(in[i]));
    return;
  }
  if (op >= 4) {  // MXFP8 element encoders and the shared exponent
    for (int64_t i = t0; i < n; i += stride) {
      uint32_t c;
      if (op == 4) c = e4m3x4_rn(in[i], 0.0f, 0.0f, 0.0f);
      else if (op == 5) c = e4m3_sr(in[i], 0xFFFFu - (aux[i] & 0xFFFFu));
      else if (op == 7)
        c = e4m3_sr_hi(in[i], (((0xFFFFu - aux[i]) & 0xFFFFu) << 8) | 0x400000F0u) >> 24;
      else c = (uint32_t)(mx_shared_exp(in[i]) + 127);
      out[i] = (uint8_t)(c & 0xFFu);
    }
    return;
  }
  const int64_t ngroups = (n + 7) / 8;
  for (int64_t gi = t0; gi < ngroups; gi += stride) {
    const int64_t e0 = gi * 8;
    float v[8];
    uint32_t r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[k] = e0 + k < n ? in[e0 + k] : 0.0f;
      r[k] = (op == 3 && e0 + k < n) ? (aux[e0 + k] & 0xFFFFu) : 0u;
    }
    f2 y[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = make_float2(v[2 * k], v[2 * k + 1]);
    const uint4 rb = make_uint4(r[0] | (r[1] << 16), r[2] | (r[3] << 16), r[4] | (r[5] << 16),
                                r[6] | (r[7] << 16));
    const uint32_t w = op == 0 ? e2m1x8_rn(y) : sr8(y, rb);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (e0 + k < n) out[e0 + k] = (uint8_t)((w >> (4 * k)) & 15u);
  }
}

__global__ void sr_bits_kernel(const SrKey key, uint32_t dir, uint64_t idx0, int64_t n,
                               uint32_t* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t idx = idx0 + (uint64_t)i;
    const uint4 w = sr_group_bits(key, dir, idx & ~(uint64_t)7);
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
  sr_bits_kernel<<<grid_for(n), 256, 0, st>>>(make_sr_key(seed, step), dir, idx0, n, out);
  return cudaGetLastError();
}

}  // namespace nvfp4
