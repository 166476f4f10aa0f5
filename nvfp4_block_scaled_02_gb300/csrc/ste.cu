// ste.cu -- scale learning: fake quantisation forward and the straight-
// through-estimator backward for single (tied) and dual (pre/post) per-block
// scales, with fp32 or FP8-rounded scales, and the export of learned scales
// to an NVFP4 encoding (Scale Learning blog, "How Scale Learning Works").
//
// Both kernels stream 1x16 row blocks with two lanes per block (8 values and
// one 128-bit load per lane per tensor), grid-stride over chunks of 8 values
// with grids of one wave of resident CTAs: each thread first issues the
// loads of its next few chunks, then computes them (two for the forward with
// fp32 scales; one for the FP8-scale forward, the backward, which loads two
// tensors, and the export; deeper runs measured slower). Per-block sums are fp32 in the fixed
// order: within each lane's 8 values, even and odd positions accumulate in
// the two halves of an f32x2 fma accumulator; half = even + odd; the block
// sum is the lower half plus the upper half (one shuffle).
#include "device.cuh"
#include "encode.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kUnrollFwd = 2;     // chunks in flight per thread: forward (fp32 scales)
constexpr int kUnrollBwd = 1;     // backward
constexpr int kUnrollExport = 1;  // export
constexpr float kFltMin = 1.175494351e-38f;

__device__ __forceinline__ bool scale_ok(float sp, float so) {
  return sp >= kFltMin && sp <= kFltMax && fabsf(so) <= kFltMax;
}

__device__ __forceinline__ bool finite8(const uint4& v) {
  return absmax_bits4(v) < 0x7F80u;
}

// FP8 block scales (Scale Learning blog, "How Scale Learning Works": the scale
// is itself quantised to FP8): per tensor g = gamax / (6 * 448) (1 for a zero
// or bad amax), rg = 1/g clamped to FLT_MAX; Q8(s) = dec(E4M3(s * rg)) * g
// for s >= 0. The raw scales must be usable too: s_pre a normal positive
// number, s_post finite and not negative, and Q8(s_pre) not below FLT_MIN.
struct Fp8Unit {
  float g, rg;
  bool bad;
};
__device__ __forceinline__ Fp8Unit fp8_unit(const float* gamax) {
  const SliceScale ss = slice_scale(*gamax, 448.0f);
  return Fp8Unit{ss.g, fminf(__frcp_rn(ss.g), kFltMax), ss.bad};
}
__device__ __forceinline__ uint32_t q8_code(float s, const Fp8Unit& u) {
  return e4m3_encode(__fmul_rn(s, u.rg));
}
__device__ __forceinline__ float q8(float s, const Fp8Unit& u) {
  return s >= 0.0f ? __fmul_rn(e4m3_value(q8_code(s, u)), u.g) : 0.0f;
}
__device__ __forceinline__ bool raw_fp8_scales_ok(float sp, float so, float spq) {
  return sp >= kFltMin && sp <= kFltMax && so >= 0.0f && so <= kFltMax && spq >= kFltMin;
}

template <bool Q8>
__device__ __forceinline__ void fakequant_chunk(const SteParams& p, const Fp8Unit& u, int64_t ch,
                                                const uint4& v, float sp, float so) {
  if constexpr (Q8) {
    const float spr = sp, sor = so;
    sp = q8(spr, u);
    so = q8(sor, u);
    if ((ch & 1) == 0 && !raw_fp8_scales_ok(spr, sor, sp)) flag(p.status, NVFP4_DEV_BAD_SCALE_BIT);
  }
  if ((ch & 1) == 0 && !scale_ok(sp, so)) flag(p.status, NVFP4_DEV_BAD_SCALE_BIT);
  if (!finite8(v)) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
  const float inv = __frcp_rn(sp);
  f2 x[4], y[4], q[4];
  unpack8(v, x);
  const f2 iv = make_float2(inv, inv);
#pragma unroll
  for (int k = 0; k < 4; ++k) y[k] = f2_mul(x[k], iv);
  e2m1x8_to_f2(e2m1x8_rn(y), q);
  __stcs(p.out + ch, dequant8(q, so));
}

template <bool Q8>
__global__ void __launch_bounds__(kThreads) fakequant_fwd_kernel(const SteParams p) {
  pdl_begin();
  constexpr int U = Q8 ? 1 : kUnrollFwd;  // the FP8-scale form has more arithmetic per chunk
  const int64_t nchunks = p.nblocks * 2;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  Fp8Unit u{1.0f, 1.0f, false};
  if constexpr (Q8) {
    u = fp8_unit(p.gamax);
    if (u.bad && blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
  }
  for (int64_t ch0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; ch0 < nchunks;
       ch0 += stride * U) {
    uint4 v[U];
    float sp[U], so[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int64_t ch = ch0 + k * stride;
      v[k] = make_uint4(0, 0, 0, 0);
      sp[k] = so[k] = 1.0f;
      if (ch < nchunks) {
        v[k] = __ldcs(p.x + ch);
        sp[k] = p.s_pre[ch >> 1];
        so[k] = p.s_post ? p.s_post[ch >> 1] : sp[k];
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (ch0 + k * stride < nchunks) fakequant_chunk<Q8>(p, u, ch0 + k * stride, v[k], sp[k], so[k]);
  }
}

// One chunk of the backward: ok = the chunk exists (every lane of the warp
// calls this together, for the pair shuffle).
template <bool TIED, bool WANT_GX, bool Q8>
__device__ __forceinline__ void scale_grad_chunk(const SteParams& p, const Fp8Unit& u, int64_t ch,
                                                 bool ok, const uint4& xv, const uint4& gv,
                                                 float sp, float so) {
  const int64_t b = ch >> 1;
  if (ok) {
    if constexpr (Q8) {
      // the gradients below are those of the rounded scales, passed through
      const float spr = sp, sor = so;
      sp = q8(spr, u);
      so = TIED ? sp : q8(sor, u);
      if ((ch & 1) == 0 && !raw_fp8_scales_ok(spr, sor, sp)) flag(p.status, NVFP4_DEV_BAD_SCALE_BIT);
    }
    if ((ch & 1) == 0 && !scale_ok(sp, so)) flag(p.status, NVFP4_DEV_BAD_SCALE_BIT);
    if (!finite8(xv) || !finite8(gv)) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
  }
  const float inv = __frcp_rn(sp);
  const float a = TIED ? 1.0f : __fmul_rn(so, inv);
  f2 x[4], g[4], r[4], q[4];
  unpack8(xv, x);
  unpack8(gv, g);
  const f2 iv = make_float2(inv, inv);
#pragma unroll
  for (int k = 0; k < 4; ++k) r[k] = f2_mul(x[k], iv);
  e2m1x8_to_f2(e2m1x8_rn(r), q);

  f2 acc0 = make_float2(0.0f, 0.0f), acc1 = acc0;
  uint32_t gx[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const bool in_x = r[k].x >= -6.0f && r[k].x <= 6.0f;
    const bool in_y = r[k].y >= -6.0f && r[k].y <= 6.0f;
    if constexpr (WANT_GX) {
      const float gxx = in_x ? (TIED ? g[k].x : __fmul_rn(g[k].x, a)) : 0.0f;
      const float gxy = in_y ? (TIED ? g[k].y : __fmul_rn(g[k].y, a)) : 0.0f;
      gx[k] = pack_bf16x2(gxx, gxy);
    }
    if constexpr (TIED) {
      const f2 t = make_float2(in_x ? __fsub_rn(q[k].x, r[k].x) : q[k].x,
                               in_y ? __fsub_rn(q[k].y, r[k].y) : q[k].y);
      acc0 = f2_fma(g[k], t, acc0);
    } else {
      acc0 = f2_fma(g[k], q[k], acc0);
      const f2 rin = make_float2(in_x ? r[k].x : 0.0f, in_y ? r[k].y : 0.0f);
      acc1 = f2_fma(g[k], rin, acc1);
    }
  }
  if constexpr (WANT_GX)
    if (ok) __stcs(p.out + ch, make_uint4(gx[0], gx[1], gx[2], gx[3]));
  const float h0 = __fadd_rn(acc0.x, acc0.y);
  const float s0 = __fadd_rn(h0, __shfl_xor_sync(0xFFFFFFFFu, h0, 1));
  if constexpr (TIED) {
    if (ok && (ch & 1) == 0) p.gs_pre[b] = s0;
  } else {
    const float h1 = __fadd_rn(acc1.x, acc1.y);
    const float s1 = __fadd_rn(h1, __shfl_xor_sync(0xFFFFFFFFu, h1, 1));
    if (ok && (ch & 1) == 0) {
      if (p.gs_post) p.gs_post[b] = s0;
      p.gs_pre[b] = __fmul_rn(-a, s1);
    }
  }
}

template <bool TIED, bool WANT_GX, bool Q8>
__global__ void __launch_bounds__(kThreads) scale_grad_bwd_kernel(const SteParams p) {
  pdl_begin();
  const int64_t nchunks = p.nblocks * 2;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  Fp8Unit u{1.0f, 1.0f, false};
  if constexpr (Q8) {
    u = fp8_unit(p.gamax);
    if (u.bad && blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
  }
  // all lanes of a warp iterate together (stride and start are warp-aligned),
  // so the pair shuffle always has its partner
  const int64_t start = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t nwarp_iters = (nchunks + stride - 1) / stride;
  for (int64_t it0 = 0; it0 < nwarp_iters; it0 += kUnrollBwd) {
    uint4 xv[kUnrollBwd], gv[kUnrollBwd];
    float sp[kUnrollBwd], so[kUnrollBwd];
#pragma unroll
    for (int k = 0; k < kUnrollBwd; ++k) {
      const int64_t ch = start + (it0 + k) * stride;
      xv[k] = gv[k] = make_uint4(0, 0, 0, 0);
      sp[k] = so[k] = 1.0f;
      if (ch < nchunks) {
        xv[k] = __ldcs(p.x + ch);
        gv[k] = __ldcs(p.gq + ch);
        sp[k] = p.s_pre[ch >> 1];
        so[k] = TIED ? sp[k] : p.s_post[ch >> 1];
      }
    }
#pragma unroll
    for (int k = 0; k < kUnrollBwd; ++k) {
      if (it0 + k >= nwarp_iters) break;  // warp-uniform
      const int64_t ch = start + (it0 + k) * stride;
      scale_grad_chunk<TIED, WANT_GX, Q8>(p, u, ch, ch < nchunks, xv[k], gv[k], sp[k], so[k]);
    }
  }
}

// Export (Scale Learning blog, "How Scale Learning Works": the post-scale is
// baked into the checkpoint, the pre-scale discarded): the fake-quant
// forward's codes (rounding at Q8(s_pre)) and the E4M3 byte of s_post, an
// NVFP4 row encoding whose de-quantisation is that forward. Two lanes per
// block, 8 codes (one 32-bit word) each; the even lane writes the scale byte.
__device__ __forceinline__ void export_chunk(const SteParams& p, const Fp8Unit& u, int64_t ch,
                                             const uint4& v, float spr, float sor) {
  const int64_t b = ch >> 1;
  const float sp = q8(spr, u);
  if ((ch & 1) == 0) {
    if (!raw_fp8_scales_ok(spr, sor, sp)) flag(p.status, NVFP4_DEV_BAD_SCALE_BIT);
    p.scales[b] = (uint8_t)(sor >= 0.0f ? q8_code(sor, u) : 0u);
  }
  if (!finite8(v)) flag(p.status, NVFP4_DEV_NONFINITE_INPUT_BIT);
  const float inv = __frcp_rn(sp);
  f2 x[4], y[4];
  unpack8(v, x);
  const f2 iv = make_float2(inv, inv);
#pragma unroll
  for (int k = 0; k < 4; ++k) y[k] = f2_mul(x[k], iv);
  __stcs(reinterpret_cast<uint32_t*>(p.codes) + ch, e2m1x8_rn(y));
}

__global__ void __launch_bounds__(kThreads) export_scales_kernel(const SteParams p) {
  pdl_begin();
  const int64_t nchunks = p.nblocks * 2;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const Fp8Unit u = fp8_unit(p.gamax);
  if (u.bad && blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, NVFP4_DEV_BAD_AMAX_BIT);
  for (int64_t ch0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; ch0 < nchunks;
       ch0 += stride * kUnrollExport) {
    uint4 v[kUnrollExport];
    float spr[kUnrollExport], sor[kUnrollExport];
#pragma unroll
    for (int k = 0; k < kUnrollExport; ++k) {
      const int64_t ch = ch0 + k * stride;
      v[k] = make_uint4(0, 0, 0, 0);
      spr[k] = sor[k] = 1.0f;
      if (ch < nchunks) {
        v[k] = __ldcs(p.x + ch);
        spr[k] = p.s_pre[ch >> 1];
        sor[k] = p.s_post ? p.s_post[ch >> 1] : spr[k];
      }
    }
#pragma unroll
    for (int k = 0; k < kUnrollExport; ++k)
      if (ch0 + k * stride < nchunks) export_chunk(p, u, ch0 + k * stride, v[k], spr[k], sor[k]);
  }
}

// Grid-stride grids sized to one wave of resident CTAs (the count is taken
// once per kernel instantiation).
template <auto K>
unsigned grid_for(int64_t nchunks) {
  static const int per_sm = resident_ctas(K, kThreads);
  const int64_t want = (nchunks + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)sm_count() * per_sm;
  return (unsigned)std::max<int64_t>(1, std::min(want, cap));
}

}  // namespace

cudaError_t launch_fakequant_fwd(const SteParams& p, cudaStream_t st) {
  const int64_t n = p.nblocks * 2;
  if (p.gamax)
    return launch_pdl(fakequant_fwd_kernel<true>, dim3(grid_for<fakequant_fwd_kernel<true>>(n)),
                      dim3(kThreads), st, p);
  return launch_pdl(fakequant_fwd_kernel<false>, dim3(grid_for<fakequant_fwd_kernel<false>>(n)),
                    dim3(kThreads), st, p);
}

template <bool TIED, bool WANT_GX, bool Q8>
cudaError_t launch_bwd_k(const SteParams& p, cudaStream_t st) {
  constexpr auto k = scale_grad_bwd_kernel<TIED, WANT_GX, Q8>;
  return launch_pdl(k, dim3(grid_for<k>(p.nblocks * 2)), dim3(kThreads), st, p);
}

template <bool Q8>
cudaError_t launch_bwd_t(const SteParams& p, cudaStream_t st) {
  const bool tied = p.s_post == nullptr, want_gx = p.out != nullptr;
  if (tied && want_gx) return launch_bwd_k<true, true, Q8>(p, st);
  if (tied) return launch_bwd_k<true, false, Q8>(p, st);
  if (want_gx) return launch_bwd_k<false, true, Q8>(p, st);
  return launch_bwd_k<false, false, Q8>(p, st);
}

cudaError_t launch_scale_grad_bwd(const SteParams& p, cudaStream_t st) {
  return p.gamax ? launch_bwd_t<true>(p, st) : launch_bwd_t<false>(p, st);
}

cudaError_t launch_export_scales(const SteParams& p, cudaStream_t st) {
  return launch_pdl(export_scales_kernel, dim3(grid_for<export_scales_kernel>(p.nblocks * 2)),
                    dim3(kThreads), st, p);
}

}  // namespace nvfp4
