// encode.cuh -- the per-block NVFP4 encoder shared by the row kernel (two
// lanes per 16-value block, 8 values each) and the column/dual kernel (one
// lane per block). The block's values are held as 4 or 8 f32x2 pairs in
// registers; nothing touches memory.
//
// Steps for one block (End-to-End 4-Bit Training, "Low-precision formats on
// Blackwell"; UE5M3 blog, math derivation; "Four Over Six", method):
//   amax -> t_k = amax * (1/(k g)) -> scale code Q(t_k) -> d_k, inv_k from the
//   per-slice table -> y = x * inv_k -> E2M1 code (RNE or stochastic) ->
//   (4/6) block sum of (x - q d_k)^2 for k = 6, 4, keep 4 iff strictly lower.
#pragma once
#include "device.cuh"

namespace nvfp4 {

// Round 8 values (4 pairs) scaled by inv to E2M1, nibble k = element k.
template <bool SR>
__device__ __forceinline__ uint32_t round8(const f2 (&x)[4], float inv, const uint4& rb) {
  f2 y[4];
  const f2 iv = make_float2(inv, inv);
#pragma unroll
  for (int k = 0; k < 4; ++k) y[k] = f2_mul(x[k], iv);
  if constexpr (!SR) return e2m1x8_rn(y);
  else return sr8(y, rb);
}
// The same with the codes' sign bits given (sign = e2m1_signs(x)): x * inv
// has the sign of x for every inv >= 0 (zeros included), so the two 4/6
// candidates of one block share them.
template <bool SR>
__device__ __forceinline__ uint32_t round8s(const f2 (&x)[4], float inv, const uint4& rb,
                                            uint32_t sign) {
  f2 y[4];
  const f2 iv = make_float2(inv, inv);
#pragma unroll
  for (int k = 0; k < 4; ++k) y[k] = f2_mul(x[k], iv);
  if constexpr (!SR) return e2m1x8_rn(y);
  else return sr8_signed(y, rb, sign);
}

// Sum over 8 values of (x - q d)^2 in the fixed order: even and odd positions
// accumulate separately with fma from +0 (one f32x2 accumulator), then
// even + odd. Also returns the decoded code values.
__device__ __forceinline__ float half_sse(const f2 (&x)[4], uint32_t codes, float d, f2 (&q)[4]) {
  e2m1x8_to_f2(codes, q);
  const f2 nd = make_float2(-d, -d);
  f2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f2 e = f2_fma(q[k], nd, x[k]);
    acc = f2_fma(e, e, acc);
  }
  return __fadd_rn(acc.x, acc.y);
}

// The 4/6 selection metric of 8 values with decoded code values q under
// `rule`: 0 = sum of squared errors (fma order of half_sse), 1 = sum of |e|
// (plain adds, same order), 2 = max |e|. Halves combine by + for rules 0 and 1
// and by max for rule 2.
__device__ __forceinline__ float half_metric_q(const f2 (&x)[4], const f2 (&q)[4], float d,
                                               int rule) {
  const f2 nd = make_float2(-d, -d);
  f2 acc = make_float2(0.0f, 0.0f);
  if (rule == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const f2 e = f2_fma(q[k], nd, x[k]);
      acc = f2_fma(e, e, acc);
    }
    return __fadd_rn(acc.x, acc.y);
  }
  if (rule == 1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const f2 e = f2_fma(q[k], nd, x[k]);
      acc = __fadd2_rn(acc, make_float2(fabsf(e.x), fabsf(e.y)));
    }
    return __fadd_rn(acc.x, acc.y);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const f2 e = f2_fma(q[k], nd, x[k]);
    acc = make_float2(fmaxf(acc.x, fabsf(e.x)), fmaxf(acc.y, fabsf(e.y)));
  }
  return fmaxf(acc.x, acc.y);
}
__device__ __forceinline__ float half_metric(const f2 (&x)[4], uint32_t codes, float d, int rule) {
  f2 q[4];
  e2m1x8_to_f2(codes, q);
  return half_metric_q(x, q, d, rule);
}
__device__ __forceinline__ float combine_halves(float h0, float h1, int rule) {
  return rule == 2 ? fmaxf(h0, h1) : __fadd_rn(h0, h1);
}

// Dequantised bf16 of 8 decoded values times d, packed as a uint4.
__device__ __forceinline__ uint4 dequant8(const f2 (&q)[4], float d) {
  const f2 dd = make_float2(d, d);
  f2 r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) r[k] = f2_mul(q[k], dd);
  return make_uint4(pack_bf16x2(r[0].x, r[0].y), pack_bf16x2(r[1].x, r[1].y),
                    pack_bf16x2(r[2].x, r[2].y), pack_bf16x2(r[3].x, r[3].y));
}

// Unpack a uint4 of 8 bf16 into 4 pairs.
__device__ __forceinline__ void unpack8(const uint4& v, f2 (&x)[4]) {
  x[0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
  x[1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
  x[2] = make_float2(bf16_lo(v.z), bf16_hi(v.z));
  x[3] = make_float2(bf16_lo(v.w), bf16_hi(v.w));
}

struct HalfResult {
  uint32_t codes;  // 8 nibbles
  uint32_t scale;  // block-scale code
  bool pick4;      // 4/6 chose target 4
  uint4 dq;        // 8 bf16
};

// One lane's half of a row block (8 values); its partner lane (lane ^ 1)
// holds the other half. amax_bits: the block's amax as bf16 bits (already
// combined over both halves). Every lane of the warp must call this.
template <int FMT, bool SR, bool FOS>
__device__ __forceinline__ HalfResult encode_half(const f2 (&x)[4], uint32_t amax_bits,
                                                  const SliceScale& ss, const float* s_d,
                                                  const float* s_inv, const uint4& rb,
                                                  bool want_dq, int rule) {
  HalfResult r;
  const float amax = __uint_as_float(amax_bits << 16);
  const uint32_t c6 = scale_encode<FMT>(__fmul_rn(amax, ss.rden6));
  const float d6 = s_d[c6], inv6 = s_inv[c6];
  const uint32_t sg = (SR && FOS) ? e2m1_signs(x) : 0u;
  const uint32_t q6 = FOS ? round8s<SR>(x, inv6, rb, sg) : round8<SR>(x, inv6, rb);
  if constexpr (!FOS) {
    r.codes = q6;
    r.scale = c6;
    r.pick4 = false;
    if (want_dq) {
      f2 q[4];
      e2m1x8_to_f2(q6, q);
      r.dq = dequant8(q, d6);
    }
  } else {
    const uint32_t c4 = scale_encode<FMT>(__fmul_rn(amax, ss.rden4));
    const float d4 = s_d[c4], inv4 = s_inv[c4];
    const uint32_t q4 = round8s<SR>(x, inv4, rb, sg);
    f2 v6[4], v4[4];
    e2m1x8_to_f2(q6, v6);
    e2m1x8_to_f2(q4, v4);
    const float h6 = half_metric_q(x, v6, d6, rule);
    const float h4 = half_metric_q(x, v4, d4, rule);
    // the lower half (lane with the block's values 0..7) first
    const float sse6 = combine_halves(h6, __shfl_xor_sync(0xFFFFFFFFu, h6, 1), rule);
    const float sse4 = combine_halves(h4, __shfl_xor_sync(0xFFFFFFFFu, h4, 1), rule);
    r.pick4 = sse4 < sse6;
    r.codes = r.pick4 ? q4 : q6;
    r.scale = r.pick4 ? c4 : c6;
    if (want_dq) {
      f2 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = r.pick4 ? v4[k] : v6[k];
      r.dq = dequant8(v, r.pick4 ? d4 : d6);
    }
  }
  return r;
}

// A whole 16-value block held by one lane as two halves of 8 (row kernel,
// column kernel). The decoded values of the candidates are not kept: the
// chosen codes are decoded again for the dequantised output.
struct BlockResult {
  uint32_t codes[2];
  uint32_t scale;
  bool pick4;
  uint4 dq[2];
};

// Where d = dec(code) * g and 1/d come from: a per-slice shared-memory table
// (one entry per scale code) or, when every row has its own outer scale, the
// same two fp32 operations done per block.
struct TableScales {
  const float* d;
  const float* inv;
  __device__ __forceinline__ void operator()(uint32_t code, float& dd, float& ii) const {
    dd = d[code];
    ii = inv[code];
  }
};
template <int FMT>
struct DirectScales {
  float g;
  __device__ __forceinline__ void operator()(uint32_t code, float& dd, float& ii) const {
    scale_entry<FMT>(code, g, dd, ii);
  }
};

// The block's amax is given as an fp32 value (encode_block_f: fp32 inputs, as
// in re-quantisation) or as bf16 bits (encode_block: bf16 inputs).
template <int FMT, bool SR, bool FOS, class Scales>
__device__ __forceinline__ BlockResult encode_block_f(const f2 (&lo)[4], const f2 (&hi)[4],
                                                      float amax, const SliceScale& ss,
                                                      const Scales& scales, const uint4& rb0,
                                                      const uint4& rb1, bool want_dq,
                                                      int rule = 0) {
  BlockResult r;
  const uint32_t c6 = scale_encode<FMT>(__fmul_rn(amax, ss.rden6));
  float d6, inv6;
  scales(c6, d6, inv6);
  const uint32_t sgl = (SR && FOS) ? e2m1_signs(lo) : 0u, sgh = (SR && FOS) ? e2m1_signs(hi) : 0u;
  const uint32_t a6 = FOS ? round8s<SR>(lo, inv6, rb0, sgl) : round8<SR>(lo, inv6, rb0);
  const uint32_t b6 = FOS ? round8s<SR>(hi, inv6, rb1, sgh) : round8<SR>(hi, inv6, rb1);
  float d = d6;
  if constexpr (!FOS) {
    r.codes[0] = a6;
    r.codes[1] = b6;
    r.scale = c6;
    r.pick4 = false;
  } else {
    const uint32_t c4 = scale_encode<FMT>(__fmul_rn(amax, ss.rden4));
    float d4, inv4;
    scales(c4, d4, inv4);
    const uint32_t a4 = round8s<SR>(lo, inv4, rb0, sgl), b4 = round8s<SR>(hi, inv4, rb1, sgh);
    const float sse6 =
        combine_halves(half_metric(lo, a6, d6, rule), half_metric(hi, b6, d6, rule), rule);
    const float sse4 =
        combine_halves(half_metric(lo, a4, d4, rule), half_metric(hi, b4, d4, rule), rule);
    r.pick4 = sse4 < sse6;
    r.codes[0] = r.pick4 ? a4 : a6;
    r.codes[1] = r.pick4 ? b4 : b6;
    r.scale = r.pick4 ? c4 : c6;
    d = r.pick4 ? d4 : d6;
  }
  if (want_dq) {
    f2 q[4];
    e2m1x8_to_f2(r.codes[0], q);
    r.dq[0] = dequant8(q, d);
    e2m1x8_to_f2(r.codes[1], q);
    r.dq[1] = dequant8(q, d);
  }
  return r;
}
template <int FMT, bool SR, bool FOS, class Scales>
__device__ __forceinline__ BlockResult encode_block(const f2 (&lo)[4], const f2 (&hi)[4],
                                                    uint32_t amax_bits, const SliceScale& ss,
                                                    const Scales& scales, const uint4& rb0,
                                                    const uint4& rb1, bool want_dq,
                                                    int rule = 0) {
  return encode_block_f<FMT, SR, FOS>(lo, hi, __uint_as_float(amax_bits << 16), ss, scales, rb0,
                                      rb1, want_dq, rule);
}

// Per-slice block-scale table in shared memory: for every code c of the
// format, d = dec(c) * g and inv = 1/d. Built by the first 256 threads.
template <int FMT>
__device__ __forceinline__ void build_scale_table(float* s_d, float* s_inv, float g) {
  for (int c = threadIdx.x; c < 256; c += blockDim.x) {
    float d, inv;
    scale_entry<FMT>((uint32_t)c, g, d, inv);
    s_d[c] = d;
    s_inv[c] = inv;
  }
}

}  // namespace nvfp4
