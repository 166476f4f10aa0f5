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

// Both block-scale codes of a block (targets 6 and 4) from one conversion:
// t6's code in bits 0..7, t4's in bits 8..15.
template <int FMT>
__device__ __forceinline__ uint32_t scale_encode2(float t6, float t4) {
  if constexpr (FMT == 0) {
    uint32_t r;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(r) : "f"(t4), "f"(t6));
    return r;
  } else {
    return ue5m3_encode(t6) | (ue5m3_encode(t4) << 8);
  }
}

// Per-slice block-scale table in shared memory, one (d, 1/d) pair per scale
// code: d = dec(code) * g, inv = 1/d. A non-negative block amax never gives
// an E4M3 code above 127 (a finite one at most 126), so only those entries
// are built; the array still has 256 entries, so no code reads outside it.
template <int FMT>
__device__ __forceinline__ void build_scale_table2(float2* tab, float g) {
  constexpr int n = FMT == 0 ? 128 : 256;
  for (int c = threadIdx.x; c < n; c += blockDim.x) {
    float d, inv;
    scale_entry<FMT>((uint32_t)c, g, d, inv);
    tab[c] = make_float2(d, inv);
  }
}

// Magnitude maximum of two bf16x2 words, lane by lane: each half of the
// result is max(|a|, |b|) of the matching halves (NaN if either is NaN); its
// sign bit is not meaningful.
__device__ __forceinline__ uint32_t bmax_abs2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// A whole 16-value block held by one lane as two halves of 8 (row kernel,
// per-token kernel, re-quantisation to NVFP4).
struct BlockResult {
  uint32_t codes[2];
  uint32_t scale;
  bool pick4;
  uint4 dq[2];
};

// Where d = dec(code) * g and 1/d come from: a per-slice shared-memory table
// (one (d, 1/d) pair per scale code, or two arrays) or, when every row has
// its own outer scale, the same two fp32 operations done per block.
struct TableScales {
  const float* d;
  const float* inv;
  __device__ __forceinline__ void operator()(uint32_t code, float& dd, float& ii) const {
    dd = d[code];
    ii = inv[code];
  }
};
struct TableScales2 {
  const float2* tab;
  __device__ __forceinline__ void operator()(uint32_t code, float& dd, float& ii) const {
    const float2 e = tab[code];
    dd = e.x;
    ii = e.y;
  }
};
template <int FMT>
struct DirectScales {
  float g;
  __device__ __forceinline__ void operator()(uint32_t code, float& dd, float& ii) const {
    scale_entry<FMT>(code, g, dd, ii);
  }
};

// One candidate scale on 8 values: y = x * inv, E2M1 codes by RNE or by the
// stochastic rounder (sign bits sg given), and, when want_v, the decoded
// code values in fp32. (Decoding the packed word costs no more than decoding
// the conversion's byte registers: the decode reads a byte of a word.)
template <bool SR>
__device__ __forceinline__ uint32_t cand8(const f2 (&x)[4], float inv, const uint4& rb,
                                          uint32_t sg, bool want_v, f2 (&v)[4]) {
  f2 y[4];
  const f2 iv = make_float2(inv, inv);
#pragma unroll
  for (int k = 0; k < 4; ++k) y[k] = f2_mul(x[k], iv);
  const uint32_t w = SR ? sr8_signed(y, rb, sg) : e2m1x8_rn(y);
  if (want_v) e2m1x8_to_f2(w, v);
  return w;
}

// Dequantised bf16 of the 4/6 choice without a per-value select:
// fma(q4, d4 or 0, q6 * (0 or d6)) is q * d of the chosen candidate bit for
// bit (the other product is a zero of the same sign: both candidates' codes
// carry the sign of x).
__device__ __forceinline__ uint4 dequant8_pick(const f2 (&v4)[4], const f2 (&v6)[4], bool pick4,
                                               float d4, float d6) {
  const float a4 = pick4 ? d4 : 0.0f, a6 = pick4 ? 0.0f : d6;
  const f2 b4 = make_float2(a4, a4), b6 = make_float2(a6, a6);
  f2 t[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) t[k] = f2_fma(v4[k], b4, f2_mul(v6[k], b6));
  return make_uint4(pack_bf16x2(t[0].x, t[0].y), pack_bf16x2(t[1].x, t[1].y),
                    pack_bf16x2(t[2].x, t[2].y), pack_bf16x2(t[3].x, t[3].y));
}

// The block's amax is given as an fp32 value (encode_block_f: fp32 inputs, as
// in re-quantisation) or as bf16 bits (encode_block: bf16 inputs). Each
// candidate's codes are decoded once for its error sum; the dequantised
// output decodes the chosen codes again (keeping both candidates' decoded
// values for a select-free dequant would hold 32 more registers per lane).
template <int FMT, bool SR, bool FOS, class Scales>
__device__ __forceinline__ BlockResult encode_block_f(const f2 (&lo)[4], const f2 (&hi)[4],
                                                      float amax, const SliceScale& ss,
                                                      const Scales& scales, const uint4& rb0,
                                                      const uint4& rb1, bool want_dq,
                                                      int rule = 0) {
  BlockResult r;
  uint32_t c6, c4 = 0;
  if constexpr (FOS) {
    const uint32_t cc =
        scale_encode2<FMT>(__fmul_rn(amax, ss.rden6), __fmul_rn(amax, ss.rden4));
    c6 = cc & 0xFFu;
    c4 = cc >> 8;
  } else {
    c6 = scale_encode<FMT>(__fmul_rn(amax, ss.rden6));
  }
  float d6, inv6;
  scales(c6, d6, inv6);
  const uint32_t sgl = SR ? e2m1_signs(lo) : 0u, sgh = SR ? e2m1_signs(hi) : 0u;
  float d = d6;
  if constexpr (!FOS) {
    f2 v[4];
    r.codes[0] = cand8<SR>(lo, inv6, rb0, sgl, false, v);
    r.codes[1] = cand8<SR>(hi, inv6, rb1, sgh, false, v);
    r.scale = c6;
    r.pick4 = false;
  } else {
    float d4, inv4;
    scales(c4, d4, inv4);
    f2 v[4];
    const uint32_t a6 = cand8<SR>(lo, inv6, rb0, sgl, true, v);
    const float l6 = half_metric_q(lo, v, d6, rule);
    const uint32_t b6 = cand8<SR>(hi, inv6, rb1, sgh, true, v);
    const float sse6 = combine_halves(l6, half_metric_q(hi, v, d6, rule), rule);
    const uint32_t a4 = cand8<SR>(lo, inv4, rb0, sgl, true, v);
    const float l4 = half_metric_q(lo, v, d4, rule);
    const uint32_t b4 = cand8<SR>(hi, inv4, rb1, sgh, true, v);
    const float sse4 = combine_halves(l4, half_metric_q(hi, v, d4, rule), rule);
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

// One lane's half (8 values, 4 pairs) of a 16-value block whose other half
// sits in lane ^ 1; amax_bits is the whole block's amax as bf16 bits. Every
// lane of the warp must call this (the two halves' sums are exchanged by a
// shuffle). With 4/6 both candidates are rounded, decoded once, their error
// sums taken in the fixed order (even and odd positions in one f32x2
// accumulator, then even + odd, then lower half + upper half), and the
// dequantised output picks the chosen candidate without a per-value select
// (dequant8_pick).
struct HalfOut {
  uint32_t codes;  // 8 nibbles
  uint32_t scale;  // block-scale code
  bool pick4;      // 4/6 chose target 4
  uint4 dq;        // 8 bf16
};
template <int FMT, bool SR, int FOS>
__device__ __forceinline__ HalfOut encode_half8(const f2 (&x)[4], uint32_t amax_bits,
                                                const SliceScale& ss, const float2* tab,
                                                const uint4& rb, bool want_dq, int rule) {
  HalfOut r;
  const float amax = __uint_as_float(amax_bits << 16);
  uint32_t c6, c4 = 0;
  if constexpr (FOS != 0) {
    const uint32_t cc =
        scale_encode2<FMT>(__fmul_rn(amax, ss.rden6), __fmul_rn(amax, ss.rden4));
    c6 = cc & 0xFFu;
    c4 = cc >> 8;
  } else {
    c6 = scale_encode<FMT>(__fmul_rn(amax, ss.rden6));
  }
  const float2 e6 = tab[c6];
  const uint32_t sg = SR ? e2m1_signs(x) : 0u;
  f2 v6[4];
  const uint32_t q6 = cand8<SR>(x, e6.y, rb, sg, FOS != 0 || want_dq, v6);
  if constexpr (FOS == 0) {
    r.codes = q6;
    r.scale = c6;
    r.pick4 = false;
    if (want_dq) r.dq = dequant8(v6, e6.x);
  } else {
    const float2 e4 = tab[c4];
    f2 v4[4];
    const uint32_t q4 = cand8<SR>(x, e4.y, rb, sg, true, v4);
    const int ru = FOS == 1 ? 0 : rule;
    const float h6 = half_metric_q(x, v6, e6.x, ru);
    const float h4 = half_metric_q(x, v4, e4.x, ru);
    const float sse6 = combine_halves(h6, __shfl_xor_sync(0xFFFFFFFFu, h6, 1), ru);
    const float sse4 = combine_halves(h4, __shfl_xor_sync(0xFFFFFFFFu, h4, 1), ru);
    r.pick4 = sse4 < sse6;
    r.codes = r.pick4 ? q4 : q6;
    r.scale = r.pick4 ? c4 : c6;
    if (want_dq) r.dq = dequant8_pick(v4, v6, r.pick4, e4.x, e6.x);
  }
  return r;
}

}  // namespace nvfp4
