// device.cuh -- sm_103a device building blocks of the NVFP4 kernels:
// bf16 unpacking, E2M1 / E4M3 / UE5M3 conversions (Blackwell cvt PTX where
// the hardware has them), Philox4x32-10, the stochastic E2M1 rounder, packed
// f32x2 arithmetic and the per-slice block-scale tables.
//
// All floating-point arithmetic here is IEEE fp32 round-to-nearest; the
// library is compiled with --fmad=false so no product/sum pair is fused unless
// written as an explicit fma.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace nvfp4 {

constexpr float kFltMax = 3.402823466e+38f;

// ---------------------------------------------------------------- bf16 ----
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// Pack two fp32 values to bf16x2 with RNE; `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// Max of |x| over the bf16 halves of 4 words, as a bf16 bit pattern (0..0x7FFF).
__device__ __forceinline__ uint32_t absmax_bits4(uint4 v) {
  uint32_t a = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
  uint32_t b = __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
  uint32_t m = __vmaxu2(a, b);
  return max(m & 0xFFFFu, m >> 16);
}

// ---------------------------------------------------------- packed f32x2 --
// Blackwell executes these as one instruction for two lanes of fp32 work
// (FMUL2 / FFMA2 / FADD2), each lane rounded to nearest like its scalar form.
using f2 = float2;
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) { return __ffma2_rn(a, b, c); }

// ----------------------------------------------------------------- E2M1 ---
// Eight fp32 values (4 pairs) -> 8 codes in one word, element 0 in bits 0..3:
// four conversions into byte registers packed by one vector move.
__device__ __forceinline__ uint32_t e2m1x8_rn(const f2 (&y)[4]) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "f"(y[0].x), "f"(y[0].y), "f"(y[1].x), "f"(y[1].y), "f"(y[2].x), "f"(y[2].y),
        "f"(y[3].x), "f"(y[3].y));
  return w;
}
// Decode the 8 codes of a word into 4 pairs (element 2k in .x of pair k):
// one vector move splits the bytes, the hardware E2M1x2 -> f16x2 conversion
// decodes each (low nibble in the low half), then exact widening to fp32.
__device__ __forceinline__ void e2m1x8_to_f2(uint32_t w, f2 (&q)[4]) {
  uint32_t h0, h1, h2, h3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
  q[0] = __half22float2(*reinterpret_cast<__half2*>(&h0));
  q[1] = __half22float2(*reinterpret_cast<__half2*>(&h1));
  q[2] = __half22float2(*reinterpret_cast<__half2*>(&h2));
  q[3] = __half22float2(*reinterpret_cast<__half2*>(&h3));
}

// --------------------------------------------------------- block scales ---
// E4M3 encode of t >= 0: RNE, saturating at 448 (cvt ... satfinite).
__device__ __forceinline__ uint32_t e4m3_encode(float t) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}"
      : "=r"(r) : "f"(0.0f), "f"(t));
  return r & 0xFFu;
}
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  uint32_t e = (c >> 3) & 15u, m = c & 7u;
  if (e == 0) return (float)m * 0.001953125f;  // m * 2^-9, exact
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}
// UE5M3 (unsigned, bias 15, exponent field 0 subnormal, all codes finite,
// max 1.875 * 2^16): RNE encode of t >= 0, saturating. No hardware path.
__device__ __forceinline__ uint32_t ue5m3_encode(float t) {
  if (!(t < 122880.0f)) return 255u;
  if (t < 6.103515625e-05f) return __float2uint_rn(__fmul_rn(t, 131072.0f));  // m * 2^-17
  uint32_t u = __float_as_uint(t);
  uint32_t r = u + 0x7FFFFu + ((u >> 20) & 1u);  // round the mantissa at bit 20
  return min((r >> 20) - (112u << 3), 255u);     // rebias exponent 127 -> 15
}
__device__ __forceinline__ float ue5m3_value(uint32_t c) {
  uint32_t e = (c >> 3) & 31u, m = c & 7u;
  if (e == 0) return (float)m * 7.62939453125e-06f;  // m * 2^-17, exact
  return __uint_as_float(((e + 112u) << 23) | (m << 20));
}
template <int FMT>
__device__ __forceinline__ uint32_t scale_encode(float t) {
  if constexpr (FMT == 0) return e4m3_encode(t); else return ue5m3_encode(t);
}
template <int FMT>
__device__ __forceinline__ float scale_value(uint32_t c) {
  if constexpr (FMT == 0) return e4m3_value(c); else return ue5m3_value(c);
}

// Per-slice constants of the two-level scale: g = gamax / (6 M) (g = 1 for a
// zero amax), and rden_k = 1 / (k g) for the targets k = 6 and k = 4 (clamped
// to FLT_MAX, so a vanishing g saturates the block scales instead of making
// 0 * inf).
struct SliceScale {
  float g, rden6, rden4;
  bool bad;
};
__device__ __forceinline__ SliceScale slice_scale(float gamax, float M) {
  SliceScale s;
  s.bad = !(gamax >= 0.0f) || gamax > kFltMax;
  float g = 1.0f;
  if (!s.bad && gamax > 0.0f) g = __fdiv_rn(gamax, __fmul_rn(6.0f, M));
  s.g = g;
  s.rden6 = fminf(__frcp_rn(__fmul_rn(6.0f, g)), kFltMax);
  s.rden4 = fminf(__frcp_rn(__fmul_rn(4.0f, g)), kFltMax);
  return s;
}
// Table entry for a block-scale code: d = dec(code) * g and inv = 1 / d
// (clamped to FLT_MAX; 0 when d == 0).
template <int FMT>
__device__ __forceinline__ void scale_entry(uint32_t code, float g, float& d, float& inv) {
  d = __fmul_rn(scale_value<FMT>(code), g);
  inv = 0.0f;
  if (d > 0.0f) inv = fminf(__frcp_rn(d), kFltMax);
}

// --------------------------------------------------------------- Philox ---
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32 -> 64 multiplies, key (seed, step) bumped by the Weyl constants
// between rounds. The ten round keys are the same for every element of a
// launch, so for the row, dual, per-token and re-quantisation kernels the
// host computes them once and passes them as launch parameters: each round's
// key XOR then reads a launch constant instead of re-deriving the key
// schedule for every group of 8 elements. The 16x16 tile and MXFP8
// quantisers derive them in the kernel (make_sr_key), which measured faster
// there: the larger parameter block changed their register allocation.
struct SrKey {
  uint32_t k0[10], k1[10];
};
__host__ __device__ inline SrKey make_sr_key(uint32_t seed, uint32_t step) {
  SrKey k;
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = seed + (uint32_t)r * 0x9E3779B9u;
    k.k1[r] = step + (uint32_t)r * 0xBB67AE85u;
  }
  return k;
}
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const SrKey& key) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;  // one 32x32 -> 64 multiply
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ key.k0[r], (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ key.k1[r], (uint32_t)p0);
  }
  return c;
}
// The 128 random bits of the group of 8 elements starting at flat index
// idx0 (idx0 % 8 == 0) of an encoding in direction dir (0 rows, 1 columns).
__device__ __forceinline__ uint4 sr_group_bits(const SrKey& key, uint32_t dir, uint64_t idx0) {
  uint64_t j = idx0 >> 3;
  return philox4x32_10(make_uint4((uint32_t)j, (uint32_t)(j >> 32), dir, 0u), key);
}
// Random bits of element k (0..7) of a group.
__device__ __forceinline__ uint32_t sr_bits_of(const uint4& w, int k) {
  uint32_t word = (k >> 1) == 0 ? w.x : (k >> 1) == 1 ? w.y : (k >> 1) == 2 ? w.z : w.w;
  return (k & 1) ? (word >> 16) : (word & 0xFFFFu);
}

// Three-input fp32 maximum (one instruction on sm_100 and later); like fmaxf
// it returns the other operands when one is NaN.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Stochastic E2M1 rounding of 8 values (4 pairs) with the group's 128 random
// bits rb (value k uses the 16-bit half k%2 of word k/2): |y| rounds up to the
// next grid value iff v / 2^16 < p, p = (|y| - lo) / (hi - lo).
// E2M1 is a small float (2 exponent bits, bias 1, 1 mantissa bit), and the
// construction is the one of the stochastic E4M3 rounder below: let P be an
// fp32 pattern whose exponent and top mantissa bit spell the lower
// neighbour's code once the exponent is rebiased (127 -> 1) and whose 22
// mantissa bits below hold f = ceil(p * 2^22). In 4 P + n, with
// n = ((0xFFFF - v) << 8) | 0x040000FC, the 0x04 byte does the rebias (mod 4
// on the two exponent bits that stay; the bits above the code are not used),
// 0xFC rounds f up to 16 bits, and the carry out of the fraction, which
// happens iff ceil(p * 2^16) > v, lifts the code in bits 24..26 to the upper
// neighbour. For |y| in [1, 6] P is the pattern of |y| (capped at 6, code 7:
// saturation, and where NaN and Inf land too). Below 1 the grid is uniform
// with spacing 1/2, and P is the pattern of 1/2 + |y|/2 rounded up, which
// lies in [1/2, 1), where fp32 values are 2^-24 apart: its mantissa is
// ceil(|y| * 2^23) = code * 2^22 + f over the exponent of 1/2, which the
// rebias turns into code 0 or 1. One maximum picks the pattern: 1/2 + |y|/2
// exceeds |y| exactly when |y| < 1. The codes (top bytes) are gathered with
// byte permutes, even values in one word and odd values in another, and
// merged as nibbles; the sign bits are those of the round-to-nearest codes
// of the same values (both copy the sign of y).
__device__ __forceinline__ uint32_t e2m1_sr_word(float y, uint32_t n) {
  const float a = fminf(fabsf(y), 6.0f);
  return (__float_as_uint(fmaxf(a, __fmaf_ru(a, 0.5f, 0.5f))) << 2) + n;
}
// sign: the sign bits of the 8 codes (bit 3 of each nibble).
__device__ __forceinline__ uint32_t sr8_signed(const f2 (&y)[4], const uint4& rb, uint32_t sign) {
  const uint32_t nw[4] = {~rb.x, ~rb.y, ~rb.z, ~rb.w};  // 0xFFFF - v in each half
  uint32_t w[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // n for the low / high half of nw[k]
    w[2 * k] = e2m1_sr_word(y[k].x, __byte_perm(nw[k], 0x040000FCu, 0x7104u));
    w[2 * k + 1] = e2m1_sr_word(y[k].y, __byte_perm(nw[k], 0x040000FCu, 0x7324u));
  }
  const uint32_t even = __byte_perm(__byte_perm(w[0], w[2], 0x0073u),
                                    __byte_perm(w[4], w[6], 0x0073u), 0x5410u);
  const uint32_t odd = __byte_perm(__byte_perm(w[1], w[3], 0x0073u),
                                   __byte_perm(w[5], w[7], 0x0073u), 0x5410u);
  return (even & 0x07070707u) | ((odd & 0x07070707u) << 4) | sign;
}
// Sign bits of the E2M1 codes of 8 values (bit 3 of each nibble).
__device__ __forceinline__ uint32_t e2m1_signs(const f2 (&y)[4]) {
  return e2m1x8_rn(y) & 0x88888888u;
}
__device__ __forceinline__ uint32_t sr8(const f2 (&y)[4], const uint4& rb) {
  return sr8_signed(y, rb, e2m1_signs(y));
}

// ------------------------------------------------- MXFP8 (E4M3 elements) --
// Signed E4M3 codes of four fp32 values (y0 in bits 0..7), round to nearest
// even, saturating to +-448 (cvt ... satfinite; the sign of y is kept).
__device__ __forceinline__ uint32_t e4m3x4_rn(float y0, float y1, float y2, float y3) {
  uint32_t w;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(w) : "f"(y0), "f"(y1), "f"(y2), "f"(y3));
  return w;
}
// Stochastic rounding onto the signed E4M3 grid, for |y| <= 448: |y| rounds
// up iff v / 2^16 < p, p the position of |y| between its two grid neighbours
// and v the 16 random bits. n8 = ((0xFFFF - v) << 8) | 0x400000F0 (the
// constant fills bytes the random bits do not use). Returns a word whose top
// byte is the magnitude code (e4m3_sr_mag_hi) or the signed code (e4m3_sr_hi).
// Construction: let P be an fp32 pattern whose exponent and top 3 mantissa
// bits spell the lower neighbour's code once the exponent is rebiased
// (127 -> 7) and whose 20 mantissa bits below hold f = ceil(p * 2^20). Then
// in 16 P + n8 the 0x40 byte does the rebias (mod 2^32; the sign bit and the
// top exponent bits fall off), 0xF0 rounds f up to 16 bits, and the carry
// out of the fraction, which happens iff ceil(f / 16) = ceil(p * 2^16) > v,
// lifts the code to the upper neighbour. For |y| >= 2^-6 (E4M3 normals) P is
// the pattern of |y| itself. Below 2^-6 the grid is uniform with spacing
// 2^-9 (the subnormals), and P is the pattern of 2^-7 + |y| / 2 rounded up:
// that value lies in [2^-7, 2^-6), where fp32 values are 2^-30 apart, so its
// mantissa is ceil(|y| * 2^29) = code * 2^20 + f over the exponent of 2^-7,
// which the rebias turns into code 0. One maximum picks the right pattern:
// 2^-7 + |y| / 2 exceeds |y| exactly when |y| < 2^-6 (and rounding it up
// never lifts it above |y| otherwise).
__device__ __forceinline__ uint32_t e4m3_sr_mag_hi(float y, uint32_t n8) {
  const float a = fabsf(y);
  return (__float_as_uint(fmaxf(a, __fmaf_ru(a, 0.5f, 0.0078125f))) << 4) + n8;
}
__device__ __forceinline__ uint32_t e4m3_sr_hi(float y, uint32_t n8) {
  return e4m3_sr_mag_hi(y, n8) | (__float_as_uint(y) & 0x80000000u);
}
// (0xFFFF - v) << 8 | 0x400000F0 for the 16-bit half h of the complemented
// draw word nw = ~w (v = half h of w): one byte permute.
__device__ __forceinline__ uint32_t e4m3_sr_n8(uint32_t nw, int h) {
  return __byte_perm(nw, 0x400000F0u, h ? 0x7324u : 0x7104u);
}
// One value, saturating: |y| >= 448 (and NaN) gives +-448 (code 0x7E).
__device__ __forceinline__ uint32_t e4m3_sr(float y, uint32_t nv) {
  const float c = __uint_as_float(__float_as_uint(fminf(fabsf(y), 448.0f)) |
                                  (__float_as_uint(y) & 0x80000000u));
  return e4m3_sr_hi(c, ((nv & 0xFFFFu) << 8) | 0x400000F0u) >> 24;
}
// Shared exponent of an MX block whose largest |value| is amax: the smallest
// e with amax <= 448 * 2^e (448 = E4M3's largest value), i.e. the unbiased
// exponent of amax minus 8, plus 1 when its significand exceeds 1.75,
// clamped to [-127, 127] (zero and fp32-subnormal amax give -127).
__device__ __forceinline__ int mx_shared_exp(float amax) {
  const uint32_t A = __float_as_uint(amax);
  int e = (int)(A >> 23) - 135 + ((A & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}
// 2^-e for e in [-127, 127] (2^-127 is an fp32 subnormal).
__device__ __forceinline__ float exp2_neg(int e) {
  return e == 127 ? __uint_as_float(0x00200000u) : __uint_as_float((uint32_t)(127 - e) << 23);
}

// ------------------------------------------------------------- cp.async ---
// 16-byte global -> shared copy that bypasses L1 (streamed data), grouped and
// awaited per thread: a thread only ever reads back the slots it filled, so
// no block-level barrier is involved.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
// The same with the source byte count given: 0 writes 16 zero bytes and reads
// nothing (a tile chunk past the tensor's edge).
__device__ __forceinline__ void cp_async16_zfill(void* smem, const void* gmem, uint32_t bytes) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------ programmatic dependent launch --
// Kernels are launched with programmatic stream serialisation (launch_pdl),
// so a kernel may be scheduled while the preceding kernel on the stream is
// still draining. Every kernel therefore waits for its predecessor to
// complete (and its writes to be visible) before it touches global memory,
// then lets its own dependent launch early; both are hardware operations
// (griddepcontrol), no-ops when the launch had no programmatic dependency.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------ division by a constant --
// n / d for 32-bit unsigned n and a divisor fixed at launch, by the
// multiply-high method of Granlund and Montgomery ("Division by invariant
// integers using multiplication", PLDI 1994, figure 4.1): with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// t = mulhi(m, n), n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0).
struct FastDiv {
  uint32_t m, s1, s2;
};
__device__ __forceinline__ uint32_t fastdiv(uint32_t n, const FastDiv& f) {
  const uint32_t t = __umulhi(n, f.m);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

// ---------------------------------------------------------- status word ---
__device__ __forceinline__ void flag(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

}  // namespace nvfp4
