// common.cuh -- device helpers shared by the quantization kernels: BF16
// unpacking, the hardware E4M3 conversion, and the exact E4M3(RN32(x / S))
// coding used by every quantizer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace w8a8 {

// ---- BF16 words -> binary32 (exact: BF16 is the top half of a binary32) ----
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max(|a|, |b|) of the two BF16 halves of each 32-bit word, as binary32.
__device__ __forceinline__ float absmax_bf16x2(uint32_t w, float m) {
  return fmaxf(m, fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w))));
}

// ---- hardware conversion: two binary32 -> two E4M3 codes ----
// cvt.rn.satfinite rounds to nearest even and clamps magnitudes beyond 448
// to 448 (NaN stays NaN).  The first source lands in the upper byte, so the
// result holds code(lo) in bits 0..7 and code(hi) in bits 8..15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// two E4M3 codes (bits 0..7, 8..15) -> two binary32 values, exactly
// (every E4M3 value is an FP16 value, and FP16 widens exactly).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t c) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  const uint16_t h_lo = (uint16_t)(h2 & 0xFFFFu), h_hi = (uint16_t)(h2 >> 16);
  float lo, hi;
  asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(h_lo));
  asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(h_hi));
  return make_float2(lo, hi);
}

// ---- per-group scale: S = RN32(amax / 448), S = 1 for an all-zero group ----
__device__ __forceinline__ float scale_from_amax(float amax) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// ---- power-of-two scale: the smallest S = 2^e with 448 S >= amax ----
// (the pages' "power-of-2 scaling factor" option, NeMo RL FP8 blog, section
// on recipe variants).  With amax = f 2^p, f in [0.5, 1), and 448 = 0.875 2^9:
// e = p - 9, plus one when f > 0.875.  x / S is then exact, so a code is the
// single rounding E4M3(x / S); S = 1 for an all-zero group.
__device__ __forceinline__ float scale_pow2_from_amax(float amax) {
  if (amax == 0.0f) return 1.0f;
  int p;
  const float f = frexpf(amax, &p);
  return ldexpf(1.0f, p - 9 + (f > 0.875f ? 1 : 0));
}

template <bool kPow2>
__device__ __forceinline__ float group_scale(float amax) {
  return kPow2 ? scale_pow2_from_amax(amax) : scale_from_amax(amax);
}

// ---- E4M3(RN32(x / S)), exactly, without a division per element ----
// The binary32 quotient RN32(x / S) is formed with Markstein's correction
// step (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990; see also
// Muller et al., "Handbook of Floating-Point Arithmetic", the section on
// division with a fused multiply-add): with r = RN32(1/S) and
// t = RN32(x r), the residual e = x - t S is exact when computed by one
// fused multiply-add, and q = RN32(t + e r) is the correctly rounded
// quotient as long as nothing overflows or underflows.  The hardware
// conversion of q then gives the E4M3 code.  Two values share each packed
// FP32x2 operation, so a pair costs three arithmetic instructions and one
// conversion, with no branch.  Scales outside [2^-100, 2^100], and scales
// given by a caller rather than derived from the data, take the correctly
// rounded division instead.  A GPU self-test compares this coding with the
// division on every (BF16 x, BF16 amax) pair the quantizers can see.
struct QuantScale {
  float s;      // S
  float r;      // RN32(1 / S)
  bool exact;   // use the division for every element
};

__device__ __forceinline__ QuantScale make_quant_scale(float s) {
  QuantScale q;
  q.s = s;
  q.r = __frcp_rn(s);
  q.exact = !(s >= 0x1p-100f && s <= 0x1p100f);
  return q;
}

// For a scale that does not come from the data's own amax (x / S may then
// overflow binary32): every element takes the division.
__device__ __forceinline__ QuantScale make_quant_scale_division(float s) {
  QuantScale q;
  q.s = s;
  q.r = 0.0f;
  q.exact = true;
  return q;
}

__device__ __forceinline__ uint32_t code_exact(float x, float s) {
  return cvt_e4m3x2(__fdiv_rn(x, s), 0.0f) & 0xFFu;
}

// Four codes by the correctly rounded division (out of line: the path of
// unusual scales only).
static __device__ __noinline__ uint32_t codes_by_division(float x0, float x1, float x2, float x3,
                                                   float s) {
  return code_exact(x0, s) | (code_exact(x1, s) << 8) | (code_exact(x2, s) << 16) |
         (code_exact(x3, s) << 24);
}

// Four codes (byte i = code of x_i) from four binary32 values, except for
// the sign of zero: an input of -0 yields +0 here (the residual of a zero
// quotient is +0), so the callers below OR the inputs' sign bits into the
// codes -- RN32(x / S) always has the sign of x, so that is exact.
__device__ __forceinline__ uint32_t quant_f32x4_unsigned_zero(float x0, float x1, float x2,
                                                              float x3, const QuantScale& qs) {
  if (qs.exact) return codes_by_division(x0, x1, x2, x3, qs.s);
  uint32_t c;
  asm("{\n\t.reg .b16 l0, l1;\n\t.reg .b64 a01, a23, rr, ns, t01, t23, e01, e23, q01, q23;\n\t"
      ".reg .f32 q0, q1, q2, q3;\n\t"
      "mov.b64 a01, {%1, %2};\n\tmov.b64 a23, {%3, %4};\n\t"
      "mov.b64 rr, {%5, %5};\n\tmov.b64 ns, {%6, %6};\n\t"
      "mul.rn.f32x2 t01, a01, rr;\n\tmul.rn.f32x2 t23, a23, rr;\n\t"
      "fma.rn.f32x2 e01, t01, ns, a01;\n\tfma.rn.f32x2 e23, t23, ns, a23;\n\t"
      "fma.rn.f32x2 q01, e01, rr, t01;\n\tfma.rn.f32x2 q23, e23, rr, t23;\n\t"
      "mov.b64 {q0, q1}, q01;\n\tmov.b64 {q2, q3}, q23;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l0, q1, q0;\n\tcvt.rn.satfinite.e4m3x2.f32 l1, q3, q2;\n\t"
      "mov.b32 %0, {l0, l1};\n\t}"
      : "=r"(c)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3), "f"(qs.r), "f"(-qs.s));
  return c;
}

// Four codes (byte i = code of x_i) from four binary32 values.
__device__ __forceinline__ uint32_t quant_f32x4(float x0, float x1, float x2, float x3,
                                                const QuantScale& qs) {
  const uint32_t c = quant_f32x4_unsigned_zero(x0, x1, x2, x3, qs);
  const uint32_t s01 = __byte_perm(__float_as_uint(x0), __float_as_uint(x1), 0x0073);
  const uint32_t s23 = __byte_perm(__float_as_uint(x2), __float_as_uint(x3), 0x0073);
  return c | (__byte_perm(s01, s23, 0x5410) & 0x80808080u);
}

// Four codes from two BF16x2 words, packed little-endian into 32 bits (the
// sign bits come straight from the words: bytes 1 and 3 of each).
__device__ __forceinline__ uint32_t quant_bf16x4(uint32_t w0, uint32_t w1, const QuantScale& qs) {
  const uint32_t c =
      quant_f32x4_unsigned_zero(bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1), qs);
  return c | (__byte_perm(w0, w1, 0x7531) & 0x80808080u);
}

// One code (the scalar path of ragged rows and tails).
__device__ __forceinline__ uint32_t quant_one(float x, const QuantScale& qs) {
  return quant_f32x4(x, 0.0f, 0.0f, 0.0f, qs) & 0xFFu;
}

// Running max of |x| over the BF16 halves of a word, kept as a BF16x2 whose
// two halves are reduced at the end (max is exact in any precision).
__device__ __forceinline__ uint32_t absmax_bf16x2_packed(uint32_t m, uint32_t w) {
  uint32_t r;
  const uint32_t a = w & 0x7FFF7FFFu;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(a));
  return r;
}
__device__ __forceinline__ float absmax_finish(uint32_t m) {
  return fmaxf(bf16_lo(m), bf16_hi(m));
}

// max |x| over N x 8 BF16 values as four independent max chains.  The
// running values keep max(|m|, |w|) as magnitude (max.xorsign.abs: the sign
// bit is a by-product and is cleared once at the end).
template <int N>
__device__ __forceinline__ float absmax_bf16x8_tree(const uint4 (&v)[N]) {
  uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m0) : "r"(v[i].x));
    asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m1) : "r"(v[i].y));
    asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(v[i].z));
    asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m3) : "r"(v[i].w));
  }
  asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m0) : "r"(m1));
  asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(m3));
  asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m0) : "r"(m2));
  return absmax_finish(m0 & 0x7FFF7FFFu);
}

// ---- dequantization: RN32(dec(code) * S), then BF16 round to nearest even ----
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two codes (bits 0..7, 8..15) times S, rounded once to binary32 each, then
// to BF16: the BF16 pair for output positions (lo, hi).
__device__ __forceinline__ uint32_t dequant_pair(uint32_t codes16, float S) {
  const float2 d = e4m3x2_to_float2((uint16_t)codes16);
  return pack_bf16x2_rn(__fmul_rn(d.x, S), __fmul_rn(d.y, S));
}

// ---- cache-hinted vector access for data touched once ----
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream_v2(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

}  // namespace w8a8
