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

// ---- E4M3(RN32(x / S)), exactly, without a division per element ----
// Let q = x / S (exact real), r = RN32(1/S), r_dn = RN32(r (1 - 2^-21)) and
// r_up = RN32(r (1 + 2^-21)).  Each of r, r_dn/r_up and the products
// t_dn = RN32(x r_dn), t_up = RN32(x r_up) adds one relative error of at
// most 2^-24, so for binary32-normal q
//     t_dn <= q (1 - 5 * 2^-24) < RN32(q) < q (1 + 5 * 2^-24) <= t_up
// (mirrored for q < 0): the two products bracket RN32(x / S).  E4M3 coding
// with round-to-nearest and saturation is monotone, so when t_dn and t_up
// get the same code, RN32(x / S) gets that code too.  (When q is a
// binary32 subnormal every candidate codes to a zero of the right sign.)
// When the codes differ -- the bracket straddles an E4M3 rounding midpoint,
// about 1 element in 60000 for normal-range values -- that element is
// recomputed with the correctly rounded division.  If r_up overflows, every
// element of the group takes the division.
struct QuantScale {
  float s;     // S
  float r_dn;  // RN32(RN32(1/S) * (1 - 2^-21))
  float r_up;  // RN32(RN32(1/S) * (1 + 2^-21))
  bool exact;  // bracket unavailable: use the division for every element
};

__device__ __forceinline__ QuantScale make_quant_scale(float s) {
  QuantScale q;
  q.s = s;
  const float r = __frcp_rn(s);
  q.r_dn = __fmul_rn(r, 1.0f - 0x1p-21f);
  q.r_up = __fmul_rn(r, 1.0f + 0x1p-21f);
  q.exact = !(q.r_up <= 3.0e38f);
  return q;
}

__device__ __forceinline__ uint32_t code_exact(float x, float s) {
  return cvt_e4m3x2(__fdiv_rn(x, s), 0.0f) & 0xFFu;
}

// The rare path, kept out of line so the hot loops stay small in the
// instruction cache: recompute with the division the bytes of `codes` whose
// bits are set in `diff`.
__device__ __noinline__ uint32_t fix_codes_exact(uint32_t codes, uint32_t diff, float x0, float x1,
                                                 float x2, float x3, float s) {
  if (diff & 0x000000FFu) codes = (codes & 0xFFFFFF00u) | code_exact(x0, s);
  if (diff & 0x0000FF00u) codes = (codes & 0xFFFF00FFu) | (code_exact(x1, s) << 8);
  if (diff & 0x00FF0000u) codes = (codes & 0xFF00FFFFu) | (code_exact(x2, s) << 16);
  if (diff & 0xFF000000u) codes = (codes & 0x00FFFFFFu) | (code_exact(x3, s) << 24);
  return codes;
}

// Four codes (byte i = code of x_i) from four binary32 values.  The two
// products per value (packed FP32x2 multiplies), the four conversions and the
// byte packing are one PTX block: t_dn codes come out as one 32-bit word and
// t_up codes as another, compared with a single test.
__device__ __forceinline__ uint32_t quant_f32x4(float x0, float x1, float x2, float x3,
                                                const QuantScale& qs) {
  if (qs.exact) return fix_codes_exact(0u, 0xFFFFFFFFu, x0, x1, x2, x3, qs.s);
  uint32_t dn, up;
  asm("{\n\t.reg .b16 l0, l1, h0, h1;\n\t.reg .b64 a01, a23, rd, ru, d01, d23, u01, u23;\n\t"
      ".reg .f32 d0, d1, d2, d3, u0, u1, u2, u3;\n\t"
      "mov.b64 a01, {%2, %3};\n\tmov.b64 a23, {%4, %5};\n\tmov.b64 rd, {%6, %6};\n\tmov.b64 ru, {%7, %7};\n\t"
      "mul.rn.f32x2 d01, a01, rd;\n\tmul.rn.f32x2 d23, a23, rd;\n\tmul.rn.f32x2 u01, a01, ru;\n\tmul.rn.f32x2 u23, a23, ru;\n\t"
      "mov.b64 {d0, d1}, d01;\n\tmov.b64 {d2, d3}, d23;\n\tmov.b64 {u0, u1}, u01;\n\tmov.b64 {u2, u3}, u23;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l0, d1, d0;\n\tcvt.rn.satfinite.e4m3x2.f32 l1, d3, d2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h0, u1, u0;\n\tcvt.rn.satfinite.e4m3x2.f32 h1, u3, u2;\n\t"
      "mov.b32 %0, {l0, l1};\n\tmov.b32 %1, {h0, h1};\n\t}"
      : "=r"(dn), "=r"(up)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3), "f"(qs.r_dn), "f"(qs.r_up));
  if (__builtin_expect(dn != up, 0)) return fix_codes_exact(dn, dn ^ up, x0, x1, x2, x3, qs.s);
  return dn;
}

// Four codes from two BF16x2 words, packed little-endian into 32 bits.
__device__ __forceinline__ uint32_t quant_bf16x4(uint32_t w0, uint32_t w1, const QuantScale& qs) {
  return quant_f32x4(bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1), qs);
}

// The bracketed coding of four values without the fallback branch: returns
// the t_dn codes and sets `diff` to the bytes whose t_up code differs.
__device__ __forceinline__ uint32_t quant_f32x4_fast(float x0, float x1, float x2, float x3,
                                                     const QuantScale& qs, uint32_t& diff) {
  uint32_t dn, up;
  asm("{\n\t.reg .b16 l0, l1, h0, h1;\n\t.reg .b64 a01, a23, rd, ru, d01, d23, u01, u23;\n\t"
      ".reg .f32 d0, d1, d2, d3, u0, u1, u2, u3;\n\t"
      "mov.b64 a01, {%2, %3};\n\tmov.b64 a23, {%4, %5};\n\tmov.b64 rd, {%6, %6};\n\tmov.b64 ru, {%7, %7};\n\t"
      "mul.rn.f32x2 d01, a01, rd;\n\tmul.rn.f32x2 d23, a23, rd;\n\tmul.rn.f32x2 u01, a01, ru;\n\tmul.rn.f32x2 u23, a23, ru;\n\t"
      "mov.b64 {d0, d1}, d01;\n\tmov.b64 {d2, d3}, d23;\n\tmov.b64 {u0, u1}, u01;\n\tmov.b64 {u2, u3}, u23;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l0, d1, d0;\n\tcvt.rn.satfinite.e4m3x2.f32 l1, d3, d2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h0, u1, u0;\n\tcvt.rn.satfinite.e4m3x2.f32 h1, u3, u2;\n\t"
      "mov.b32 %0, {l0, l1};\n\tmov.b32 %1, {h0, h1};\n\t}"
      : "=r"(dn), "=r"(up)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3), "f"(qs.r_dn), "f"(qs.r_up));
  diff = dn ^ up;
  return dn;
}

// Eight codes from one 16-byte word of eight BF16 values, with a single
// (rarely taken) branch to the exact fallback.
__device__ __forceinline__ uint2 quant_bf16x8(const uint4& v, const QuantScale& qs) {
  const float x0 = bf16_lo(v.x), x1 = bf16_hi(v.x), x2 = bf16_lo(v.y), x3 = bf16_hi(v.y);
  const float x4 = bf16_lo(v.z), x5 = bf16_hi(v.z), x6 = bf16_lo(v.w), x7 = bf16_hi(v.w);
  uint2 c;
  if (qs.exact) {
    c.x = fix_codes_exact(0u, 0xFFFFFFFFu, x0, x1, x2, x3, qs.s);
    c.y = fix_codes_exact(0u, 0xFFFFFFFFu, x4, x5, x6, x7, qs.s);
    return c;
  }
  uint32_t d0, d1;
  c.x = quant_f32x4_fast(x0, x1, x2, x3, qs, d0);
  c.y = quant_f32x4_fast(x4, x5, x6, x7, qs, d1);
  if (__builtin_expect((d0 | d1) != 0u, 0)) {
    if (d0) c.x = fix_codes_exact(c.x, d0, x0, x1, x2, x3, qs.s);
    if (d1) c.y = fix_codes_exact(c.y, d1, x4, x5, x6, x7, qs.s);
  }
  return c;
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
