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

// ---- E4M3(RN32(x / S)) for two elements ----
// The quotient is needed only as far as its E4M3 code.  t = RN32(x * r) with
// r = RN32(1/S) lies within 2.5 binary32 ulps of RN32(x / S) (two relative
// rounding errors of 2^-24 plus half an ulp).  Coding is monotone, so when
// t - 8 ulps and t + 8 ulps get the same code, every value between them --
// RN32(x / S) included -- gets that code too.  Otherwise (t within 8 ulps of
// an E4M3 rounding midpoint: about 1 element in 60000) the element is
// recomputed with the correctly rounded division.  Magnitudes step by bit
// patterns; a pattern that runs past the binary32 range becomes NaN, whose
// code differs, so such elements also take the exact path.
struct QuantScale {
  float s;     // S
  float r;     // RN32(1 / S)
  bool exact;  // 1/S overflows: use the division for every element
};

__device__ __forceinline__ QuantScale make_quant_scale(float s) {
  QuantScale q;
  q.s = s;
  q.r = __frcp_rn(s);
  q.exact = !(q.r <= 3.0e38f);
  return q;
}

__device__ __forceinline__ uint32_t quant_pair(float x0, float x1, const QuantScale& qs) {
  if (qs.exact) return cvt_e4m3x2(__fdiv_rn(x0, qs.s), __fdiv_rn(x1, qs.s));
  const float t0 = __fmul_rn(x0, qs.r), t1 = __fmul_rn(x1, qs.r);
  uint32_t c = cvt_e4m3x2(t0, t1);
  const uint32_t a0 = __float_as_uint(t0) & 0x7FFFFFFFu;
  const uint32_t a1 = __float_as_uint(t1) & 0x7FFFFFFFu;
  const uint32_t clo = cvt_e4m3x2(__uint_as_float(a0 > 8u ? a0 - 8u : 0u),
                                  __uint_as_float(a1 > 8u ? a1 - 8u : 0u));
  const uint32_t chi = cvt_e4m3x2(__uint_as_float(a0 + 8u), __uint_as_float(a1 + 8u));
  const uint32_t diff = clo ^ chi;
  if (__builtin_expect(diff != 0u, 0)) {
    if (diff & 0x00FFu) c = (c & 0xFF00u) | (cvt_e4m3x2(__fdiv_rn(x0, qs.s), 0.0f) & 0x00FFu);
    if (diff & 0xFF00u) c = (c & 0x00FFu) | (cvt_e4m3x2(0.0f, __fdiv_rn(x1, qs.s)) & 0xFF00u);
  }
  return c;
}

// Four codes from two BF16x2 words, packed little-endian into 32 bits.
__device__ __forceinline__ uint32_t quant_bf16x4(uint32_t w0, uint32_t w1, const QuantScale& qs) {
  const uint32_t c0 = quant_pair(bf16_lo(w0), bf16_hi(w0), qs);
  const uint32_t c1 = quant_pair(bf16_lo(w1), bf16_hi(w1), qs);
  return c0 | (c1 << 16);
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
