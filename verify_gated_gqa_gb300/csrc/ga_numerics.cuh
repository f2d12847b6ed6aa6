// Rounding-exact device numerics for the prologue and gate work of the attention path.
//
// The method rounds to bf16 at fixed points (pegainfer PR #1151, the commit that adds the
// attention reader: the norms cast once, cos/sin bf16 with the rotation rounding in
// bf16, the sigmoid rounded before the final product). The reference values are defined
// in double precision. These helpers compute in fp32 only (FP64 is slow on this part)
// and certify the bf16 rounding: an fp32 result whose error bound keeps it away from a
// bf16 rounding midpoint rounds to the same bf16 value as the exact result; the rare
// element closer than the bound to a midpoint takes an exact path (a double-float
// product for the norm, a table of every bf16 input for the sigmoid).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace ga {

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}
__device__ __forceinline__ uint16_t bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// True when y's lower 16 bits lie within `margin` of 0x8000 (a bf16 rounding midpoint).
__device__ __forceinline__ bool near_bf16_midpoint(float y, int margin) {
  const int lo = (int)(__float_as_uint(y) & 0xFFFFu) - 0x8000;
  return lo <= margin && lo >= -margin;
}

// Knuth's TwoSum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Sum of squares kept as an unevaluated pair hi + lo (error about 2^-40 relative). The
// squares of bf16 values are exact in fp32; TwoSum captures each addition's error.
struct SumSq {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add(float x) {
    float s, e;
    two_sum(hi, x * x, s, e);
    hi = s;
    lo += e;
  }
  __device__ __forceinline__ void merge(const SumSq& o) {
    float s, e;
    two_sum(hi, o.hi, s, e);
    hi = s;
    lo += o.lo + e;
  }
};

// The row's inverse RMS, 1 / sqrt(sum / 256 + 1e-6), as h + l good to about 2^-40
// relative (the sum's own error). From rsqrt's estimate r0, one Newton step carried in
// double-float: with a r0^2 = 1 - e (e about 2^-22, formed exactly up to 2^-46),
// r = r0 (1 + e/2 + 3e^2/8).
struct InvRms {
  float h, l;
};
__device__ __forceinline__ InvRms inv_rms_df(const SumSq& s) {
  constexpr float kEpsHi = 1e-6f;
  constexpr float kEpsLo = 2.5247573e-15f;  // 1e-6 - kEpsHi
  float ah, al;
  two_sum(s.hi * (1.0f / 256.0f), kEpsHi, ah, al);
  al += s.lo * (1.0f / 256.0f) + kEpsLo;
  const float r0 = rsqrtf(ah);
  const float sq = r0 * r0;
  const float sqe = fmaf(r0, r0, -sq);          // r0^2 = sq + sqe exactly
  const float th = ah * sq;
  float te = fmaf(ah, sq, -th);                 // ah sq = th + te exactly
  te = fmaf(ah, sqe, te);
  te = fmaf(al, sq, te);
  const float e = (1.0f - th) - te;             // 1 - th is exact (th within 2^-20 of 1)
  InvRms r;
  r.h = r0;
  r.l = r0 * fmaf(0.375f * e, e, 0.5f * e);
  return r;
}

// Norm of one element, exact: y = bf16(x (1 + w) r) with r = rh + rl. x w is exact in fp32
// (8 x 8 significant bits) and TwoSum makes x + x w exact; the product with rh + rl is
// carried as an unevaluated sum, renormalised to s + t with |t| <= half an ulp of s. An s
// that is not a bf16 midpoint rounds like s + t (a midpoint is at least one ulp away); an
// s on a midpoint is nudged one ulp toward t before the rounding.
__device__ __forceinline__ float norm_elem_exact(float x, float w, float rh, float rl) {
  const float xw = x * w;
  float ph, pl;
  two_sum(x, xw, ph, pl);
  const float yh = ph * rh;
  const float yl = fmaf(ph, rh, -yh) + fmaf(ph, rl, pl * rh);
  const float s = yh + yl;
  const float t = yl - (s - yh);
  uint32_t u = __float_as_uint(s);
  if ((u & 0xFFFFu) == 0x8000u && t != 0.0f) u += ((t > 0.0f) == (s > 0.0f)) ? 1u : 0xFFFFFFFFu;
  return bf16_round(__uint_as_float(u));
}

// Norm of one element, fast path: (x (1 + w)) r as fma(x, w, x) then fma(p, rh, p rl): two
// roundings of at most half an ulp (plus about 2^-40), so the result is within 2 fp32
// ulps of the exact value and rounds to the exact bf16 unless it lies within 2 ulps of a
// bf16 midpoint. norm_elem returns the exact bf16 value either way.
__device__ __forceinline__ float norm_fast(float x, float w, InvRms r) {
  const float p = fmaf(x, w, x);
  return fmaf(p, r.h, p * r.l);
}
__device__ __forceinline__ float norm_elem(float x, float w, InvRms r) {
  const float y = norm_fast(x, w, r);
  if (!near_bf16_midpoint(y, 3)) return bf16_round(y);
  return norm_elem_exact(x, w, r.h, r.l);
}

// Two e4m3 codes (low byte first) as floats; every e4m3 value is exact in f16 and f32.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  const __half2_raw hr =
      __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xFFFFu), __NV_E4M3);
  return __half22float2(__half2(hr));
}

// Rotate-half RoPE of one pair with bf16 rounding after each product and after the sum;
// every step is exact in fp32 before its rounding, so this is the definition itself.
__device__ __forceinline__ void rope_pair(float a, float b, float c, float s, float& ya,
                                          float& yb) {
  ya = bf16_round(bf16_round(a * c) - bf16_round(b * s));
  yb = bf16_round(bf16_round(b * c) + bf16_round(a * s));
}

}  // namespace ga
