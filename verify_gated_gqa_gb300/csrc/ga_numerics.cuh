// Rounding-exact device numerics for the prologue work of the attention path.
//
// The method rounds to bf16 at fixed points (pegainfer PR #1151, the commit that adds the
// attention reader: the norms cast once, cos/sin bf16 with the rotation rounding in
// bf16, the sigmoid rounded before the final product). The reference values are defined
// in double precision. These helpers compute in fp32 and certify the bf16 rounding: an
// fp32 result whose error bound keeps it away from a bf16 rounding midpoint rounds to
// the same bf16 value as the double result; the rare element closer than the bound to
// a midpoint is recomputed with the same double operations the definition uses.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace ga {

// fp32 results whose error is at most 4 fp32 ulps are certified when they sit more than
// kMidMargin fp32 ulps away from a bf16 midpoint (the lower 16 bits equal 0x8000 there).
constexpr int kMidMargin = 8;

__device__ __forceinline__ bool near_bf16_midpoint(float y) {
  const int lo = (int)(__float_as_uint(y) & 0xFFFFu) - 0x8000;
  return lo <= kMidMargin && lo >= -kMidMargin;
}

// bf16 (nearest, ties to even) of a finite double in bf16's normal range, as a float.
__device__ __forceinline__ float bf16_of_double(double x) {
  unsigned long long u = (unsigned long long)__double_as_longlong(x);
  u += 0x00000FFFFFFFFFFFull + ((u >> 45) & 1ull);
  u &= ~0x00001FFFFFFFFFFFull;
  return (float)__longlong_as_double((long long)u);
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}
__device__ __forceinline__ uint16_t bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
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

// Inverse RMS: fp32 value (<= 2.5 ulp error) and the double value the definition uses,
// 1 / sqrt(sum / 256 + eps) in double.
__device__ __forceinline__ float inv_rms_f32(const SumSq& s) {
  return 1.0f / sqrtf((s.hi + s.lo) * (1.0f / 256.0f) + 1e-6f);
}
__device__ __forceinline__ double inv_rms_f64(const SumSq& s) {
  return 1.0 / sqrt(((double)s.hi + (double)s.lo) / 256.0 + 1e-6);
}

// Out-of-line double-precision recomputation (rare): kept out of the hot loops so that
// they stay small.
static __device__ __noinline__ float norm_elem_slow(float x, float w, float hi, float lo) {
  SumSq ss;
  ss.hi = hi;
  ss.lo = lo;
  return bf16_of_double(((double)x * inv_rms_f64(ss)) * (1.0 + (double)w));
}
static __device__ __noinline__ float sigmoid_slow(float g) {
  return bf16_of_double(1.0 / (1.0 + exp(-(double)g)));
}

// bf16 of x * inv_rms * (1 + w) for a bf16 x and a bf16 weight w.
__device__ __forceinline__ float norm_elem(float x, float w, float r32, const SumSq& ss) {
  const float y = (x * r32) * (1.0f + w);
  if (!near_bf16_midpoint(y)) return bf16_round(y);
  return norm_elem_slow(x, w, ss.hi, ss.lo);
}

// Rotate-half RoPE of one pair with bf16 rounding after each product and after the sum;
// every step is exact in fp32 before its rounding, so this is the definition itself.
__device__ __forceinline__ void rope_pair(float a, float b, float c, float s, float& ya,
                                          float& yb) {
  ya = bf16_round(bf16_round(a * c) - bf16_round(b * s));
  yb = bf16_round(bf16_round(b * c) + bf16_round(a * s));
}

// bf16(sigmoid(g)) = bf16(1 / (1 + e^-g)); fp32 error <= 3 ulps (expf is within 2 ulps).
__device__ __forceinline__ float sigmoid_bf16(float g) {
  const float y = 1.0f / (1.0f + expf(-g));
  if (!near_bf16_midpoint(y)) return bf16_round(y);
  return sigmoid_slow(g);
}

}  // namespace ga
