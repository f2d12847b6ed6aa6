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

__device__ __forceinline__ bool near_bf16_midpoint(float y, int margin = kMidMargin) {
  const int lo = (int)(__float_as_uint(y) & 0xFFFFu) - 0x8000;
  return lo <= margin && lo >= -margin;
}

// bf16 (nearest, ties to even) of a finite double within bf16's range, as a float. Below
// 2^-126 bf16 is subnormal, a multiple of 2^-133.
__device__ __forceinline__ float bf16_of_double(double x) {
  if (fabs(x) < 0x1p-126) return (float)(rint(x * 0x1p133) * 0x1p-133);
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

// Fast path of norm_elem: the fp32 value before its bf16 rounding. When
// near_bf16_midpoint() of it holds, the element needs norm_elem_slow.
__device__ __forceinline__ float norm_elem_f32(float x, float w, float r32) {
  return (x * r32) * (1.0f + w);
}
// Fast sigmoid of a bf16 g for the epilogue: 1 / (1 + 2^(-g log2 e)) with the exponent
// split exactly (g has 8 significant bits, kL2eHi 16, so -g * kL2eHi is exact in fp32; the
// small remainder -g * kL2eLo is applied as a first-order factor), ex2.approx and
// rcp.approx. Over every bf16 g whose sigmoid is a normal fp32 number the result is within
// a few fp32 ulps (checked exhaustively on the device against the double definition); the
// caller rounds it to bf16 unless it lies within kSigmoidMargin ulps of a bf16 midpoint,
// or g is outside that range, and then sigmoid_slow is the answer: returns false for those.
// Where 2^-g*log2e is below 2^-32 the sum 1 + e is exactly 1 and so is the bf16 result.
constexpr int kSigmoidMargin = 12;
constexpr float kL2eHi = 1.44268798828125f;          // 47274 / 2^15: log2(e) to 16 bits
constexpr float kL2eLo = 7.05260771340736e-06f;      // log2(e) - kL2eHi
__device__ __forceinline__ bool sigmoid_fast(float g, float& y) {
  const float th = -g * kL2eHi;
  // the remainder from a clamped g, so that an infinite g gives 0 * finite, not 0 * inf
  // (a NaN g still gives NaN through th)
  const float tl = -fminf(fmaxf(g, -256.0f), 256.0f) * kL2eLo;
  float e0, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(th));
  const float e = fmaf(e0, tl * 0.6931471805599453f, e0);
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  y = r;
  return th <= 120.0f && !near_bf16_midpoint(r, kSigmoidMargin);
}

// Norm of one element with a double-float product, good to about 2^-46 relative: y =
// bf16(x * (1 + w) * r64), where r64 = rh + rl is the row's double inverse RMS. x * w is
// exact in fp32 (8 x 8 significant bits) and TwoSum makes x + x*w exact; the product with
// rh + rl is carried as an unevaluated sum, renormalised to s + t with |t| <= half an
// ulp of s. An s that is not a bf16 midpoint rounds like s + t (a midpoint is at least
// one ulp away); an s on a midpoint is nudged one ulp toward t before the rounding.
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
