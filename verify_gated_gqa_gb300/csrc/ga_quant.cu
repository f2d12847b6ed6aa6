// e4m3 cache rows with one fp32 scale each (TensorFold PR #1080, "qwen CUDA: long-prompt
// prefill 5.4x faster", the prompt-chain commit: e4m3 cache rows with an fp32 scale each,
// widened to bf16 in the slot; the rope-kernel commit: the e4m3 scales come from
// reductions over the row). For each (token, head) row of 256 bf16 values:
//   sc = fp32(max|x| / 448),  q = e4m3(fp32(x / sc))  (nearest, ties to even, saturating),
// a zero row giving sc = 0 and q = 0. Both divisions are IEEE divisions rounded to nearest.
//
// Eight lanes per row, four rows per warp; lane j holds dims 32k + 4j .. +3 (k = 0..7), as in
// the prologue, so the row maximum reduces over the row's 8 lanes in three shuffle steps.
// The inverse, widening rows back to bf16(fp32(code * scale)), serves prefill over e4m3
// caches: prefill reads every key tile once per row tile, so its rows are widened once in
// HBM rather than at every visit.
#include <cuda_fp8.h>

#include "ga_internal.h"
#include "ga_numerics.cuh"
#include "ga_sm100.cuh"

namespace ga {
namespace {

constexpr int kRowsPerBlock = 32;   // 8 warps x 4 rows
constexpr float kE4m3Max = 448.0f;

__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const uint16_t* __restrict__ x,
                                                            long long n_rows,
                                                            uint8_t* __restrict__ q,
                                                            float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int j = lane & 7;
  const long long row = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 3);
  if (row >= n_rows) return;   // whole row groups leave together
  const unsigned gmask = 0xFFu << (lane & 24);
  const uint2* xs = reinterpret_cast<const uint2*>(x + row * kDim) + j;
  uint2 xv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) xv[k] = __ldg(xs + 8 * k);
  auto val = [](uint32_t w, int hi) {
    return __uint_as_float(hi ? (w & 0xFFFF0000u) : (w << 16));
  };
  float a = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    a = fmaxf(fmaxf(fmaxf(a, fabsf(val(xv[k].x, 0))), fabsf(val(xv[k].x, 1))),
              fmaxf(fabsf(val(xv[k].y, 0)), fabsf(val(xv[k].y, 1))));
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) a = fmaxf(a, __shfl_xor_sync(gmask, a, off, 8));
  const float sc = __fdiv_rn(a, kE4m3Max);
  uint32_t* qo = reinterpret_cast<uint32_t*>(q + row * kDim) + j;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint32_t packed = 0;
    if (sc > 0.f) {
      const float v0 = __fdiv_rn(val(xv[k].x, 0), sc), v1 = __fdiv_rn(val(xv[k].x, 1), sc);
      const float v2 = __fdiv_rn(val(xv[k].y, 0), sc), v3 = __fdiv_rn(val(xv[k].y, 1), sc);
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v2, v3), __NV_SATFINITE, __NV_E4M3);
      packed = (lo & 0xFFFFu) | (hi << 16);
    }
    qo[8 * k] = packed;   // bytes of dims 32k + 4j .. +3, lowest dim first
  }
  if (j == 0) scale[row] = sc;
}

// The widened rows: bf16(fp32(code * scale)) per element, the value the attention reads
// from an e4m3 cache row. One thread per 8 codes (an 8-byte load, a 16-byte store); the 32
// threads of a row share its scale.
__global__ void __launch_bounds__(256) dequantize_e4m3_kernel(const uint8_t* __restrict__ q,
                                                              const float* __restrict__ scale,
                                                              long long n_rows,
                                                              uint16_t* __restrict__ out) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_rows * (kDim / 8)) return;
  const float sc = __ldg(scale + i / (kDim / 8));
  const uint2 c = __ldg(reinterpret_cast<const uint2*>(q) + i);
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = e4m3x2_to_float2((k < 2 ? c.x : c.y) >> (16 * (k & 1)));
    w[k] = pack_bf16x2(f.x * sc, f.y * sc);
  }
  reinterpret_cast<uint4*>(out)[i] = make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

cudaError_t launch_dequantize_e4m3(const uint8_t* q, const float* scale, long long n_rows,
                                   uint16_t* out, cudaStream_t s) {
  const long long n = n_rows * (kDim / 8);
  dequantize_e4m3_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(q, scale, n_rows, out);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const uint16_t* x, long long n_rows, uint8_t* q, float* scale,
                                 cudaStream_t s) {
  const unsigned grid = (unsigned)((n_rows + kRowsPerBlock - 1) / kRowsPerBlock);
  quantize_e4m3_kernel<<<grid, 256, 0, s>>>(x, n_rows, q, scale);
  return cudaGetLastError();
}

}  // namespace ga
