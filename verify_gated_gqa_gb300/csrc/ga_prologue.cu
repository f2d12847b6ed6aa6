// Prologue: (1+w) RMSNorm and partial RoPE of head rows, once per row (pegainfer PR
// #1151, "feat(qwen4): add the QSA sparse-attention kernel and its golden", §What changed:
// all twelve query heads of a KV head read the same prepared key; the query rows take
// the same norm with w_q at their own positions).
//
// One warp per (token, head) row of 256 bf16: lane l holds dims 8l .. 8l+7 (one 16-byte
// load and store, so a warp reads and writes 512 contiguous bytes). Memory-bound. Keys:
// [T][2][256] -> [T][2][256]. Queries: the q halves of the fused rows [rows][24][512] ->
// [rows][24][256].
#include "ga_internal.h"
#include "ga_numerics.cuh"
#include "ga_sm100.cuh"

namespace ga {
namespace {

__device__ __forceinline__ float lo_f(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hi_f(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return (uint32_t)bf16_bits(a) | ((uint32_t)bf16_bits(b) << 16);
}

// rows are (token, head) pairs, heads_per_tok heads per token; row `row` reads 256 values
// at src + row * src_stride and writes 256 at dst + row * 256. Token t sits at position
// pos_base + t, or, with kSeq, at sp.seq_base[t / sp.rows_per_seq] + t % sp.rows_per_seq.
template <bool kSeq>
__global__ void __launch_bounds__(256) prologue_kernel(const uint16_t* __restrict__ src,
                                                       int src_stride, int heads_per_tok,
                                                       const uint16_t* __restrict__ w_norm,
                                                       const uint16_t* __restrict__ cos_tab,
                                                       const uint16_t* __restrict__ sin_tab,
                                                       long long n_rows, int pos_base,
                                                       const __grid_constant__ SeqPositions sp,
                                                       uint16_t* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const long long tok = row / heads_per_tok;
  const int pos = kSeq ? sp.seq_base[tok / sp.rows_per_seq] + (int)(tok % sp.rows_per_seq)
                       : pos_base + (int)tok;

  const uint4 xv = __ldg(reinterpret_cast<const uint4*>(src + row * src_stride) + lane);
  const uint4 wv = __ldg(reinterpret_cast<const uint4*>(w_norm) + lane);
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
  float x[8], w[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = lo_f(xw[i]);
    x[2 * i + 1] = hi_f(xw[i]);
    w[2 * i] = lo_f(ww[i]);
    w[2 * i + 1] = hi_f(ww[i]);
  }
  SumSq ss;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss.add(x[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    SumSq o;
    o.hi = __shfl_xor_sync(0xffffffffu, ss.hi, off);
    o.lo = __shfl_xor_sync(0xffffffffu, ss.lo, off);
    // merge in a fixed order (lower lane first) so every lane holds the same pair
    if (lane & off) {
      SumSq t = o;
      t.merge(ss);
      ss = t;
    } else {
      ss.merge(o);
    }
  }
  const InvRms r = inv_rms_df(ss);
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = norm_elem(x[i], w[i], r);

  // Partial RoPE: dims 0..31 (lanes 0..3) pair with dims 32..63 (lanes 4..7).
  float partner[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) partner[i] = __shfl_xor_sync(0xffffffffu, y[i], 4);
  if (lane < 8) {
    const int pair0 = (lane & 3) * 8;  // pair index of this lane's first dim
    const uint4 cv = __ldg(reinterpret_cast<const uint4*>(cos_tab + (long long)pos * kHalfRot + pair0));
    const uint4 sv = __ldg(reinterpret_cast<const uint4*>(sin_tab + (long long)pos * kHalfRot + pair0));
    const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
    const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float c = (i & 1) ? hi_f(cw[i >> 1]) : lo_f(cw[i >> 1]);
      const float s = (i & 1) ? hi_f(sw[i >> 1]) : lo_f(sw[i >> 1]);
      float ya, yb;
      if (lane < 4) {
        rope_pair(y[i], partner[i], c, s, ya, yb);
        y[i] = ya;
      } else {
        rope_pair(partner[i], y[i], c, s, ya, yb);
        y[i] = yb;
      }
    }
  }
  uint4 o;
  o.x = pack2(y[0], y[1]);
  o.y = pack2(y[2], y[3]);
  o.z = pack2(y[4], y[5]);
  o.w = pack2(y[6], y[7]);
  reinterpret_cast<uint4*>(dst + row * kDim)[lane] = o;
}

}  // namespace

cudaError_t launch_k_prologue(const uint16_t* k_raw, const uint16_t* w_k, const uint16_t* cos_tab,
                              const uint16_t* sin_tab, int n_tok, int pos_base, uint16_t* k_prep,
                              int* status, cudaStream_t s) {
  (void)status;
  const long long n_rows = (long long)n_tok * kKvHeads;
  const unsigned grid = (unsigned)((n_rows + 7) / 8);
  prologue_kernel<false><<<grid, 256, 0, s>>>(k_raw, kDim, kKvHeads, w_k, cos_tab, sin_tab,
                                              n_rows, pos_base, SeqPositions{}, k_prep);
  return cudaGetLastError();
}

cudaError_t launch_q_prologue(const uint16_t* qg, const uint16_t* w_q, const uint16_t* cos_tab,
                              const uint16_t* sin_tab, int rows, int q_base, uint16_t* q_prep,
                              cudaStream_t s) {
  const long long n_rows = (long long)rows * kHeads;
  const unsigned grid = (unsigned)((n_rows + 7) / 8);
  prologue_kernel<false><<<grid, 256, 0, s>>>(qg, kQgStride, kHeads, w_q, cos_tab, sin_tab,
                                              n_rows, q_base, SeqPositions{}, q_prep);
  return cudaGetLastError();
}

cudaError_t launch_q_prologue_seq(const uint16_t* qg, const uint16_t* w_q, const uint16_t* cos_tab,
                                  const uint16_t* sin_tab, int n_tok, const SeqPositions& sp,
                                  uint16_t* q_prep, cudaStream_t s) {
  const long long n_rows = (long long)n_tok * kHeads;
  const unsigned grid = (unsigned)((n_rows + 7) / 8);
  prologue_kernel<true><<<grid, 256, 0, s>>>(qg, kQgStride, kHeads, w_q, cos_tab, sin_tab, n_rows,
                                             0, sp, q_prep);
  return cudaGetLastError();
}

}  // namespace ga
