// Prologue: (1+w) RMSNorm and partial RoPE of head rows, once per row (pegainfer PR
// #1151, "feat(qwen4): add the QSA sparse-attention kernel and its golden", §What changed:
// all twelve query heads of a KV head read the same prepared key; the query rows take
// the same norm with w_q at their own positions).
//
// Eight lanes per (token, head) row of 256 bf16, four rows per warp. Lane j of a row holds
// dims 32k + 4j .. 32k + 4j + 3 for k = 0..7 (eight 8-byte loads and stores; the eight
// lanes of a row read 64 contiguous bytes per k). The rotated pairs (d, d + 32), d < 32,
// then sit in one lane (k = 0 and k = 1), so every lane takes part in the rotation and the
// row's sum of squares needs three shuffle steps. Keys: [T][2][256] -> [T][2][256].
// Queries: the q halves of the fused rows [rows][24][512] -> [rows][24][256].
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
constexpr int kRowsPerBlock = 32;   // 8 warps x 4 rows
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
  const int j = lane & 7;
  const long long row = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 3);
  // whole row groups leave together: the shuffles below stay within a group of 8 lanes
  if (row >= n_rows) return;
  const unsigned gmask = 0xFFu << (lane & 24);
  const long long tok = row / heads_per_tok;
  int pos = pos_base + (int)tok;
  if (kSeq) {
    if (sp.n_seq > 0) {
      // the sequence holding packed token tok: the last b with row_start[b] <= tok
      int lo = 0, hi = sp.n_seq - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sp.row_start[mid] <= tok) lo = mid;
        else hi = mid - 1;
      }
      pos = sp.seq_base[lo] + (int)(tok - sp.row_start[lo]);
    } else {
      pos = sp.seq_base[tok / sp.rows_per_seq] + (int)(tok % sp.rows_per_seq);
    }
  }

  const uint2* xs = reinterpret_cast<const uint2*>(src + row * src_stride) + j;
  const uint2* ws = reinterpret_cast<const uint2*>(w_norm) + j;
  uint2 xv[8], wv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    xv[k] = __ldg(xs + 8 * k);
    wv[k] = __ldg(ws + 8 * k);
  }
  // sum of squares: two independent TwoSum chains per lane, then the row's 8 lanes in a
  // fixed order (lower lane first) so every lane of the row holds the same pair
  SumSq s0, s1;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    s0.add(lo_f(xv[k].x));
    s1.add(hi_f(xv[k].x));
    s0.add(lo_f(xv[k].y));
    s1.add(hi_f(xv[k].y));
  }
  s0.merge(s1);
  SumSq ss = s0;
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) {
    SumSq o;
    o.hi = __shfl_xor_sync(gmask, ss.hi, off, 8);
    o.lo = __shfl_xor_sync(gmask, ss.lo, off, 8);
    if (j & off) {
      SumSq t = o;
      t.merge(ss);
      ss = t;
    } else {
      ss.merge(o);
    }
  }
  const InvRms r = inv_rms_df(ss);

  // normed values (fp32 values whose bf16 rounding is the exact one: the fast result when
  // it is clear of a bf16 midpoint, else the exact bf16 value itself)
  auto norm4 = [&](int k, float (&y)[4]) {
    const float xk[4] = {lo_f(xv[k].x), hi_f(xv[k].x), lo_f(xv[k].y), hi_f(xv[k].y)};
    const float wk[4] = {lo_f(wv[k].x), hi_f(wv[k].x), lo_f(wv[k].y), hi_f(wv[k].y)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      y[i] = norm_fast(xk[i], wk[i], r);
      if (near_bf16_midpoint(y[i], 3)) y[i] = norm_elem_exact(xk[i], wk[i], r.h, r.l);
    }
  };
  uint2* out = reinterpret_cast<uint2*>(dst + row * kDim) + j;
  {
    // Partial RoPE on dims 0..63: pair p = 4j + i is (dim p, dim p + 32), both in this lane.
    float ya[4], yb[4];
    norm4(0, ya);
    norm4(1, yb);
    const uint2 cv = __ldg(reinterpret_cast<const uint2*>(cos_tab + (long long)pos * kHalfRot) + j);
    const uint2 sv = __ldg(reinterpret_cast<const uint2*>(sin_tab + (long long)pos * kHalfRot) + j);
    const float c[4] = {lo_f(cv.x), hi_f(cv.x), lo_f(cv.y), hi_f(cv.y)};
    const float sn[4] = {lo_f(sv.x), hi_f(sv.x), lo_f(sv.y), hi_f(sv.y)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float oa, ob;
      rope_pair(bf16_round(ya[i]), bf16_round(yb[i]), c[i], sn[i], oa, ob);
      ya[i] = oa;
      yb[i] = ob;
    }
    out[0] = make_uint2(pack2(ya[0], ya[1]), pack2(ya[2], ya[3]));
    out[8] = make_uint2(pack2(yb[0], yb[1]), pack2(yb[2], yb[3]));
  }
#pragma unroll
  for (int k = 2; k < 8; ++k) {
    float y[4];
    norm4(k, y);
    out[8 * k] = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
  }
}

}  // namespace

cudaError_t launch_k_prologue(const uint16_t* k_raw, const uint16_t* w_k, const uint16_t* cos_tab,
                              const uint16_t* sin_tab, int n_tok, int pos_base, uint16_t* k_prep,
                              int* status, cudaStream_t s) {
  (void)status;
  const long long n_rows = (long long)n_tok * kKvHeads;
  const unsigned grid = (unsigned)((n_rows + kRowsPerBlock - 1) / kRowsPerBlock);
  prologue_kernel<false><<<grid, 256, 0, s>>>(k_raw, kDim, kKvHeads, w_k, cos_tab, sin_tab,
                                              n_rows, pos_base, SeqPositions{}, k_prep);
  return cudaGetLastError();
}

cudaError_t launch_q_prologue(const uint16_t* qg, const uint16_t* w_q, const uint16_t* cos_tab,
                              const uint16_t* sin_tab, int rows, int q_base, uint16_t* q_prep,
                              cudaStream_t s) {
  const long long n_rows = (long long)rows * kHeads;
  const unsigned grid = (unsigned)((n_rows + kRowsPerBlock - 1) / kRowsPerBlock);
  prologue_kernel<false><<<grid, 256, 0, s>>>(qg, kQgStride, kHeads, w_q, cos_tab, sin_tab,
                                              n_rows, q_base, SeqPositions{}, q_prep);
  return cudaGetLastError();
}

cudaError_t launch_q_prologue_seq(const uint16_t* qg, const uint16_t* w_q, const uint16_t* cos_tab,
                                  const uint16_t* sin_tab, int n_tok, const SeqPositions& sp,
                                  uint16_t* q_prep, cudaStream_t s) {
  const long long n_rows = (long long)n_tok * kHeads;
  const unsigned grid = (unsigned)((n_rows + kRowsPerBlock - 1) / kRowsPerBlock);
  prologue_kernel<true><<<grid, 256, 0, s>>>(qg, kQgStride, kHeads, w_q, cos_tab, sin_tab, n_rows,
                                             0, sp, q_prep);
  return cudaGetLastError();
}

}  // namespace ga
