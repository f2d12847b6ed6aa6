// Prologue: (1+w) RMSNorm and partial RoPE of head rows, once per row (pegainfer PR
// #1151, "feat(qwen4): add the QSA sparse-attention kernel and its golden", §What changed:
// all twelve query heads of a KV head read the same prepared key; the query rows take
// the same norm with w_q at their own positions).
//
// Sixteen lanes (a half-warp) per (token, head) row of 256 bf16. Lane l holds the rotated
// pair dims 2l, 2l+1 and 32+2l, 33+2l (so both members of every RoPE pair (d, d+32) sit in
// one lane) and the pass-through dims 64 + 64k + 4l .. +3 for k = 0..2: 16 values in five
// loads, every load instruction of the half-warp one contiguous 64- or 128-byte run. The
// kernel is persistent: each half-warp walks rows with a stride of all half-warps, the
// next row's values in flight while the current one is computed.
//
// Exact rounding at low cost. The result must be the bf16 rounding of the exact
// x (1 + w) / sqrt(mean(x^2) + eps). The fast path sums the squares in plain fp32 (each
// square of a bf16 value is exact; a pairwise tree of depth 4 in the lane, then 4 shuffle
// levels: relative error at most 8u, u = 2^-24), adds eps (u), takes rsqrtf and one Newton
// step (about 1.5u), and forms fma(x, w, x) * r (two roundings): in all under 8u relative,
// which is under 8 fp32 ulps of the result. A result whose low 16 bits lie more than 9 ulps
// from the bf16 midpoint 0x8000 therefore rounds to the bf16 value of the exact result.
// Rows with an element inside that margin (about one in fourteen) take the exact path for
// those elements: the sum of squares as a TwoSum pair, the inverse RMS as a double-float,
// and a double-float product (ga_numerics.cuh).
#include "ga_internal.h"
#include "ga_numerics.cuh"
#include "ga_sm100.cuh"

namespace ga {
namespace {

__device__ __forceinline__ float lo_f(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hi_f(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Straight from a word of two bf16 values by mixed-precision FMAs (bf16 operands widened
// exactly, fp32 addend, one rounding), so the values need no unpacking on the integer pipe:
// lo^2 + hi^2 rounded once (hi^2 is exact), as fmaf(lo, lo, hi * hi).
__device__ __forceinline__ float sumsq2(uint32_t xw) {
  float t;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "fma.rn.f32.bf16 %0, hi, hi, 0f80000000;\n\t"
      "fma.rn.f32.bf16 %0, lo, lo, %0;\n\t}"
      : "=f"(t)
      : "r"(xw));
  return t;
}
// fl(x + x w) of the two halves, as fmaf(x, w, x): x w is exact (-0 as the addend keeps its
// sign), then x is added with one rounding.
__device__ __forceinline__ void xw_plus_x2(uint32_t xw, uint32_t ww, float& p0, float& p1) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh, one;\n\t"
      "mov.b32 {xl, xh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\tmov.b16 one, 0x3F80;\n\t"
      "fma.rn.f32.bf16 %0, xl, wl, 0f80000000;\n\t"
      "fma.rn.f32.bf16 %0, xl, one, %0;\n\t"
      "fma.rn.f32.bf16 %1, xh, wh, 0f80000000;\n\t"
      "fma.rn.f32.bf16 %1, xh, one, %1;\n\t}"
      : "=f"(p0), "=f"(p1)
      : "r"(xw), "r"(ww));
}

constexpr int kThreads = 256;          // 16 half-warps, one row each at a time
constexpr int kBlocksPerSm = 3;
constexpr int kFastMargin = 9;         // fp32 ulps around a bf16 midpoint (see above)

// The 16 values of a lane: words 0 and 1 hold dims (2l, 2l+1) and (32+2l, 33+2l); words
// 2..7 the pass-through dims, two bf16 per word, in the order of the loads.
struct RowVals {
  uint32_t w[8];
};

__device__ __forceinline__ void load_row(const uint16_t* p, int l, RowVals& v) {
  v.w[0] = __ldg(reinterpret_cast<const uint32_t*>(p) + l);
  v.w[1] = __ldg(reinterpret_cast<const uint32_t*>(p + 32) + l);
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const uint2 t = __ldg(reinterpret_cast<const uint2*>(p + 64 + 64 * k) + l);
    v.w[2 + 2 * k] = t.x;
    v.w[3 + 2 * k] = t.y;
  }
}

// One run of rows: (token, head) pairs over n_heads heads head0 .. head0+n_heads-1 of a
// token that has heads_per_tok heads. Row r is token r / n_heads, head head0 + r % n_heads;
// it reads 256 values at src + (token * heads_per_tok + head) * src_stride and writes 256 at
// dst + (token * heads_per_tok + head) * 256, normed with w_norm. Token t sits at position
// pos_base + t, or, with kSeq, at the position its sequence gives (SeqPositions).
struct PrologueRows {
  const uint16_t* src;
  uint16_t* dst;
  const uint16_t* w_norm;
  long long n_rows;   // callers keep it below 2^31
  int src_stride, heads_per_tok, head0, n_heads, pos_base;
};

// The rows first, first + stride, ... of one run, by this half-warp.
template <bool kSeq>
__device__ __forceinline__ void prologue_walk(const PrologueRows& run, int first, int stride,
                                              const uint16_t* __restrict__ cos_tab,
                                              const uint16_t* __restrict__ sin_tab,
                                              const SeqPositions& sp) {
  const uint16_t* __restrict__ src = run.src;
  uint16_t* __restrict__ dst = run.dst;
  const int src_stride = run.src_stride, heads_per_tok = run.heads_per_tok;
  const int head0 = run.head0, n_heads = run.n_heads, pos_base = run.pos_base;
  const int l = threadIdx.x & 15;
  const unsigned hmask = 0xFFFFu << (threadIdx.x & 16);   // this half-warp's lanes
  // rows are walked as (token, head) pairs: no division inside the loop
  const int n_rows32 = (int)run.n_rows;
  int row = first;
  if (row >= n_rows32) return;   // whole half-warps leave together
  const int stride_tok = stride / n_heads, stride_head = stride - stride_tok * n_heads;
  int tok = row / n_heads, head = row - tok * n_heads;

  // this lane's norm weights, in the value order of RowVals (two bf16 per word)
  RowVals wv;
  load_row(run.w_norm, l, wv);
  // element offset of the row (token t, head hd) in an array of rows stride_el values apart
  auto row_off = [&](int t, int hd, int stride_el) -> long long {
    return ((long long)t * heads_per_tok + head0 + hd) * stride_el;
  };
  auto position = [&](int t) -> int {
    if (!kSeq) return pos_base + t;
    if (sp.n_seq > 0) {
      // the sequence holding packed token t: the last b with row_start[b] <= t
      int lo = 0, hi = sp.n_seq - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sp.row_start[mid] <= t) lo = mid;
        else hi = mid - 1;
      }
      return sp.seq_base[lo] + (t - sp.row_start[lo]);
    }
    return sp.seq_base[t / sp.rows_per_seq] + t % sp.rows_per_seq;
  };

  RowVals cur;
  load_row(src + row_off(tok, head, src_stride), l, cur);
  while (true) {
    int ntok = tok + stride_tok, nhead = head + stride_head;
    if (nhead >= n_heads) {
      nhead -= n_heads;
      ++ntok;
    }
    const bool more = row + stride < n_rows32;
    RowVals nxt;
    if (more) load_row(src + row_off(ntok, nhead, src_stride), l, nxt);
    const int pos = position(tok);
    const uint32_t cw = __ldg(reinterpret_cast<const uint32_t*>(cos_tab + (long long)pos * kHalfRot) + l);
    const uint32_t sw = __ldg(reinterpret_cast<const uint32_t*>(sin_tab + (long long)pos * kHalfRot) + l);

    // fast sum of squares: pairs by one fma (the second square is exact), then a tree
    float t8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t8[i] = sumsq2(cur.w[i]);
#pragma unroll
    for (int i = 0; i < 4; ++i) t8[i] = t8[2 * i] + t8[2 * i + 1];
    t8[0] = t8[0] + t8[1];
    t8[2] = t8[2] + t8[3];
    float ssum = t8[0] + t8[2];
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) ssum += __shfl_xor_sync(hmask, ssum, off, 16);
    const float a = fmaf(ssum, 1.0f / 256.0f, kEps);
    const float r0 = rsqrtf(a);
    const float rf = fmaf(0.5f * r0, fmaf(-(a * r0), r0, 1.0f), r0);   // one Newton step

    // distance of each result's low 16 bits from the bf16 midpoint, shifted so that
    // "within the margin" reads d <= 2 * margin; the smallest decides the exact path
    // (one multiply-add per value: the low 16 bits moved to the top, the offset added there)
    float y[16];
    uint32_t dmin = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float p0, p1;
      xw_plus_x2(cur.w[i], wv.w[i], p0, p1);
      y[2 * i] = p0 * rf;
      y[2 * i + 1] = p1 * rf;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
      dmin = min(dmin, __float_as_uint(y[i]) * 65536u + ((uint32_t)(kFastMargin - 0x8000) << 16));
    const bool near_any = dmin <= (2u * kFastMargin) << 16;
    if (__any_sync(hmask, near_any)) {
      // exact path for this row: the sum of squares as a TwoSum pair, combined over the
      // row's 16 lanes in a fixed order (lower lane first) so every lane holds the same pair
      float x[16], w[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[2 * i] = lo_f(cur.w[i]);
        x[2 * i + 1] = hi_f(cur.w[i]);
        w[2 * i] = lo_f(wv.w[i]);
        w[2 * i + 1] = hi_f(wv.w[i]);
      }
      SumSq s0, s1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        s0.add(x[2 * i]);
        s1.add(x[2 * i + 1]);
      }
      s0.merge(s1);
      SumSq ss = s0;
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) {
        SumSq o;
        o.hi = __shfl_xor_sync(hmask, ss.hi, off, 16);
        o.lo = __shfl_xor_sync(hmask, ss.lo, off, 16);
        if (l & off) {
          SumSq t = o;
          t.merge(ss);
          ss = t;
        } else {
          ss.merge(o);
        }
      }
      const InvRms r = inv_rms_df(ss);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (near_bf16_midpoint(y[i], kFastMargin)) y[i] = norm_elem_exact(x[i], w[i], r.h, r.l);
    }

    // partial RoPE: values 0, 1 are dims 2l, 2l+1 (a) and 2, 3 are dims 32+2l, 33+2l (b)
    float oa0, ob0, oa1, ob1;
    rope_pair(bf16_round(y[0]), bf16_round(y[2]), lo_f(cw), lo_f(sw), oa0, ob0);
    rope_pair(bf16_round(y[1]), bf16_round(y[3]), hi_f(cw), hi_f(sw), oa1, ob1);
    uint16_t* out = dst + row_off(tok, head, kDim);
    reinterpret_cast<uint32_t*>(out)[l] = pack_bf16x2(oa0, oa1);
    reinterpret_cast<uint32_t*>(out + 32)[l] = pack_bf16x2(ob0, ob1);
#pragma unroll
    for (int k = 0; k < 3; ++k)
      reinterpret_cast<uint2*>(out + 64 + 64 * k)[l] =
          make_uint2(pack_bf16x2(y[4 + 4 * k], y[5 + 4 * k]), pack_bf16x2(y[6 + 4 * k], y[7 + 4 * k]));

    if (!more) break;
    row += stride;
    tok = ntok;
    head = nhead;
    cur = nxt;
  }
}

// One persistent grid over up to two runs of rows: every half-warp walks its rows of run0,
// then its rows of run1 (n_rows 0: none), the two runs dealt as one sequence of rows so that
// the half-warps' shares differ by one row at most.
template <bool kSeq>
__global__ void __launch_bounds__(kThreads, kBlocksPerSm)
    prologue_kernel(const __grid_constant__ PrologueRows run0,
                    const __grid_constant__ PrologueRows run1,
                    const uint16_t* __restrict__ cos_tab, const uint16_t* __restrict__ sin_tab,
                    const __grid_constant__ SeqPositions sp) {
  const int stride = gridDim.x * (kThreads / 16);
  const int hw = blockIdx.x * (kThreads / 16) + (threadIdx.x >> 4);
  prologue_walk<kSeq>(run0, hw, stride, cos_tab, sin_tab, sp);
  if (run1.n_rows > 0) {
    // the first row of run1 in this half-warp's share of the joined sequence
    const int first = (int)((((long long)hw - run0.n_rows) % stride + stride) % stride);
    prologue_walk<kSeq>(run1, first, stride, cos_tab, sin_tab, sp);
  }
}

unsigned prologue_grid(long long n_rows, int sm_count) {
  const long long need = (n_rows + kThreads / 16 - 1) / (kThreads / 16);
  const long long cap = (long long)(sm_count > 0 ? sm_count : 1) * kBlocksPerSm;
  return (unsigned)(need < cap ? need : cap);
}

PrologueRows k_rows(const uint16_t* k_raw, const uint16_t* w_k, int n_tok, int pos_base,
                    uint16_t* k_prep) {
  return PrologueRows{k_raw, k_prep, w_k, (long long)n_tok * kKvHeads, kDim, kKvHeads, 0,
                      kKvHeads, pos_base};
}
PrologueRows q_rows(const uint16_t* qg, const uint16_t* w_q, int rows, int q_base, int head0,
                    int n_heads, uint16_t* q_prep) {
  return PrologueRows{qg, q_prep, w_q, (long long)rows * n_heads, kQgStride, kHeads, head0,
                      n_heads, q_base};
}
PrologueRows no_rows() { return PrologueRows{nullptr, nullptr, nullptr, 0, 0, 1, 0, 1, 0}; }

}  // namespace

cudaError_t launch_k_prologue(const uint16_t* k_raw, const uint16_t* w_k, const uint16_t* cos_tab,
                              const uint16_t* sin_tab, int n_tok, int pos_base, uint16_t* k_prep,
                              int sm_count, cudaStream_t s) {
  const PrologueRows run = k_rows(k_raw, w_k, n_tok, pos_base, k_prep);
  prologue_kernel<false><<<prologue_grid(run.n_rows, sm_count), kThreads, 0, s>>>(
      run, no_rows(), cos_tab, sin_tab, SeqPositions{});
  return cudaGetLastError();
}

cudaError_t launch_q_prologue(const uint16_t* qg, const uint16_t* w_q, const uint16_t* cos_tab,
                              const uint16_t* sin_tab, int rows, int q_base, int head0,
                              int n_heads, uint16_t* q_prep, int sm_count, cudaStream_t s) {
  const PrologueRows run = q_rows(qg, w_q, rows, q_base, head0, n_heads, q_prep);
  prologue_kernel<false><<<prologue_grid(run.n_rows, sm_count), kThreads, 0, s>>>(
      run, no_rows(), cos_tab, sin_tab, SeqPositions{});
  return cudaGetLastError();
}

cudaError_t launch_qk_prologue(const uint16_t* k_raw, const uint16_t* w_k, int n_tok,
                               int k_pos_base, uint16_t* k_prep, const uint16_t* qg,
                               const uint16_t* w_q, int rows, int q_base, uint16_t* q_prep,
                               const uint16_t* cos_tab, const uint16_t* sin_tab, int sm_count,
                               cudaStream_t s) {
  const PrologueRows rk = k_rows(k_raw, w_k, n_tok, k_pos_base, k_prep);
  const PrologueRows rq = q_rows(qg, w_q, rows, q_base, 0, kHeads, q_prep);
  prologue_kernel<false><<<prologue_grid(rk.n_rows + rq.n_rows, sm_count), kThreads, 0, s>>>(
      rk, rq, cos_tab, sin_tab, SeqPositions{});
  return cudaGetLastError();
}

cudaError_t launch_q_prologue_seq(const uint16_t* qg, const uint16_t* w_q, const uint16_t* cos_tab,
                                  const uint16_t* sin_tab, int n_tok, const SeqPositions& sp,
                                  uint16_t* q_prep, int sm_count, cudaStream_t s) {
  const PrologueRows run = q_rows(qg, w_q, n_tok, 0, 0, kHeads, q_prep);
  prologue_kernel<true><<<prologue_grid(run.n_rows, sm_count), kThreads, 0, s>>>(
      run, no_rows(), cos_tab, sin_tab, sp);
  return cudaGetLastError();
}

}  // namespace ga
