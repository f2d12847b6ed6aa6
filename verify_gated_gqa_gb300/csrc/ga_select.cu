// Selection mask from the indexer's block scores (pegainfer PR #1151, "feat(qwen4): add the
// QSA sparse-attention kernel and its golden": the attention reads the indexer's selection
// AND causality as its mask; the commit moving to the real geometry keeps 512 blocks for a
// budget of 2048 tokens, so a block is 4 consecutive keys).
//
// One CTA of 128 threads per query row r at position p = q_base + r. The row's candidates
// are the blocks b = 0 .. nc-1 holding a key j <= p, nc = min(ceil(T / 4), p / 4 + 1); it
// keeps the top_k highest scores, a tie going to the lower block index. Thread t holds
// blocks t + 128 i (i < 16) as order-preserving unsigned keys, and 0 for b >= nc: below
// every score's key, so padding never outranks a candidate, and any padding block that
// does get marked is hidden by causality (its keys lie after p).
//
// A radix select over four 8-bit digits finds the top_k-th largest key tau. Each warp
// counts its keys that match the prefix so far into a histogram of its own (shared-memory
// atomics; no same-address contention between warps), and warp 0 sums the four and finds
// the digit. When the digit's bin is taken whole the select stops early: the kept keys are
// then those whose prefix is at least tau's, with no tie to break. Otherwise the `need`
// keys equal to tau with the lowest block indices are kept, ranked by a block-wide count in
// index order. Kept blocks become a bitmask (one ballot per 32 blocks), and the row's T
// mask bytes (1 = visible) go out as 16-byte stores; only the store that straddles p
// computes causality byte by byte.
#include "ga_internal.h"

namespace ga {
namespace {

constexpr int kBlockTokens = GA_INDEX_BLOCK_TOKENS;   // 4
constexpr int kSelThreads = 128;
constexpr int kSelMaxBlocks = GA_MASKED_MAX_TOKENS / kBlockTokens;   // 2048
constexpr int kSelKeys = kSelMaxBlocks / kSelThreads;                // 16 per thread
constexpr int kSelWarps = kSelThreads / 32;
static_assert(kSelKeys * kSelThreads == kSelMaxBlocks, "blocks per row");
static_assert(kSelKeys * kSelWarps == kSelMaxBlocks / 32,
              "one bitmask word and one tie count per (key slot, warp); two per lane");

// IEEE order as unsigned order: negative values have every bit flipped, others the sign
// bit set. Adding +0 first turns -0 into +0 (round to nearest), so the two tie as the values
// do.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return u ^ ((uint32_t)((int)u >> 31) | 0x80000000u);
}

struct SelShared {
  uint32_t bits[kSelMaxBlocks / 32];        // bit b % 32 of word b / 32: block b kept
  alignas(16) int whist[kSelWarps][256];    // one digit histogram per warp
  int tie_base[kSelKeys * kSelWarps];       // entry i * 4 + warp
  int s_digit, s_need, s_all;
};

// One radix pass over digit P, the key's byte 3 - P: each warp counts its keys that match
// the prefix so far (every key in the first pass) into its own histogram, and warp 0 sums
// the four and finds the bin holding the need-th largest matching key. Returns true when
// that bin is taken whole.
template <int P>
__device__ __forceinline__ bool radix_pass(SelShared& sh, const uint32_t (&key)[kSelKeys],
                                           uint32_t& prefix, int& need, int lane, int warp) {
  constexpr uint32_t kMask = P == 0 ? 0u : (0xFFFFFFFFu << (32 - 8 * P));
  uint4* wh4 = reinterpret_cast<uint4*>(sh.whist[warp]);
  wh4[lane] = make_uint4(0, 0, 0, 0);
  wh4[lane + 32] = make_uint4(0, 0, 0, 0);
  __syncwarp();
  int* wh = sh.whist[warp];
#pragma unroll
  for (int i = 0; i < kSelKeys; ++i) {
    const uint32_t d = __byte_perm(key[i], 0, 0x4440 + (3 - P));
    if (P == 0 || (key[i] & kMask) == prefix) atomicAdd(wh + d, 1);
  }
  __syncthreads();
  if (warp == 0) {
    // lane l sums bins 8l .. 8l+7 over the warps; the digit is in the lane where the keys
    // in higher bins are fewer than `need` and those in its bins and higher are at least
    // `need`
    int c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      const uint4 x = reinterpret_cast<const uint4*>(sh.whist[w])[2 * lane];
      const uint4 y = reinterpret_cast<const uint4*>(sh.whist[w])[2 * lane + 1];
      c[0] += (int)x.x; c[1] += (int)x.y; c[2] += (int)x.z; c[3] += (int)x.w;
      c[4] += (int)y.x; c[5] += (int)y.y; c[6] += (int)y.z; c[7] += (int)y.w;
    }
    int sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) sum += c[j];
    int incl = sum;   // keys in the bins of lanes lane .. 31
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_down_sync(0xFFFFFFFFu, incl, off);
      if (lane + off < 32) incl += v;
    }
    const int above = incl - sum;
    if (above < need && need <= incl) {
      int acc = above;
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        if (acc < need && acc + c[j] >= need) {
          sh.s_digit = 8 * lane + j;
          sh.s_need = need - acc;
          sh.s_all = (need - acc) == c[j];
        }
        acc += c[j];
      }
    }
  }
  __syncthreads();
  prefix |= (uint32_t)sh.s_digit << (24 - 8 * P);
  need = sh.s_need;
  return sh.s_all != 0;
}

__global__ void __launch_bounds__(kSelThreads, 10) select_mask_kernel(
    const float* __restrict__ scores, long long ld_scores, int T, int q_base, int top_k,
    uint8_t* __restrict__ mask, long long ld_mask) {
  __shared__ SelShared sh;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  const int p = q_base + r;
  const int nb = (T + kBlockTokens - 1) / kBlockTokens;
  const int nc = min(nb, p / kBlockTokens + 1);

  if (top_k >= nc) {
    // every candidate is kept: the causal row
    for (int w = tid; w < kSelMaxBlocks / 32; w += kSelThreads)
      sh.bits[w] = 32 * w + 32 <= nc ? 0xFFFFFFFFu
                                     : (32 * w >= nc ? 0u : (1u << (nc - 32 * w)) - 1u);
  } else {
    const float* row = scores + (long long)r * ld_scores;
    uint32_t key[kSelKeys];
#pragma unroll
    for (int i = 0; i < kSelKeys; ++i) {
      const int b = tid + i * kSelThreads;
      key[i] = b < nc ? order_key(__ldg(row + b)) : 0u;
    }
    uint32_t prefix = 0;       // the digits of tau found so far
    uint32_t pmask = 0xFF000000u;
    int need = top_k;          // keys still to take among those that match the prefix
    bool whole = radix_pass<0>(sh, key, prefix, need, lane, warp);
    if (!whole) {
      pmask = 0xFFFF0000u;
      whole = radix_pass<1>(sh, key, prefix, need, lane, warp);
    }
    if (!whole) {
      pmask = 0xFFFFFF00u;
      whole = radix_pass<2>(sh, key, prefix, need, lane, warp);
    }
    if (!whole) {
      pmask = 0xFFFFFFFFu;
      whole = radix_pass<3>(sh, key, prefix, need, lane, warp);
    }
    if (whole) {
      // the bin is taken whole: the kept keys are those whose prefix is at least tau's
#pragma unroll
      for (int i = 0; i < kSelKeys; ++i) {
        const unsigned m = __ballot_sync(0xFFFFFFFFu, (key[i] & pmask) >= prefix);
        if (lane == 0) sh.bits[i * kSelWarps + warp] = m;
      }
    } else {
      // keys above tau are kept; of the keys equal to tau, the `need` lowest block indices.
      // Index order is (i, warp, lane), so the rank of a tie is the ties in earlier
      // (i, warp) groups plus those in lower lanes of its own warp.
      unsigned tie[kSelKeys];
#pragma unroll
      for (int i = 0; i < kSelKeys; ++i) {
        tie[i] = __ballot_sync(0xFFFFFFFFu, key[i] == prefix);
        if (lane == 0) sh.tie_base[i * kSelWarps + warp] = __popc(tie[i]);
      }
      __syncthreads();
      if (warp == 0) {
        const int a0 = sh.tie_base[2 * lane], a1 = sh.tie_base[2 * lane + 1];
        int incl = a0 + a1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
          if (lane >= off) incl += v;
        }
        const int excl = incl - a0 - a1;
        sh.tie_base[2 * lane] = excl;
        sh.tie_base[2 * lane + 1] = excl + a0;
      }
      __syncthreads();
      const unsigned lower = (1u << lane) - 1u;
#pragma unroll
      for (int i = 0; i < kSelKeys; ++i) {
        const bool is_tie = (tie[i] >> lane) & 1u;
        const int rank = sh.tie_base[i * kSelWarps + warp] + __popc(tie[i] & lower);
        const unsigned m = __ballot_sync(0xFFFFFFFFu, key[i] > prefix || (is_tie && rank < need));
        if (lane == 0) sh.bits[i * kSelWarps + warp] = m;
      }
    }
  }
  __syncthreads();

  // key j is visible iff j <= p and block j / 4 is kept
  uint8_t* out = mask + (long long)r * ld_mask;
  const int nvec = T / 16;
  for (int v = tid; v < nvec; v += kSelThreads) {
    const uint32_t nib = (sh.bits[v >> 3] >> (4 * (v & 7))) & 0xFu;   // blocks 4v .. 4v+3
    uint32_t word[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) word[q] = ((nib >> q) & 1u) * 0x01010101u;
    if (16 * v + 15 > p) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int vis = p - (16 * v + 4 * q) + 1;   // keys of block 4v + q at or before p
        word[q] &= vis >= 4 ? 0xFFFFFFFFu : (vis <= 0 ? 0u : (1u << (8 * vis)) - 1u);
      }
    }
    *reinterpret_cast<uint4*>(out + 16 * v) = make_uint4(word[0], word[1], word[2], word[3]);
  }
  for (int j = nvec * 16 + tid; j < T; j += kSelThreads)
    out[j] = (j <= p && ((sh.bits[j >> 7] >> ((j >> 2) & 31)) & 1u)) ? 1 : 0;
}

}  // namespace

cudaError_t launch_select_mask(const float* scores, long long ld_scores, int rows, int T,
                               int q_base, int top_k, uint8_t* mask, long long ld_mask,
                               cudaStream_t s) {
  select_mask_kernel<<<rows, kSelThreads, 0, s>>>(scores, ld_scores, T, q_base, top_k, mask,
                                                  ld_mask);
  return cudaGetLastError();
}

}  // namespace ga
