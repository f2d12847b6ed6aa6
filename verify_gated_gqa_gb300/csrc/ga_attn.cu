// Flash-style gated GQA attention forward for sm_103a (tcgen05 + TMA + TMEM).
//
// What it computes (pegainfer PR #1151, "feat(qwen4): add the QSA sparse-attention
// kernel and its golden", §Semantics and the commit that adds the attention reader):
// per query head h and row r, q = (1+w_q) RMSNorm of the q half of the fused row,
// rotated on dims 0..63 at position q_base + r; s_j = bf16(q . k_j) / 16 against the
// prepared keys of KV head h / 12; softmax over the visible keys with the weights rounded
// to bf16 before the context reduction; o = bf16(sum_j w_j v_j); out = bf16(o * bf16(
// sigmoid(gate))).
//
// Softmax recurrence (system1-omni PR #202, "cuda: widen the attention query tile on
// sm_89 and sm_120", first review §Kernel change: running max, exp2, row sum, rescale of
// O; masked lanes add exactly +0). Here the running maximum M is an integer in base-2
// units, P = bf16(2^(t - M)) with t = s * log2(e), and O and l are rescaled by the exact
// power of two 2^(M_old - M_new) only when the tile maximum exceeds M by more than 8.
// bf16 rounding commutes with power-of-two scaling, so every row's weights are exactly
// bf16(e^s) up to a common power of two, whatever the tile schedule: a row's bits do
// not depend on which tile or window computes it.
//
// Structure (one CTA per SM, persistent, 384 threads in three warpgroups):
//   warp 0     TMA producer: K and V tiles of 128 keys x 256 dims (64 KiB, four 16 KiB
//              128-byte-swizzled column blocks) through three tile slots;
//   warp 1     allocates the 512 TMEM columns and issues every tcgen05.mma, all at full
//              rate (N >= 128): S = Q K^T (M=128, N=128, K=256; Q read from TMEM), then
//              O += P V (M=128, N=256, K=128; P from shared memory, V MN-major);
//   warps 4-7  softmax, one query row per thread: S is copied to registers and its TMEM
//              columns released at once (so the next S = Q K^T overlaps this softmax),
//              P = bf16(2^(t - M)) goes to shared memory, the rare O rescale;
//   warps 8-11 the edge of each work item, off the critical path: the next item's Q
//              (norm, RoPE) into TMEM, and the gated epilogue (O drained to bf16
//              registers first so the next item's P V can start, then the gate and
//              16-byte stores). Rows of upcoming items are prefetched into L2.
// Tensor memory (512 columns x 128 lanes, lane = query row): O [0, 256) fp32, Q
// [256, 384) bf16 pairs, S [384, 512) fp32.
// Work items are (query head, 128-row tile), longest first, dealt to the CTAs in a
// serpentine order so each CTA's total work evens out.
#include "ga_internal.h"
#include "ga_numerics.cuh"
#include "ga_sm100.cuh"

namespace ga {
namespace {

constexpr int kSlots = 3;
constexpr int kChunkBytes = kTileN * 128;     // 128 keys x 64 dims of bf16
constexpr int kTileBytes = 4 * kChunkBytes;   // 128 keys x 256 dims
constexpr int kThreads = 384;     // three warpgroups
// Register split (setmaxnreg): the kernel is launched at kLaunchRegs per thread; the
// producer/MMA warpgroup gives registers back and the softmax and edge warpgroups take
// them. The shares add up to the launch total: 128*56 + 2*128*224 = 384*168, and on each
// SM sub-partition (one warp of each warpgroup) 32*(56 + 224 + 224) <= 16384.
constexpr int kLaunchRegs = 168;
constexpr int kRegsIssue = 56;
constexpr int kRegsWork = 224;
static_assert(128 * kRegsIssue + 2 * 128 * kRegsWork == kThreads * kLaunchRegs, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;      // O accumulator: 256 columns (fp32)
constexpr uint32_t kTmemQ = 256;    // Q: 128 columns of bf16 pairs (A operand of Q K^T)
constexpr uint32_t kTmemS = 384;    // S: 128 columns (fp32)
constexpr float kLog2eOver16 = 1.4426950408889634f / 16.0f;
constexpr int kLazyRescale = 8;     // rescale when the tile maximum exceeds M by > 2^8

static_assert(kTileN == 128, "this kernel is laid out for 128-key tiles");

struct AttnSmem {
  uint8_t tile[kSlots][kTileBytes];   // K or V tiles (1024-byte aligned)
  uint8_t p[2][kChunkBytes];          // P: 128 rows x 128 keys, two swizzled 64-key columns
  float stat_l[kTileM];               // softmax -> edge: the row sum l of the finished item
  float stat_m[kTileM];               // and its running maximum M
  uint4 w_q[kDim / 8];                // the query norm weight, staged once
  uint64_t full[kSlots], empty[kSlots];
  uint64_t q_full, q_empty, s_full, s_free, p_full, p_empty;
  uint64_t o_ready, o_done, o_free, st_full, st_empty, drain;
  uint32_t tmem_base;
  int abort;
};

// ------------------------------------------------------------------ work items
struct Item {
  int h, mt;          // query head, 128-row tile
  int n;              // key tiles to visit
  bool masked;        // mask mode: visit only the key tiles listed in `tiles`
  uint64_t tiles[2];  // mask mode: bit kt set for every key tile with a visible key
};

__device__ __forceinline__ int item_index(int round, int cta, int G) {
  return round * G + ((round & 1) ? (G - 1 - cta) : cta);
}

__device__ __forceinline__ Item make_item(const AttnArgs& a, int idx) {
  Item it;
  it.mt = a.row_tiles - 1 - idx / kHeads;  // later row tiles see more keys: longest first
  it.h = idx % kHeads;
  it.masked = a.mode == kModeMask;
  it.tiles[0] = it.tiles[1] = 0;
  if (a.mode == kModeCausal) {
    const int last_row = min(a.rows, (it.mt + 1) * kTileM) - 1;
    const int key_end = min(a.T, a.q_base + last_row + 1);
    it.n = (key_end + kTileN - 1) / kTileN;
  } else if (a.mode == kModeBidir) {
    it.n = (a.T + kTileN - 1) / kTileN;
  } else {
    const uint8_t* f = a.tile_flags + (size_t)it.mt * a.key_tiles;
    for (int kt = 0; kt < a.key_tiles; ++kt)
      if (f[kt]) it.tiles[kt >> 6] |= (1ull << (kt & 63));
    it.n = __popcll(it.tiles[0]) + __popcll(it.tiles[1]);
  }
  return it;
}

// Walks the key tiles of an item in order: 0 .. n-1, or the set bits of a mask-mode item.
struct TileCursor {
  uint64_t w0, w1;
  __device__ __forceinline__ explicit TileCursor(const Item& it) : w0(it.tiles[0]), w1(it.tiles[1]) {}
  __device__ __forceinline__ int next(const Item& it, int j) {
    if (!it.masked) return j;
    if (w0) {
      const int kt = __ffsll((long long)w0) - 1;
      w0 &= w0 - 1;
      return kt;
    }
    const int kt = 64 + __ffsll((long long)w1) - 1;
    w1 &= w1 - 1;
    return kt;
  }
};

// The CTA's sequence of work items that have key tiles (items without any, in mask
// mode, are skipped here and answered by the edge warps).
struct ItemWalk {
  int round = 0;
  __device__ __forceinline__ bool next(const AttnArgs& a, Item& out) {
    const int G = gridDim.x;
    for (;; ++round) {
      const int idx = item_index(round, blockIdx.x, G);
      if (idx >= a.n_items) return false;
      out = make_item(a, idx);
      if (out.n > 0) {
        ++round;
        return true;
      }
    }
  }
};

__device__ __forceinline__ void record_abort(int* status, int code) {
  if (code) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------ warp 0: producer
__device__ void producer_loop(AttnSmem& sm, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                              const AttnArgs& a, volatile int* abort, uint32_t& cnt) {
  auto load_tile = [&](const CUtensorMap* map, int kvh, int kt) -> bool {
    const uint32_t slot = cnt % kSlots;
    if (!mbar_wait(&sm.empty[slot], ((cnt / kSlots) & 1) ^ 1, abort)) return false;
    mbar_expect_tx(&sm.full[slot], kTileBytes);
    for (int c = 0; c < 4; ++c)
      tma_load_3d(sm.tile[slot] + c * kChunkBytes, map, &sm.full[slot], c * 64, kvh, kt * kTileN);
    ++cnt;
    return true;
  };
  ItemWalk walk;
  Item it;
  while (walk.next(a, it)) {
    const int kvh = it.h / kGroup;
    TileCursor ck(it), cv(it);
    // Ring order = MMA order: K0, then (K_j, V_{j-1}) for j >= 1, then V_{n-1}.
    if (!load_tile(tm_k, kvh, ck.next(it, 0))) return;
    for (int j = 1; j < it.n; ++j) {
      if (!load_tile(tm_k, kvh, ck.next(it, j))) return;
      if (!a.weights_pass && !load_tile(tm_v, kvh, cv.next(it, j - 1))) return;
    }
    if (!a.weights_pass && !load_tile(tm_v, kvh, cv.next(it, it.n - 1))) return;
  }
}

__device__ void producer(AttnSmem& sm, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                         const AttnArgs& a, volatile int* abort) {
  uint32_t cnt = 0;
  producer_loop(sm, tm_k, tm_v, a, abort, cnt);
  if (*abort) {
    // let the loads already issued into the slots land before exit
    const uint32_t first = cnt > (uint32_t)kSlots ? cnt - kSlots : 0;
    for (uint32_t c = first; c < cnt; ++c)
      mbar_wait_quiet(&sm.full[c % kSlots], (c / kSlots) & 1, 100000000LL);
  }
}

// ------------------------------------------------------------------ warp 1: MMA issuer
__device__ void mma_loop(AttnSmem& sm, const AttnArgs& a, uint32_t tmem, volatile int* abort) {
  constexpr uint32_t kIdQK = idesc_bf16(128, kTileN, false, false);
  constexpr uint32_t kIdPV = idesc_bf16(128, kDim, false, true);
  const uint32_t p_addr = smem_u32(sm.p[0]);
  uint32_t cnt = 0;       // tile-slot sequence (same order as the producer)
  uint32_t g = 0;         // global key-tile counter: S, P and PV phases
  uint32_t it_done = 0;

  auto take = [&](uint32_t& slot) -> bool {
    slot = cnt % kSlots;
    if (!mbar_wait(&sm.full[slot], (cnt / kSlots) & 1, abort)) return false;
    tc_fence_after();
    ++cnt;
    return true;
  };
  auto issue_pv = [&](int j, uint32_t gj) -> bool {
    uint32_t slot;
    if (!take(slot)) return false;
    if (j == 0 && it_done > 0 && !mbar_wait(&sm.o_free, (it_done - 1) & 1, abort)) return false;
    if (!mbar_wait(&sm.p_full, gj & 1, abort)) return false;
    tc_fence_after();
    const uint32_t v_addr = smem_u32(sm.tile[slot]);
#pragma unroll
    for (int kk = 0; kk < kTileN / 16; ++kk) {
      const uint64_t ad = sdesc_sw128(p_addr + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024);
      const uint64_t bd = sdesc_sw128(v_addr + kk * 2048, kChunkBytes, 1024);
      umma_ss(tmem + kTmemO, ad, bd, kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
    }
    umma_commit(&sm.empty[slot]);
    umma_commit(&sm.p_empty);
    umma_commit(&sm.o_ready);
    return true;
  };

  ItemWalk walk;
  Item it;
  while (walk.next(a, it)) {
    if (!mbar_wait(&sm.q_full, it_done & 1, abort)) return;
    tc_fence_after();
    for (int j = 0; j < it.n; ++j, ++g) {
      uint32_t slot;
      if (!take(slot)) return;
      // S is free once the softmax warps have copied the previous tile's S out
      if (g > 0 && !mbar_wait(&sm.s_free, (g - 1) & 1, abort)) return;
      tc_fence_after();
      const uint32_t k_addr = smem_u32(sm.tile[slot]);
#pragma unroll
      for (int kk = 0; kk < kDim / 16; ++kk) {
        const uint64_t bd = sdesc_sw128(k_addr + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024);
        umma_ts(tmem + kTmemS, tmem + kTmemQ + kk * 8, bd, kIdQK, kk > 0 ? 1u : 0u);
      }
      umma_commit(&sm.empty[slot]);
      umma_commit(&sm.s_full);
      if (j == it.n - 1) umma_commit(&sm.q_empty);
      if (!a.weights_pass && j >= 1 && !issue_pv(j - 1, g - 1)) return;
    }
    if (!a.weights_pass) {
      if (!issue_pv(it.n - 1, g - 1)) return;
      umma_commit(&sm.o_done);
    }
    ++it_done;
  }
}

// Issue every MMA, then wait (bounded) until all of them completed, so that tensor
// memory is never released under an MMA in flight.
__device__ void mma_issuer(AttnSmem& sm, const AttnArgs& a, uint32_t tmem, volatile int* abort) {
  mma_loop(sm, a, tmem, abort);
  umma_commit(&sm.drain);
  mbar_wait_quiet(&sm.drain, 0, 100000000LL);
}

// ------------------------------------------------------------------ shared helpers
__device__ __forceinline__ float lo_f(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hi_f(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return (uint32_t)bf16_bits(a) | ((uint32_t)bf16_bits(b) << 16);
}

// Wait in all 32 lanes and agree on the outcome, so that the warp-collective TMEM loads and
// stores that follow always run with the whole warp (or the whole warp leaves).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// Visibility of the 32 keys kt*128 + 32*ch .. +31 for one row: bit k <-> key +k.
__device__ __forceinline__ uint32_t chunk_visibility(const AttnArgs& a, int row, int kt, int ch,
                                                     bool valid) {
  if (!valid) return 0u;
  if (a.mode == kModeMask)
    return __ldg(a.mask_bits + (size_t)row * a.mask_words + kt * (kTileN / 32) + ch);
  const int first = kt * kTileN + ch * 32;
  int n = (a.mode == kModeCausal) ? (a.q_base + row - first + 1) : (a.T - first);
  n = max(0, min(32, n));
  return n >= 32 ? 0xFFFFFFFFu : ((1u << n) - 1u);
}

// ------------------------------------------------------------------ warps 4-7: softmax
// Weights pass: bf16(bf16(2^(t - M)) / l) for the keys of one tile (bf16 score pairs in
// sb[0 .. 63], hidden ones -inf), with the main pass's final M and l, written to
// weights[h][row][kt*128 ..].
__device__ __forceinline__ void weights_tile(const AttnArgs& a, const uint32_t (&sb)[kTileN],
                                             int h, int row, int kt, int M, float l_final) {
  const float mf = (float)M;
  uint16_t* wrow = a.weights + ((size_t)h * a.rows + row) * (size_t)a.T + (size_t)kt * kTileN;
  const int ncol = min(kTileN, a.T - kt * kTileN);
  const bool vec = (ncol == kTileN) && ((a.T & 7) == 0);
#pragma unroll
  for (int ch = 0; ch < kTileN / 32; ++ch) {
    uint32_t pk[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t w = sb[ch * 16 + k];
      const float p0 = bf16_round(ex2_approx(fmaf(lo_f(w), kLog2eOver16, -mf)));
      const float p1 = bf16_round(ex2_approx(fmaf(hi_f(w), kLog2eOver16, -mf)));
      pk[k] = pack2(p0 / l_final, p1 / l_final);
    }
    if (vec) {
      uint4* dst = reinterpret_cast<uint4*>(wrow + ch * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (ch * 32 + k < ncol)
          wrow[ch * 32 + k] = (uint16_t)((k & 1) ? (pk[k >> 1] >> 16) : (pk[k >> 1] & 0xFFFFu));
    }
  }
}

__device__ void softmax_worker(AttnSmem& sm, const AttnArgs& a, uint32_t tmem,
                               volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t s_taddr = tmem + kTmemS + lane_off;
  uint32_t g = 0, it_done = 0;
  ItemWalk walk;
  Item it;
  while (walk.next(a, it)) {
    const int row = it.mt * kTileM + r;
    const bool valid = row < a.rows;
    const int h = it.h;
    int M = 0;
    bool hasM = false;
    float l = 0.f;
    float l_final = 0.f;  // weights pass: the main pass's l (relative to its final M)
    if (a.weights_pass && valid) {
      M = (int)a.row_stats[((size_t)h * a.rows + row) * 2];
      l_final = a.row_stats[((size_t)h * a.rows + row) * 2 + 1];
      hasM = l_final > 0.f;
    }
    TileCursor cursor(it);
    for (int j = 0; j < it.n; ++j, ++g) {
      const int kt = cursor.next(it, j);
      if (!warp_wait(&sm.s_full, g & 1, abort)) return;
      tc_fence_after();
      // S -> registers (four loads, one wait), packed in place as bf16 pairs (the score's
      // own rounding); then the columns are released
      uint32_t sb[kTileN];
      tmem_ld32(s_taddr + 0, *reinterpret_cast<uint32_t(*)[32]>(sb));
      tmem_ld32(s_taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(sb + 32));
      tmem_ld32(s_taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(sb + 64));
      tmem_ld32(s_taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(sb + 96));
      tmem_wait_ld(sb);
      tc_fence_before();
      mbar_arrive(&sm.s_free);   // the next S = Q K^T may overwrite these columns now
#pragma unroll
      for (int ch = 0; ch < kTileN / 32; ++ch) {
        const uint32_t vis = chunk_visibility(a, row, kt, ch, valid);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          // hidden keys read as -inf: weight exactly 0, never the maximum
          const int e = ch * 32 + 2 * k;
          const float s0 = ((vis >> (2 * k)) & 1u) ? __uint_as_float(sb[e]) : -INFINITY;
          const float s1 = ((vis >> (2 * k + 1)) & 1u) ? __uint_as_float(sb[e + 1]) : -INFINITY;
          sb[ch * 16 + k] = pack_bf16x2(s0, s1);   // writes an index already read
        }
      }

      if (a.weights_pass) {
        if (valid && hasM) weights_tile(a, sb, h, row, kt, M, l_final);
        continue;
      }
      // tile maximum of the bf16 scores
      float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
      for (int k = 0; k < kTileN / 2; k += 2) {
        m0 = fmaxf(m0, lo_f(sb[k]));
        m1 = fmaxf(m1, hi_f(sb[k]));
        m2 = fmaxf(m2, lo_f(sb[k + 1]));
        m3 = fmaxf(m3, hi_f(sb[k + 1]));
      }
      const float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
      bool rescale = false;
      int newM = M;
      if (mx != -INFINITY) {
        const int need = (int)ceilf(mx * kLog2eOver16);
        if (!hasM) {
          newM = need;
          hasM = true;
        } else if (need > M + kLazyRescale) {
          newM = need;
          rescale = true;
        }
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O must hold every earlier P.V before it is scaled (the PV of global tile g-1)
        if (!warp_wait(&sm.o_ready, (g - 1) & 1, abort)) return;
        tc_fence_after();
        const float f = rescale ? exp2f((float)(M - newM)) : 1.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < kDim; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + kTmemO + lane_off + c0, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
          tmem_st32(tmem + kTmemO + lane_off + c0, o);
        }
        tmem_wait_st();
        l *= f;
      }
      M = newM;
      const float mf = hasM ? (float)M : 0.f;
      // P = bf16(2^(t - M)), t = bf16(s) * log2(e) / 16, into shared memory once the
      // previous P.V has read the buffer; l sums the rounded P
      if (g > 0 && !warp_wait(&sm.p_empty, (g - 1) & 1, abort)) return;
      float la = 0.f, lb = 0.f;
#pragma unroll
      for (int cd = 0; cd < kTileN / 8; ++cd) {
        uint32_t pk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t w = sb[cd * 4 + k];
          const float p0 = ex2_approx(fmaf(lo_f(w), kLog2eOver16, -mf));
          const float p1 = ex2_approx(fmaf(hi_f(w), kLog2eOver16, -mf));
          pk[k] = pack_bf16x2(p0, p1);
          la += lo_f(pk[k]);
          lb += hi_f(pk[k]);
        }
        uint8_t* dst = sm.p[cd >> 3] + sw128_offset((uint32_t)r, (uint32_t)(cd & 7));
        *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      l += la + lb;
      fence_async_smem();
      mbar_arrive(&sm.p_full);
    }
    if (!a.weights_pass) {
      // hand l and M of this item to the edge warps
      if (it_done > 0 && !warp_wait(&sm.st_empty, (it_done - 1) & 1, abort)) return;
      sm.stat_l[r] = l;
      sm.stat_m[r] = hasM ? (float)M : 0.f;
      mbar_arrive(&sm.st_full);
    }
    ++it_done;
  }
}

// ------------------------------------------------------------------ warps 8-11: edge
// Norm of 8 dims (4 words of bf16 pairs, weights wv) with the row's double inverse RMS
// rh + rl: exact bf16 values in y.
__device__ __forceinline__ void norm8_exact(const uint4& xv, const uint4& wv, float rh, float rl,
                                            float (&y)[8]) {
  const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    y[2 * k] = norm_elem_exact(lo_f(xs[k]), lo_f(ww[k]), rh, rl);
    y[2 * k + 1] = norm_elem_exact(hi_f(xs[k]), hi_f(ww[k]), rh, rl);
  }
}

// (1+w) RMSNorm and partial RoPE of one query row into registers, as the bf16 pairs of
// its TMEM lane (word c holds dims 2c and 2c+1); rows past the end give zeros. The sum
// of squares is carried as hi + lo, the inverse RMS taken in double once per row, and
// every element's product is formed in double-float, so no element needs a second pass.
__device__ __forceinline__ void prep_q_compute(const AttnSmem& sm, const AttnArgs& a, int h,
                                               int row, bool valid, uint32_t (&q)[kDim / 2]) {
  if (!valid) {
#pragma unroll
    for (int k = 0; k < kDim / 2; ++k) q[k] = 0u;
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(a.qg + ((size_t)row * kHeads + h) * kQgStride);
  const uint4* wq = sm.w_q;
  // pass 1: the sum of squares over the row (32 loads in flight, consumed as they land)
  SumSq acc[4];
  {
    uint4 v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __ldg(src + i);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      acc[i & 3].add(lo_f(v[i].x)); acc[i & 3].add(hi_f(v[i].x));
      acc[i & 3].add(lo_f(v[i].y)); acc[i & 3].add(hi_f(v[i].y));
      acc[i & 3].add(lo_f(v[i].z)); acc[i & 3].add(hi_f(v[i].z));
      acc[i & 3].add(lo_f(v[i].w)); acc[i & 3].add(hi_f(v[i].w));
    }
  }
  acc[0].merge(acc[1]);
  acc[2].merge(acc[3]);
  acc[0].merge(acc[2]);
  const double r64 = inv_rms_f64(acc[0]);
  const float rh = (float)r64;
  const float rl = (float)(r64 - (double)rh);
  // pass 2 (the row is in L1 now). Dims 0..63 with the rotation: dims 8c..8c+7 pair
  // with dims 8c+32..8c+39.
  const int pos = a.q_base + row;
  const uint4* cp = reinterpret_cast<const uint4*>(a.cos_tab + (size_t)pos * kHalfRot);
  const uint4* sp = reinterpret_cast<const uint4*>(a.sin_tab + (size_t)pos * kHalfRot);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float ya[8], yb[8];
    norm8_exact(__ldg(src + c), wq[c], rh, rl, ya);
    norm8_exact(__ldg(src + c + 4), wq[c + 4], rh, rl, yb);
    const uint4 cv = __ldg(cp + c), sv = __ldg(sp + c);
    const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
    const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float cs = (e & 1) ? hi_f(cw[e >> 1]) : lo_f(cw[e >> 1]);
      const float sn = (e & 1) ? hi_f(sw[e >> 1]) : lo_f(sw[e >> 1]);
      float ra, rb;
      rope_pair(ya[e], yb[e], cs, sn, ra, rb);
      ya[e] = ra;
      yb[e] = rb;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      q[4 * c + k] = pack2(ya[2 * k], ya[2 * k + 1]);
      q[16 + 4 * c + k] = pack2(yb[2 * k], yb[2 * k + 1]);
    }
  }
  // dims 64..255 pass through the rotation
#pragma unroll
  for (int c = 8; c < 32; ++c) {
    float y[8];
    norm8_exact(__ldg(src + c), wq[c], rh, rl, y);
#pragma unroll
    for (int k = 0; k < 4; ++k) q[4 * c + k] = pack2(y[2 * k], y[2 * k + 1]);
  }
}

// The prepared row into this thread's TMEM lane at Q. Every lane of the warp runs it
// (the stores are warp-collective).
__device__ __forceinline__ void store_q_tmem(const uint32_t (&q)[kDim / 2], uint32_t q_taddr) {
#pragma unroll
  for (int grp = 0; grp < 4; ++grp)
    tmem_st32(q_taddr + 32 * grp, *reinterpret_cast<const uint32_t(*)[32]>(q + 32 * grp));
  tmem_wait_st();
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// The 512 bytes at byte offset `half` (0: q, 512: gate) of this thread's fused row.
__device__ __forceinline__ void prefetch_row(const AttnArgs& a, const Item& it, int r, int half) {
  const int row = it.mt * kTileM + r;
  if (row >= a.rows) return;
  const uint8_t* p = reinterpret_cast<const uint8_t*>(a.qg + ((size_t)row * kHeads + it.h) * kQgStride) + half;
#pragma unroll
  for (int i = 0; i < 4; ++i) prefetch_l2(p + 128 * i);
}

// Outputs of a work item none of whose key tiles is visible (mask mode): every row is
// hidden, its output row and statistics are zero.
__device__ void write_hidden_rows(const AttnArgs& a, const Item& it, int r) {
  const int row = it.mt * kTileM + r;
  if (row >= a.rows || a.weights_pass) return;
  uint4* o = reinterpret_cast<uint4*>(a.out + (size_t)row * kOutRow + it.h * kDim);
  for (int i = 0; i < 32; ++i) o[i] = make_uint4(0, 0, 0, 0);
  if (a.row_stats) {
    a.row_stats[((size_t)it.h * a.rows + row) * 2] = 0.f;
    a.row_stats[((size_t)it.h * a.rows + row) * 2 + 1] = 0.f;
  }
  if (a.hidden_rows && it.h == 0) atomicAdd(a.hidden_rows, 1);
}

// One 32-dim batch of the gate with the exact sigmoid wherever the fast one is not
// certified (rare: a gate whose sigmoid lies near a bf16 midpoint, or a very negative gate).
// o0..o3 are the batch's bf16 pairs of O / l; the batch's 4 output words are rewritten.
__device__ __noinline__ void gate_batch_slow(const uint4* gp, uint4* op, uint4 o0, uint4 o1,
                                             uint4 o2, uint4 o3) {
  const uint4 ov[4] = {o0, o1, o2, o3};
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const uint4 gv = gp[i];
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    const uint32_t ow[4] = {ov[i].x, ov[i].y, ov[i].z, ov[i].w};
    uint32_t res[4];
    for (int k = 0; k < 4; ++k) {
      float s0, s1;
      if (!sigmoid_fast(lo_f(gw[k]), s0)) s0 = sigmoid_slow(lo_f(gw[k]));
      if (!sigmoid_fast(hi_f(gw[k]), s1)) s1 = sigmoid_slow(hi_f(gw[k]));
      res[k] = pack2(lo_f(ow[k]) * bf16_round(s0), hi_f(ow[k]) * bf16_round(s1));
    }
    op[i] = make_uint4(res[0], res[1], res[2], res[3]);
  }
}

// Gated epilogue of one finished item: out = bf16(bf16(O / l) * bf16(sigmoid(gate))).
// O is drained to bf16 registers first and released, then the gate is applied.
__device__ __forceinline__ bool epilogue(AttnSmem& sm, const AttnArgs& a, const Item& it, uint32_t tmem,
                         uint32_t lane_off, int r, uint32_t it_done, volatile int* abort) {
  const int row = it.mt * kTileM + r;
  const bool valid = row < a.rows;
  const int h = it.h;
  if (!warp_wait(&sm.st_full, it_done & 1, abort)) return false;
  const float l = sm.stat_l[r];
  const float M = sm.stat_m[r];
  if (!warp_wait(&sm.o_done, it_done & 1, abort)) return false;
  tc_fence_after();
  const float inv = l > 0.f ? 1.0f / l : 0.f;
  uint32_t ob[kDim / 2];
#pragma unroll
  for (int c = 0; c < kDim / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(tmem + kTmemO + lane_off + c * 32, o);
    tmem_wait_ld(o);
#pragma unroll
    for (int k = 0; k < 16; ++k)
      ob[c * 16 + k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
  }
  tc_fence_before();
  mbar_arrive(&sm.o_free);
  mbar_arrive(&sm.st_empty);
  if (!valid) return true;
  const uint4* gp = reinterpret_cast<const uint4*>(a.qg + ((size_t)row * kHeads + h) * kQgStride + kDim);
  uint4* op = reinterpret_cast<uint4*>(a.out + (size_t)row * kOutRow + h * kDim);
#pragma unroll
  for (int q4 = 0; q4 < 8; ++q4) {       // 32 dims at a time, 4 loads in flight
    uint4 gv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) gv[i] = __ldg(gp + q4 * 4 + i);
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t gw[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
      uint32_t res[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t ow = ob[(q4 * 4 + i) * 4 + k];
        float s0, s1;
        ok &= sigmoid_fast(lo_f(gw[k]), s0);
        ok &= sigmoid_fast(hi_f(gw[k]), s1);
        res[k] = pack2(lo_f(ow) * bf16_round(s0), hi_f(ow) * bf16_round(s1));
      }
      op[q4 * 4 + i] = make_uint4(res[0], res[1], res[2], res[3]);
    }
    if (!ok) {
      const int b = q4 * 16;
      gate_batch_slow(gp + q4 * 4, op + q4 * 4, make_uint4(ob[b], ob[b + 1], ob[b + 2], ob[b + 3]),
                      make_uint4(ob[b + 4], ob[b + 5], ob[b + 6], ob[b + 7]),
                      make_uint4(ob[b + 8], ob[b + 9], ob[b + 10], ob[b + 11]),
                      make_uint4(ob[b + 12], ob[b + 13], ob[b + 14], ob[b + 15]));
    }
  }
  if (a.row_stats) {
    a.row_stats[((size_t)h * a.rows + row) * 2] = M;
    a.row_stats[((size_t)h * a.rows + row) * 2 + 1] = l;
  }
  if (a.hidden_rows && h == 0 && l == 0.f) atomicAdd(a.hidden_rows, 1);
  return true;
}

__device__ void edge_worker(AttnSmem& sm, const AttnArgs& a, uint32_t tmem, volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t q_taddr = tmem + kTmemQ + lane_off;
  const int G = gridDim.x;
  int round = 0;
  // the CTA's next item with key tiles; items without any are answered on the way
  auto next_item = [&](Item& out) -> bool {
    for (;; ++round) {
      const int idx = item_index(round, blockIdx.x, G);
      if (idx >= a.n_items) return false;
      out = make_item(a, idx);
      if (out.n > 0) {
        ++round;
        return true;
      }
      write_hidden_rows(a, out, r);
    }
  };
  // Q of the next item is computed into registers while the tensor cores work on the
  // current one, and stored into TMEM as soon as the current item's last S = Q K^T has
  // read Q; then the current item's epilogue runs once its last P V is done.
  uint32_t q[kDim / 2];
  Item cur, nxt;
  if (!next_item(cur)) return;
  prep_q_compute(sm, a, cur.h, cur.mt * kTileM + r, cur.mt * kTileM + r < a.rows, q);
  store_q_tmem(q, q_taddr);
  tc_fence_before();
  mbar_arrive(&sm.q_full);
  uint32_t it_done = 0;
  while (true) {
    const bool have_next = next_item(nxt);
    if (!a.weights_pass) prefetch_row(a, cur, r, 512);   // the current item's gates
    if (have_next) {
      prep_q_compute(sm, a, nxt.h, nxt.mt * kTileM + r, nxt.mt * kTileM + r < a.rows, q);
      if (!warp_wait(&sm.q_empty, it_done & 1, abort)) return;
      tc_fence_after();
      store_q_tmem(q, q_taddr);
      tc_fence_before();
      mbar_arrive(&sm.q_full);
    }
    if (!a.weights_pass && !epilogue(sm, a, cur, tmem, lane_off, r, it_done, abort)) return;
    ++it_done;
    if (!have_next) break;
    cur = nxt;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &sm.abort;
  if (threadIdx.x == 0) {
    sm.abort = 0;
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    mbar_init(&sm.q_full, 128);
    mbar_init(&sm.q_empty, 1);
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_free, 128);
    mbar_init(&sm.p_full, 128);
    mbar_init(&sm.p_empty, 1);
    mbar_init(&sm.o_ready, 1);
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.o_free, 128);
    mbar_init(&sm.st_full, 128);
    mbar_init(&sm.st_empty, 128);
    mbar_init(&sm.drain, 1);
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (threadIdx.x < kDim / 8) sm.w_q[threadIdx.x] = __ldg(reinterpret_cast<const uint4*>(a.w_q) + threadIdx.x);
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue));
    if (warp == 0 && lane == 0) producer(sm, &tm_k, &tm_v, a, abort);
    if (warp == 1 && lane == 0) mma_issuer(sm, a, tmem, abort);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsWork));
    if (warp < 8) softmax_worker(sm, a, tmem, abort);
    else edge_worker(sm, a, tmem, abort);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && sm.abort) record_abort(a.status, sm.abort);
}

}  // namespace

size_t attn_smem_bytes() { return sizeof(AttnSmem) + 1024; }

cudaError_t attn_set_smem_attribute() {
  return cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)attn_smem_bytes());
}

cudaError_t launch_attn(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const AttnArgs& a,
                        int grid, cudaStream_t s) {
  attn_kernel<<<grid, kThreads, attn_smem_bytes(), s>>>(tm_k, tm_v, a);
  return cudaGetLastError();
}

}  // namespace ga
