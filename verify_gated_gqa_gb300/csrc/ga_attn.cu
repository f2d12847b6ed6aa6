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
// Structure (one CTA per SM, persistent, 192 threads):
//   warp 0     TMA producer: K and V tiles of 64 keys in 8 KiB chunks (64 keys x 64 dims,
//              128-byte swizzle) through a 28-slot ring (224 KiB) of shared memory;
//   warp 1     allocates the 512 TMEM columns and issues every tcgen05.mma:
//              S = Q K^T (M=128, N=64, K=256; Q read from TMEM) into one of two TMEM S
//              buffers, then O += P V (P read from TMEM over S, V MN-major, N=64 a chunk);
//   warps 2-5  one query row per thread: Q prep (norm, RoPE) straight into TMEM, the
//              softmax over each S tile (P written back over S in TMEM), the rare O
//              rescale, and the gated epilogue with 16-byte bf16 stores. The next work
//              item's Q is prepared before the current item's epilogue, so the tensor
//              core starts the next item's S = Q K^T while O is drained.
// Tensor memory (512 columns x 128 lanes, lane = query row): O [0, 256) fp32, Q
// [256, 384) bf16 pairs, S0 [384, 448) and S1 [448, 512) fp32 with P as bf16 pairs over
// their first 32 columns. Keeping Q in TMEM leaves shared memory to the K/V ring, which
// is what keeps enough loads in flight to cover the L2 latency.
// Work items are (query head, 128-row tile), longest first, dealt to the CTAs in a
// serpentine order so each CTA's total work evens out.
#include "ga_internal.h"
#include "ga_numerics.cuh"
#include "ga_sm100.cuh"

namespace ga {
namespace {

constexpr int kSlots = 28;
constexpr int kChunkBytes = kTileN * 128;  // 64 keys x 64 bf16 (one 128-byte-swizzle column)
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;      // O accumulator: 256 columns (fp32)
constexpr uint32_t kTmemQ = 256;    // Q: 128 columns of bf16 pairs (A operand of Q K^T)
constexpr uint32_t kTmemS = 384;    // S buffers: 2 x 64 columns; P (bf16 pairs) over S
constexpr uint32_t kSCols = kTileN; // fp32 columns of one S buffer
constexpr float kLog2eOver16 = 1.4426950408889634f / 16.0f;
constexpr int kLazyRescale = 8;     // rescale when the tile maximum exceeds M by > 2^8

struct alignas(1024) AttnSmem {
  uint8_t ring[kSlots][kChunkBytes];
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  uint64_t q_full, q_empty, o_ready, o_done, o_free;
  uint64_t s_full[2], p_full[2];
  uint64_t drain;
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

__device__ __forceinline__ void record_abort(int* status, int code) {
  if (code) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------ warp 0: producer
__device__ void producer_loop(AttnSmem& sm, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                              const AttnArgs& a, volatile int* abort, uint32_t& chunk) {
  auto load_tile = [&](const CUtensorMap* map, int kvh, int kt) -> bool {
    for (int c = 0; c < 4; ++c) {
      const uint32_t slot = chunk % kSlots;
      const uint32_t phase = (chunk / kSlots) & 1;
      if (!mbar_wait(&sm.empty[slot], phase ^ 1, abort)) return false;
      mbar_expect_tx(&sm.full[slot], kChunkBytes);
      tma_load_3d(sm.ring[slot], map, &sm.full[slot], c * 64, kvh, kt * kTileN);
      ++chunk;
    }
    return true;
  };
  const int G = gridDim.x;
  for (int round = 0;; ++round) {
    const int idx = item_index(round, blockIdx.x, G);
    if (idx >= a.n_items) break;
    const Item it = make_item(a, idx);
    if (it.n == 0) continue;
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
  uint32_t chunk = 0;
  producer_loop(sm, tm_k, tm_v, a, abort, chunk);
  if (*abort) {
    // let the loads already issued into the last kSlots slots land before exit
    const uint32_t first = chunk > (uint32_t)kSlots ? chunk - kSlots : 0;
    for (uint32_t c = first; c < chunk; ++c)
      mbar_wait_quiet(&sm.full[c % kSlots], (c / kSlots) & 1, 100000000LL);
  }
}

// ------------------------------------------------------------------ warp 1: MMA issuer
__device__ void mma_loop(AttnSmem& sm, const AttnArgs& a, uint32_t tmem,
                         volatile int* abort) {
  constexpr uint32_t kIdQK = idesc_bf16(128, kTileN, false, false);
  constexpr uint32_t kIdPV = idesc_bf16(128, 64, false, true);
  uint32_t chunk = 0;
  uint32_t g = 0;   // global tile counter (selects the S buffer and its phase)
  uint32_t it_done = 0;

  auto take_chunk = [&](uint32_t& slot) -> bool {
    slot = chunk % kSlots;
    if (!mbar_wait(&sm.full[slot], (chunk / kSlots) & 1, abort)) return false;
    tc_fence_after();
    ++chunk;
    return true;
  };
  auto issue_pv = [&](int j, uint32_t gj) -> bool {
    const uint32_t b = gj & 1, u = gj >> 1;
    if (j == 0 && it_done > 0 && !mbar_wait(&sm.o_free, (it_done - 1) & 1, abort)) return false;
    if (!mbar_wait(&sm.p_full[b], u & 1, abort)) return false;
    tc_fence_after();
    const uint32_t p_tmem = tmem + kTmemS + b * kSCols;
    for (int c = 0; c < 4; ++c) {
      uint32_t slot;
      if (!take_chunk(slot)) return false;
      const uint32_t v_addr = smem_u32(sm.ring[slot]);
      for (int kk = 0; kk < kTileN / 16; ++kk) {
        const uint64_t bd = sdesc_sw128(v_addr + kk * 2048, kChunkBytes, 1024);
        umma_ts(tmem + kTmemO + c * 64, p_tmem + kk * 8, bd, kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(&sm.empty[slot]);
    }
    umma_commit(&sm.o_ready);
    return true;
  };

  const int G = gridDim.x;
  for (int round = 0;; ++round) {
    const int idx = item_index(round, blockIdx.x, G);
    if (idx >= a.n_items) break;
    const Item it = make_item(a, idx);
    if (it.n == 0) continue;
    if (!mbar_wait(&sm.q_full, it_done & 1, abort)) return;
    tc_fence_after();
    for (int j = 0; j < it.n; ++j, ++g) {
      const uint32_t b = g & 1;
      if (a.weights_pass && g >= 2) {
        // S buffer b is free once the rows have read tile g-2 from it
        if (!mbar_wait(&sm.p_full[b], ((g >> 1) - 1) & 1, abort)) return;
      }
      const uint32_t s_tmem = tmem + kTmemS + b * kSCols;
      for (int c = 0; c < 4; ++c) {
        uint32_t slot;
        if (!take_chunk(slot)) return;
        const uint32_t k_addr = smem_u32(sm.ring[slot]);
        for (int k4 = 0; k4 < 4; ++k4) {
          const uint64_t bd = sdesc_sw128(k_addr + k4 * 32, 16, 1024);
          umma_ts(s_tmem, tmem + kTmemQ + (c * 4 + k4) * 8, bd, kIdQK, (c | k4) ? 1u : 0u);
        }
        umma_commit(&sm.empty[slot]);
      }
      umma_commit(&sm.s_full[b]);
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

// ------------------------------------------------------------------ warps 2-5: rows
__device__ __forceinline__ float lo_f(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hi_f(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return (uint32_t)bf16_bits(a) | ((uint32_t)bf16_bits(b) << 16);
}

// Normalise one 16-byte chunk (8 dims) of a row: bf16((x * r) * (1 + w)).
__device__ __forceinline__ void norm_chunk(const uint4& xv, const uint4& wv, float r32,
                                           const SumSq& ss, float (&y)[8]) {
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    y[2 * k] = norm_elem(lo_f(xw[k]), lo_f(ww[k]), r32, ss);
    y[2 * k + 1] = norm_elem(hi_f(xw[k]), hi_f(ww[k]), r32, ss);
  }
}

// (1+w) RMSNorm and partial RoPE of one query row, written as bf16 pairs into this
// thread's TMEM lane at Q (column c holds dims 2c and 2c+1). Every lane of the warp runs
// it (the stores are warp-collective); lanes of rows past the end store zeros.
__device__ __noinline__ void prep_q_tmem(const AttnArgs& a, int h, int row, bool valid,
                                         uint32_t q_taddr) {
  const uint4* src = reinterpret_cast<const uint4*>(a.qg + ((size_t)(valid ? row : 0) * kHeads + h) * kQgStride);
  const uint4* wq = reinterpret_cast<const uint4*>(a.w_q);
  SumSq ss;
  float r32 = 0.f;
  if (valid) {
    SumSq acc[4];
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
      const uint4 v = __ldg(src + i);
      acc[i & 3].add(lo_f(v.x)); acc[i & 3].add(hi_f(v.x));
      acc[i & 3].add(lo_f(v.y)); acc[i & 3].add(hi_f(v.y));
      acc[i & 3].add(lo_f(v.z)); acc[i & 3].add(hi_f(v.z));
      acc[i & 3].add(lo_f(v.w)); acc[i & 3].add(hi_f(v.w));
    }
    acc[0].merge(acc[1]);
    acc[2].merge(acc[3]);
    acc[0].merge(acc[2]);
    ss = acc[0];
    r32 = inv_rms_f32(ss);
  }
  uint32_t w[32];
  // dims 0..63: chunk c (dims 8c..8c+7) pairs with chunk c + 4 (dims 8c+32..)
  if (valid) {
    const int pos = a.q_base + row;
    const uint4* cp = reinterpret_cast<const uint4*>(a.cos_tab + (size_t)pos * kHalfRot);
    const uint4* sp = reinterpret_cast<const uint4*>(a.sin_tab + (size_t)pos * kHalfRot);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float ya[8], yb[8];
      norm_chunk(__ldg(src + c), __ldg(wq + c), r32, ss, ya);
      norm_chunk(__ldg(src + c + 4), __ldg(wq + c + 4), r32, ss, yb);
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
        w[4 * c + k] = pack2(ya[2 * k], ya[2 * k + 1]);
        w[16 + 4 * c + k] = pack2(yb[2 * k], yb[2 * k + 1]);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k) w[k] = 0u;
  }
  tmem_st32(q_taddr, w);
  // dims 64..255 pass through the rotation
#pragma unroll 1
  for (int grp = 1; grp < 4; ++grp) {
    if (valid) {
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float y[8];
        norm_chunk(__ldg(src + 8 * grp + cc), __ldg(wq + 8 * grp + cc), r32, ss, y);
#pragma unroll
        for (int k = 0; k < 4; ++k) w[4 * cc + k] = pack2(y[2 * k], y[2 * k + 1]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) w[k] = 0u;
    }
    tmem_st32(q_taddr + 32 * grp, w);
  }
  tmem_wait_st();
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

// Visibility of the 32 keys kt*64 + 32*ch .. +31 for one row: bit k <-> key +k.
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

// Hidden keys read as -inf: their weight is exactly 0 and they never raise the maximum.
__device__ __forceinline__ void mask_chunk(uint32_t (&s)[32], uint32_t vis) {
  if (vis != 0xFFFFFFFFu) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (!((vis >> k) & 1u)) s[k] = 0xFF800000u;
  }
}

// Weights pass: bf16(bf16(2^(t - M)) / l) for visible keys, with the main pass's final M
// and l, written to weights[h][row][kt*64 ..]. Every lane of the warp runs it (the TMEM
// loads are warp-collective); only lanes with `active` compute and store.
__device__ void weights_tile(const AttnArgs& a, uint32_t s_tmem, int h, int row, int kt, int M,
                             float l_final, bool active) {
  const float mf = (float)M;
  uint16_t* wrow = a.weights + ((size_t)h * a.rows + row) * (size_t)a.T + (size_t)kt * kTileN;
  const int ncol = min(kTileN, a.T - kt * kTileN);
  const bool vec = (ncol == kTileN) && ((a.T & 7) == 0);
#pragma unroll 1
  for (int ch = 0; ch < kTileN / 32; ++ch) {
    uint32_t s[32];
    tmem_ld32(s_tmem + ch * 32, s);
    tmem_wait_ld(s);
    if (!active) continue;
    mask_chunk(s, chunk_visibility(a, row, kt, ch, true));
    uint32_t pk[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t sb = pack_bf16x2(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1]));
      const float p0 = bf16_round(ex2_approx(fmaf(lo_f(sb), kLog2eOver16, -mf)));
      const float p1 = bf16_round(ex2_approx(fmaf(hi_f(sb), kLog2eOver16, -mf)));
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

// Wait in all 32 lanes and agree on the outcome, so that the warp-collective TMEM loads and
// stores that follow always run with the whole warp (or the whole warp leaves).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

__device__ void row_worker(AttnSmem& sm, const AttnArgs& a, uint32_t tmem, volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t q_taddr = tmem + kTmemQ + lane_off;
  uint32_t g = 0, it_done = 0;
  const int G = gridDim.x;
  int round = 0;

  // This CTA's next work item that has key tiles; items without any (mask mode) are
  // answered on the way.
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

  Item it;
  if (!next_item(it)) return;
  prep_q_tmem(a, it.h, it.mt * kTileM + r, it.mt * kTileM + r < a.rows, q_taddr);
  tc_fence_before();
  mbar_arrive(&sm.q_full);
  while (true) {
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
      const uint32_t b = g & 1;
      const uint32_t s_tmem = tmem + kTmemS + b * kSCols + lane_off;
      if (!warp_wait(&sm.s_full[b], (g >> 1) & 1, abort)) return;
      tc_fence_after();
      if (a.weights_pass) {
        weights_tile(a, s_tmem, h, row, kt, M, l_final, valid && hasM);
        tc_fence_before();
        mbar_arrive(&sm.p_full[b]);
        continue;
      }
      // pass 1: the tile maximum over the visible raw fp32 scores (bf16 rounding is
      // monotone, so the rounded maximum is the maximum of the rounded scores)
      float mx = -INFINITY;
#pragma unroll 1
      for (int ch = 0; ch < kTileN / 32; ++ch) {
        uint32_t s[32];
        tmem_ld32(s_tmem + ch * 32, s);
        tmem_wait_ld(s);
        mask_chunk(s, chunk_visibility(a, row, kt, ch, valid));
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          m0 = fmaxf(m0, __uint_as_float(s[k]));
          m1 = fmaxf(m1, __uint_as_float(s[k + 1]));
          m2 = fmaxf(m2, __uint_as_float(s[k + 2]));
          m3 = fmaxf(m3, __uint_as_float(s[k + 3]));
        }
        mx = fmaxf(mx, fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)));
      }

      bool rescale = false;
      int newM = M;
      if (mx != -INFINITY) {
        const int need = (int)ceilf(bf16_round(mx) * kLog2eOver16);
        if (!hasM) {
          newM = need;
          hasM = true;
        } else if (need > M + kLazyRescale) {
          newM = need;
          rescale = true;
        }
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O must hold every earlier P.V before it is scaled (PV of global tile g-1)
        if (!warp_wait(&sm.o_ready, (g - 1) & 1, abort)) return;
        tc_fence_after();
        const float f = rescale ? exp2f((float)(M - newM)) : 1.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 32) {
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
      // pass 2: P = bf16(2^(t - M)), t = bf16(s) * log2(e) / 16, written back as bf16 pairs
      // over the S columns this pass has already read; l sums the rounded P
#pragma unroll 1
      for (int ch = 0; ch < kTileN / 32; ++ch) {
        uint32_t s[32];
        tmem_ld32(s_tmem + ch * 32, s);
        tmem_wait_ld(s);
        mask_chunk(s, chunk_visibility(a, row, kt, ch, valid));
        uint32_t pk[16];
        float la = 0.f, lb = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint32_t sb = pack_bf16x2(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1]));
          const float p0 = ex2_approx(fmaf(lo_f(sb), kLog2eOver16, -mf));
          const float p1 = ex2_approx(fmaf(hi_f(sb), kLog2eOver16, -mf));
          pk[k] = pack_bf16x2(p0, p1);
          la += lo_f(pk[k]);
          lb += hi_f(pk[k]);
        }
        l += la + lb;
        tmem_st16(s_tmem + ch * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sm.p_full[b]);
    }

    // ---- the next item's Q, as soon as this item's last S = Q K^T has read Q
    Item nxt;
    const bool more = next_item(nxt);
    if (more) {
      if (!warp_wait(&sm.q_empty, it_done & 1, abort)) return;
      tc_fence_after();
      prep_q_tmem(a, nxt.h, nxt.mt * kTileM + r, nxt.mt * kTileM + r < a.rows, q_taddr);
      tc_fence_before();
      mbar_arrive(&sm.q_full);
    }
    if (!a.weights_pass) {
      // ---- gated epilogue: out = bf16(bf16(O / l) * bf16(sigmoid(gate)))
      if (!warp_wait(&sm.o_done, it_done & 1, abort)) return;
      tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      const uint4* gp = reinterpret_cast<const uint4*>(a.qg + ((size_t)(valid ? row : 0) * kHeads + h) * kQgStride + kDim);
      uint4* op = reinterpret_cast<uint4*>(a.out + (size_t)(valid ? row : 0) * kOutRow + h * kDim);
  #pragma unroll 1
      for (int c0 = 0; c0 < 256; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + kTmemO + lane_off + c0, o);
        tmem_wait_ld(o);
        if (valid) {
          uint32_t res[16];
  #pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const uint4 gv = __ldg(gp + (c0 >> 3) + q4);
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
  #pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int e = q4 * 8 + 2 * k;
              const float o0 = bf16_round(__uint_as_float(o[e]) * inv);
              const float o1 = bf16_round(__uint_as_float(o[e + 1]) * inv);
              res[q4 * 4 + k] = pack2(o0 * sigmoid_bf16(lo_f(gw[k])), o1 * sigmoid_bf16(hi_f(gw[k])));
            }
          }
  #pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            op[(c0 >> 3) + q4] = make_uint4(res[4 * q4], res[4 * q4 + 1], res[4 * q4 + 2], res[4 * q4 + 3]);
        }
      }
      if (valid) {
        if (a.row_stats) {
          a.row_stats[((size_t)h * a.rows + row) * 2] = (float)M;
          a.row_stats[((size_t)h * a.rows + row) * 2 + 1] = l;
        }
        if (a.hidden_rows && h == 0 && l == 0.f) atomicAdd(a.hidden_rows, 1);
      }
      tc_fence_before();
      mbar_arrive(&sm.o_free);
    }
    ++it_done;
    if (!more) break;
    it = nxt;
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
    mbar_init(&sm.o_ready, 1);
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.o_free, 128);
    mbar_init(&sm.drain, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 128);
    }
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    if (lane == 0) producer(sm, &tm_k, &tm_v, a, abort);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer(sm, a, tmem, abort);
  } else {
    row_worker(sm, a, tmem, abort);
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
