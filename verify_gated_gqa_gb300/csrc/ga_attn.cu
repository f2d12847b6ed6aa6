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
// Structure (one CTA per SM, persistent, 512 threads in four warpgroups):
//   warp 0     TMA producer: each item's prepared Q tile and gate tile (the gate halves of
//              its fused rows), then its K and V tiles of 128 keys x 256 dims (64 KiB, four
//              16 KiB 128-byte-swizzled column blocks), through three tile slots (the whole
//              warp runs the loop, one elected lane issues the copies);
//   warp 1     allocates the 512 TMEM columns and issues every S = Q K^T (M=128, N=128,
//              K=256; Q dims 0..127 read from TMEM, dims 128..255 from shared memory);
//   warp 2     issues every O += P V (M=128, N=256, K=128; P from tensor memory, V
//              MN-major), so a tile's P V need not wait behind the next tile's Q K^T
//              issue. Both at full rate (N >= 128); in each, the whole warp runs the issue
//              loop and one elected lane issues (a lone lane in a divergent branch issued
//              too slowly to keep the N=128 MMAs back to back);
//   warps 4-11 softmax, two warpgroups, one per 64-key half of each S tile, one query row
//              per thread: S is copied to registers and its TMEM columns released at once
//              (so the next S = Q K^T overlaps this softmax); the two halves exchange their
//              row maxima through shared memory and take the same M; P = bf16(2^(t - M))
//              goes to tensor memory, each half its own 64 keys (and the tensor cores read
//              each half as soon as it is written), and each half rescales its half of O
//              when needed;
//   warps 12-15 the edge of each work item: the current item's gate tile from its ring
//              slot into registers and its bf16 sigmoids while the item's tiles run, the
//              next item's prepared Q tile (normed and rotated by the query prologue) into
//              TMEM as soon as the current item's last S = Q K^T has read Q, then the gated
//              epilogue of the current item.
// The edge code is kept in short loops: the four roles run different code at once and
// share the SM's instruction cache, which long unrolled sequences would overflow.
// Over e4m3 caches (verify), the kernel runs as clusters of two CTAs, one per half of a
// query group, that walk the same key tiles: each CTA loads the e4m3 codes of its 64 keys of
// a K or V tile into the back of its slot, widens them to bf16(fp32(code * scale)) and
// writes the bf16 rows into its own slot and into its peer's (distributed shared memory),
// so every code is widened once; the MMA warps wait until both halves are in.
// Tensor memory (512 columns x 128 lanes, lane = query row): O [0, 256) fp32, S [256, 384)
// fp32, Q dims 0..127 [384, 448) and P [448, 512) as bf16 pairs. Q dims 128..255 stay in
// shared memory for the item, where P used to go: P is written to tensor memory with one
// store per thread and read from there by the P V MMAs.
// Work items are (query head, 128-row tile), longest first, dealt to the CTAs in a
// serpentine order so each CTA's total work evens out. The kernel is compiled once per
// visibility mode (causal, bidirectional, stored mask) and for the weights pass, so each
// variant carries only its own code.
#include <cuda_fp8.h>

#include "ga_internal.h"
#include "ga_numerics.cuh"
#include "ga_sm100.cuh"

namespace ga {
namespace {

constexpr int kSlots = 3;       // single CTAs: a ring of three 64 KiB slots (Q, gate, K, V tiles)
constexpr int kPairSlots = 4;   // CTA pairs: four 32 KiB slots for K and V halves, then a
                                // 64 KiB staging buffer (Q tiles, gate tiles, output tiles)
constexpr int kMaxSlots = 4;
// e4m3 caches: each CTA of a pair holds the codes of its 64 keys of a tile (64 x 256 bytes)
// until they are widened, in eight 2 KiB pieces of 8 keys, each inside rows that only one
// edge warp writes: edge warp w widens keys 16w .. 16w+15 of the CTA's half into bf16 rows
// 64 rank + 16w .. + 15 of the four 64-dim blocks, and its keys 16w + 8s .. + 7 wait in its
// rows of block 2 + s. A warp's writes then only ever cover its own codes.
constexpr int kRawKeys = 64;
constexpr int kRawBytes = kRawKeys * 256;
__device__ __forceinline__ uint32_t raw_piece_offset(int w, int s, uint32_t rank) {
  return (uint32_t)(2 + s) * 16384u + (rank * (uint32_t)kRawKeys + 16u * (uint32_t)w) * 128u;
}
constexpr int kChunkBytes = kTileN * 128;     // 128 keys x 64 dims of bf16
constexpr int kTileBytes = 4 * kChunkBytes;   // 128 keys x 256 dims
constexpr int kHalfTileBytes = kTileBytes / 2;   // a CTA pair: each CTA's half of a K or V tile
static_assert(kPairSlots * kHalfTileBytes + kTileBytes == kSlots * kTileBytes,
              "a pair's ring and staging buffer take the single ring's bytes");
template <bool kPair>
__host__ __device__ constexpr int ring_slots() { return kPair ? kPairSlots : kSlots; }
constexpr int kThreads = 512;     // four warpgroups
constexpr int kEdgeThread0 = 384; // first thread of the edge warpgroup (warps 12-15)
// Register split (setmaxnreg): the kernel is launched at kLaunchRegs per thread; the
// producer/MMA and softmax warpgroups give registers back and the edge warpgroup takes
// them. The shares add up to the launch total: 128*(64 + 2*112 + 224) = 512*128, and on
// each SM sub-partition (one warp of each warpgroup) 32*(64 + 2*112 + 224) = 16384.
constexpr int kLaunchRegs = 128;
constexpr int kRegsIssue = 64;
constexpr int kRegsSoftmax = 112;
constexpr int kRegsEdge = 224;
static_assert(128 * (kRegsIssue + 2 * kRegsSoftmax + kRegsEdge) == kThreads * kLaunchRegs,
              "register split");
constexpr int kHalfKeys = kTileN / 2;   // keys per softmax warpgroup in a tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;      // O accumulator: 256 columns (fp32)
constexpr uint32_t kTmemS = 256;    // S: 128 columns (fp32)
constexpr uint32_t kTmemQ = 384;    // Q dims 0..127: 64 columns of bf16 pairs (A of Q K^T)
constexpr uint32_t kTmemP = 448;    // P: 64 columns of bf16 pairs, 32 per 64-key half (A of P V)
constexpr float kLog2eOver16 = 1.4426950408889634f / 16.0f;
constexpr int kLazyRescale = 8;     // rescale when the tile maximum exceeds M by > 2^8

// Items of the gated passes (causal, bidirectional, stored mask) carry a gate tile in the
// ring; the weights pass and the verify partials have no gated epilogue.
// Few-row verify windows, over bf16 or e4m3 caches: the same items, softmax and partials.
template <int kMode>
__host__ __device__ constexpr bool is_verify() { return kMode == kModeVerify || kMode == kModeVerify8; }

template <int kMode, bool kW>
__host__ __device__ constexpr bool has_gate() { return !kW && !is_verify<kMode>(); }

static_assert(kTileN == 128, "this kernel is laid out for 128-key tiles");

struct AttnSmem {
  uint8_t tile[kSlots][kTileBytes];   // K or V tiles (1024-byte aligned)
  uint8_t qhi[2][kChunkBytes];        // Q dims 128..255 of the item: two swizzled 64-dim blocks
  float stat_l[2][kTileM];            // softmax -> edge: each half's row sum l of the item
  float stat_m[kTileM];               // and the running maximum M
  uint16_t mx[2][2][kTileM];          // tile g: each half's row maximum (bf16 bits), by g % 2
  uint64_t full[kMaxSlots], empty[kMaxSlots];
  uint64_t conv[kSlots];              // e4m3 caches: the slot's tile is widened (or seen: Q)
  uint64_t peer_free[kSlots];         // e4m3 caches: the peer's slot is free for the next fill
  uint64_t q_full, q_empty, s_full, s_free;
  uint64_t p_full[2], p_empty[2];     // per 64-key half of P
  uint64_t o_done, o_free, st_full, st_empty, drain, drain_pv, q_read, g_read, mx_bar;
  uint64_t stg_full, stg_empty, o_st;   // CTA pairs: the staging buffer, the output tile in it
  uint32_t tmem_base;
  int abort;
};

// A ring slot's bytes: slot s of the single ring, or of a pair's ring of half tiles; a pair's
// staging buffer follows its ring.
template <bool kPair>
__device__ __forceinline__ uint8_t* slot_ptr(AttnSmem& sm, uint32_t s) {
  return reinterpret_cast<uint8_t*>(sm.tile) + s * (uint32_t)(kPair ? kHalfTileBytes : kTileBytes);
}
__device__ __forceinline__ uint8_t* staging_ptr(AttnSmem& sm) {
  return reinterpret_cast<uint8_t*>(sm.tile) + kPairSlots * kHalfTileBytes;
}

// ------------------------------------------------------------------ work items
struct Item {
  int h, mt;          // query head (verify: the first query head of the half), 128-row tile
  int n;              // key tiles to visit
  int seq, half, kt0; // verify: sequence, half of the query group, first key tile of the chunk
                      // (batch: seq is the item's sequence)
  int row0, rows, qb, T;  // the item's sequence: first (packed) row, rows, position of its
                          // row 0 (q_base), keys; the call's own values outside batch mode
  uint64_t tiles[2];  // mask mode: bit kt set for every key tile with a visible key
};

// Causal visibility (key j <= position of the row), for one sequence or a batch of them.
template <int kMode>
__host__ __device__ constexpr bool is_causal() { return kMode == kModeCausal || kMode == kModeBatch; }

__device__ __forceinline__ int item_index(int round, int cta, int G) {
  return round * G + ((round & 1) ? (G - 1 - cta) : cta);
}

// The item a CTA takes in a round. Over e4m3 caches the CTAs run in clusters of two (ranks
// blockIdx.x % 2): the pair takes the items 2p and 2p + 1, the two halves of one query
// group over the same key chunk, the pairs dealt like single items. CTA pairs of the
// gated passes (kPair) deal pair items to the clusters; both CTAs take the same one.
template <int kMode, bool kPair = false>
__device__ __forceinline__ int walk_index(int round) {
  if (kMode == kModeVerify8)
    return 2 * item_index(round, blockIdx.x >> 1, gridDim.x >> 1) + (blockIdx.x & 1);
  if (kPair) return item_index(round, blockIdx.x >> 1, gridDim.x >> 1);
  return item_index(round, blockIdx.x, gridDim.x);
}

// CTA pairs (kPair): item idx is (row tile, pair of neighbouring query heads of one KV
// group); the even CTA of the cluster takes the first head, the odd one the second, so
// both walk the same key tiles under the same visibility.
template <int kMode, bool kPair = false>
__device__ __forceinline__ Item make_item(const AttnArgs& a, int idx) {
  Item it;
  it.seq = it.half = it.kt0 = 0;
  it.tiles[0] = it.tiles[1] = 0;
  it.row0 = 0;
  it.rows = a.rows;
  it.qb = a.q_base;
  it.T = a.T;
  if (kMode == kModeBatch) {
    const int per_entry = kPair ? kHeads / 2 : kHeads;
    const uint32_t e = a.batch_entry[idx / per_entry];
    const int piece = (int)(e >> 16);
    it.h = kPair ? 2 * (idx % per_entry) + (int)(blockIdx.x & 1) : idx % kHeads;
    it.mt = (int)(e & 0xFFFFu);
    it.seq = a.batch_seq[piece];
    it.row0 = a.batch_row0[piece];
    it.rows = a.batch_rows[piece];
    it.qb = a.batch_qbase[piece];
    it.T = it.qb + it.rows;
    const int last_row = min(it.rows, (it.mt + 1) * kTileM) - 1;
    it.n = (it.qb + last_row + 1 + kTileN - 1) / kTileN;
    return it;
  }
  if (is_verify<kMode>()) {
    // (chunk, sequence, KV head, half): the two halves of a query group are neighbours, so
    // the CTAs that run them read each K/V tile at about the same time (the second from L2)
    it.half = idx & 1;
    const int kvh = (idx >> 1) & 1;
    const int rest = idx >> 2;
    it.seq = rest % a.n_seq;
    const int c = rest / a.n_seq;
    it.h = kvh * kGroup + kVerifyHeadsPerTile * it.half;
    it.mt = 0;
    it.kt0 = c * a.chunk_tiles;
    const int tiles = (a.seq_len[it.seq] + a.vrows + kTileN - 1) / kTileN;
    it.n = max(0, min(a.chunk_tiles, tiles - it.kt0));
    return it;
  }
  const int per_tile = kPair ? a.n_heads / 2 : a.n_heads;
  it.mt = a.row_tiles - 1 - idx / per_tile;  // later row tiles see more keys: longest first
  it.h = a.head0 + (kPair ? 2 * (idx % per_tile) + (int)(blockIdx.x & 1) : idx % per_tile);
  if (kMode == kModeCausal) {
    const int last_row = min(a.rows, (it.mt + 1) * kTileM) - 1;
    const int key_end = min(a.T, a.q_base + last_row + 1);
    it.n = (key_end + kTileN - 1) / kTileN;
  } else if (kMode == kModeBidir) {
    it.n = (a.T + kTileN - 1) / kTileN;
  } else {
    // the row tile's 64 flag bytes (0 or 1 each) in four 16-byte loads; each word's four
    // flags become four bits by one multiply (the products land on distinct bits, so no
    // carry joins them)
    static_assert(kMaskFlagStride == 64, "one 64-bit tile map per row tile");
    const uint4* f = reinterpret_cast<const uint4*>(a.tile_flags + (size_t)it.mt * kMaskFlagStride);
    uint64_t m = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(f + q);
      const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        m |= (uint64_t)((((wd[i] & 0x01010101u) * 0x00204081u) >> 21) & 0xFu) << (16 * q + 4 * i);
    }
    if (a.key_tiles < 64) m &= (1ull << a.key_tiles) - 1ull;
    it.tiles[0] = m;
    it.n = __popcll(m);
  }
  return it;
}

// Walks the key tiles of an item in order: 0 .. n-1, or the set bits of a mask-mode item.
template <int kMode>
struct TileCursor {
  uint64_t w0, w1;
  int base;
  __device__ __forceinline__ explicit TileCursor(const Item& it)
      : w0(it.tiles[0]), w1(it.tiles[1]), base(it.kt0) {}
  __device__ __forceinline__ int next(int j) {
    if (kMode != kModeMask) return base + j;
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
template <int kMode, bool kPair = false>
struct ItemWalk {
  int round = 0;
  __device__ __forceinline__ bool next(const AttnArgs& a, Item& out) {
    for (;; ++round) {
      const int idx = walk_index<kMode, kPair>(round);
      if (idx >= a.n_items) return false;
      out = make_item<kMode, kPair>(a, idx);
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

// Wait in all 32 lanes and agree on the outcome, so that the warp-collective TMEM loads and
// stores (and elected MMA issues) that follow always run with the whole warp (or the whole warp leaves).
// kCluster: acquire at cluster scope, for barriers that the peer CTA of a pair arrives on.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait<kCluster>(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// The MMA issue and commit forms of a single CTA or of a CTA pair (cta_group::2).
template <bool kPair>
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
  if (kPair) umma_ts_pair_warp(d, a, b, id, acc);
  else umma_ts_warp(d, a, b, id, acc);
}
template <bool kPair>
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  if (kPair) umma_ss_pair_warp(d, a, b, id, acc);
  else umma_ss_warp(d, a, b, id, acc);
}
// A pair's commit arrives on the barrier of both CTAs.
template <bool kPair>
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  if (kPair) umma_commit_pair_both_warp(bar);
  else umma_commit_warp(bar);
}
// One arrival on a barrier the MMA warps wait on: per thread in a single CTA and in a
// pair's even CTA (whose barriers they are); per warp, remotely, from a pair's odd CTA
// (kRelease: at cluster scope, after generic shared-memory writes the pair's MMAs read).
template <bool kPair, bool kRelease = false>
__device__ __forceinline__ void arrive_for_mma(uint64_t* bar) {
  if (!kPair || (blockIdx.x & 1) == 0) {
    mbar_arrive(bar);
    return;
  }
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    if (kRelease) mbar_arrive_remote(mapa_shared(smem_u32(bar), 0));
    else mbar_arrive_remote_cta(mapa_shared(smem_u32(bar), 0));
  }
}

// ------------------------------------------------------------------ warp 0: producer
template <int kMode, bool kW, bool kPair>
__device__ void producer_loop(AttnSmem& sm, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                              const CUtensorMap* tm_v, const CUtensorMap* tm_g, const AttnArgs& a,
                              volatile int* abort, uint32_t& cnt) {
  // One tile into the next slot. A Q tile is four 64-dim boxes at (dim, head, row r0), a
  // verify Q tile 6 heads x vrows rows per box; a gate tile four 64-value boxes of the
  // fused rows at (256 + dim, head, row r0); a K or V tile is one copy of all four 64-dim
  // blocks (the key/value map lists the block index as its outermost dimension, so the box
  // lands as four consecutive 16 KiB blocks) at (0, key r0, head, 0[, sequence]).
  const int lane = threadIdx.x & 31;
  auto load_tile = [&](const CUtensorMap* map, bool kv, int head, int r0, int seq,
                       uint32_t bytes, int x0 = 0) -> bool {
    const uint32_t slot = cnt % kSlots;
    if (!warp_wait(&sm.empty[slot], ((cnt / kSlots) & 1) ^ 1, abort)) return false;
    if (kMode == kModeVerify8 && lane == 0)   // the peer may copy into this slot's next fill
      mbar_arrive_remote(mapa_shared(smem_u32(&sm.peer_free[slot]), (blockIdx.x & 1) ^ 1u));
    mbar_expect_tx_warp(&sm.full[slot], bytes);
    if (kv) {
      if (seq < 0)
        tma_load_4d_warp(sm.tile[slot], map, &sm.full[slot], 0, r0, head, 0);
      else if (kMode == kModeVerify)   // read by this query group's two CTAs only: evicted first
        tma_load_5d_warp_evict_first(sm.tile[slot], map, &sm.full[slot], 0, r0, head, 0, seq);
      else
        tma_load_5d_warp(sm.tile[slot], map, &sm.full[slot], 0, r0, head, 0, seq);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tma_load_3d_warp(sm.tile[slot] + c * kChunkBytes, map, &sm.full[slot], x0 + c * 64, head,
                         r0);
    }
    ++cnt;
    return true;
  };
  ItemWalk<kMode, kPair> walk;
  Item it;
  while (walk.next(a, it)) {
    const int kvh = it.h / kGroup;
    TileCursor<kMode> ck(it), cv(it);
    // Coordinates of key tile kt: token r0 and outer index (verify: the sequence, or with
    // paged caches the page; -1 for the four-dimensional prefill map). For paged caches
    // the warp holds a window of 32 consecutive page-table entries, one per lane, so one
    // coalesced read serves 32 entries. An entry outside the pool is recorded in the
    // status word and its tile read past the pool's end, which yields zeros.
    int win0 = -1, win_page = 0;
    auto kv_at = [&](int kt, int& r0) -> int {
      if (!is_verify<kMode>() && kMode != kModeBatch) {
        r0 = kt * kTileN;
        return -1;
      }
      if (a.page_table == nullptr) {
        r0 = kt * kTileN;
        return it.seq;
      }
      const int e = kt / a.page_tiles;
      r0 = (kt - e * a.page_tiles) * kTileN;
      if (win0 < 0 || e < win0 || e >= win0 + 32) {
        win0 = e;
        const int idx = e + lane;
        win_page = idx < a.max_pages ? __ldg(a.page_table + (size_t)it.seq * a.max_pages + idx) : 0;
      }
      int page = __shfl_sync(0xffffffffu, win_page, e - win0);
      if (page < 0 || page >= a.n_pages) {
        if (lane == 0) record_abort(a.status, kDevBadPage);
        page = a.n_pages;
      }
      return page;
    };
    // e4m3 caches: this CTA's 64 keys of the tile (eight boxes of 8 keys x 256 bytes) into
    // its edge warps' rows of the slot, where they widen them (and copy them to the peer)
    auto load_raw8 = [&](const CUtensorMap* map, int kt) -> bool {
      const uint32_t slot = cnt % kSlots;
      const uint32_t rank = blockIdx.x & 1;
      if (!warp_wait(&sm.empty[slot], ((cnt / kSlots) & 1) ^ 1, abort)) return false;
      if (lane == 0)   // the peer may copy into this slot's next fill
        mbar_arrive_remote(mapa_shared(smem_u32(&sm.peer_free[slot]), rank ^ 1u));
      mbar_expect_tx_warp(&sm.full[slot], kRawBytes);
#pragma unroll
      for (int w = 0; w < 4; ++w)
#pragma unroll
        for (int piece = 0; piece < 2; ++piece)
          tma_load_4d_warp(sm.tile[slot] + raw_piece_offset(w, piece, rank), map, &sm.full[slot],
                           0, kvh, kt * kTileN + kRawKeys * (int)rank + 16 * w + 8 * piece, it.seq);
      ++cnt;
      return true;
    };
    // CTA pairs: this CTA's half of a K or V tile into a 32 KiB slot of the pair ring (K:
    // keys 64 rank .. + 63 of the tile, four 8 KiB blocks of 64 dims; V: dims 128 rank ..
    // + 127, two 16 KiB blocks of 128 keys). Its bytes complete on the even CTA's full
    // barrier, which expects both halves; the odd CTA's own barrier only counts the fill.
    auto load_half = [&](const CUtensorMap* map, bool is_v, int kt) -> bool {
      const uint32_t slot = cnt % kPairSlots;
      const uint32_t rank = blockIdx.x & 1;
      if (!warp_wait(&sm.empty[slot], ((cnt / kPairSlots) & 1) ^ 1, abort)) return false;
      if (rank == 0) mbar_expect_tx_warp(&sm.full[slot], 2 * kHalfTileBytes);
      else mbar_arrive_elect_warp(&sm.full[slot]);
      const uint32_t bar = mapa_shared(smem_u32(&sm.full[slot]), 0);
      uint8_t* dst = slot_ptr<true>(sm, slot);
      int r0;
      const int outer = kv_at(kt, r0);   // batch mode: the page, r0 within it
      const int key0 = is_v ? r0 : r0 + kHalfKeys * (int)rank;
      const int blk0 = is_v ? 2 * (int)rank : 0;
      if (outer < 0)
        tma_load_4d_pair_warp(dst, map, bar, 0, key0, kvh, blk0);
      else
        tma_load_5d_pair_warp(dst, map, bar, 0, key0, kvh, blk0, outer);
      ++cnt;
      return true;
    };
    auto load_k = [&](int kt) -> bool {
      if (kPair) return load_half(tm_k, false, kt);
      if (kMode == kModeVerify8) return load_raw8(tm_k, kt);
      int r0;
      const int outer = kv_at(kt, r0);
      return load_tile(tm_k, true, kvh, r0, outer, kTileBytes);
    };
    auto load_v = [&](int kt) -> bool {
      if (kPair) return load_half(tm_v, true, kt);
      if (kMode == kModeVerify8) return load_raw8(tm_v, kt);
      int r0;
      const int outer = kv_at(kt, r0);
      return load_tile(tm_v, true, kvh, r0, outer, kTileBytes);
    };
    // Ring order: the item's prepared Q (for the edge warps), then in MMA order K0,
    // (K_j, V_{j-1}) for j >= 1, V_{n-1}; the gate tile (gated passes) just before V_0.
    // A pair's ring holds only the K and V halves (Q and gate tiles go through the staging
    // buffer, loaded by warp 3).
    if (kPair) {
    } else if (is_verify<kMode>()) {
      if (!load_tile(tm_q, false, it.h, it.seq * a.vrows, -1,
                     4u * kVerifyHeadsPerTile * a.vrows * 128u)) return;
    } else {
      if (!load_tile(tm_q, false, it.h, it.row0 + it.mt * kTileM, -1, kTileBytes)) return;
    }
    auto load_gate = [&]() -> bool {
      return kPair || !has_gate<kMode, kW>() ||
             load_tile(tm_g, false, it.h, it.row0 + it.mt * kTileM, -1, kTileBytes, kDim);
    };
    if (!load_k(ck.next(0))) return;
    for (int j = 1; j < it.n; ++j) {
      if (!load_k(ck.next(j))) return;
      if (j == 1 && !load_gate()) return;
      if (!kW && !load_v(cv.next(j - 1))) return;
    }
    if (it.n == 1 && !load_gate()) return;
    if (!kW && !load_v(cv.next(it.n - 1))) return;
  }
}

template <int kMode, bool kW, bool kPair>
__device__ void producer(AttnSmem& sm, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                         const CUtensorMap* tm_v, const CUtensorMap* tm_g, const AttnArgs& a,
                         volatile int* abort) {
  uint32_t cnt = 0;
  producer_loop<kMode, kW, kPair>(sm, tm_q, tm_k, tm_v, tm_g, a, abort, cnt);
  if (*abort) {
    if (kPair && (blockIdx.x & 1) && cnt > 0) {
      // this CTA's K and V halves complete on the peer's barriers, not on its own: give the
      // copies in flight (from memory: microseconds) about a millisecond to land
      const long long t0 = clock64();
      while (clock64() - t0 < (1LL << 21)) {
      }
    }
    // let the loads already issued into the slots land before exit
    constexpr uint32_t kRing = (uint32_t)ring_slots<kPair>();
    const uint32_t first = cnt > kRing ? cnt - kRing : 0;
    for (uint32_t c = first; c < cnt; ++c)
      mbar_wait_quiet(&sm.full[c % kRing], (c / kRing) & 1, 100000000LL);
  }
}

// ------------------------------------------------------------------ warp 3: staging (pairs)
// A pair CTA's staging buffer takes, in turn, each item's prepared Q tile and its gate tile
// (fill 2i and 2i + 1 for the CTA's i-th item), each four 64-dim boxes of 128 rows. The edge
// warps hand a Q fill back only after the previous item's output tile, written into the
// same buffer after they copied Q out, has been read by its tensor stores; so the next item's
// Q is in shared memory long before the current item ends, and its gate tile follows once
// the output is out.
template <int kMode, bool kPair>
__device__ void stage_producer(AttnSmem& sm, const CUtensorMap* tm_q, const CUtensorMap* tm_g,
                               const AttnArgs& a, volatile int* abort) {
  uint8_t* stg = staging_ptr(sm);
  uint32_t f = 0;   // fills issued
  auto load = [&](const CUtensorMap* map, int head, int r0, int x0) -> bool {
    if (f > 0 && !warp_wait(&sm.stg_empty, (f - 1) & 1, abort)) return false;
    mbar_expect_tx_warp(&sm.stg_full, kTileBytes);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      tma_load_3d_warp(stg + c * kChunkBytes, map, &sm.stg_full, x0 + c * 64, head, r0);
    ++f;
    return true;
  };
  ItemWalk<kMode, kPair> walk;
  Item it;
  while (walk.next(a, it)) {
    const int r0 = it.row0 + it.mt * kTileM;
    if (!load(tm_q, it.h, r0, 0)) break;
    if (!load(tm_g, it.h, r0, kDim)) break;
  }
  // on the way out after an abort, the last fill (never waited for by a consumer) lands first
  if (*abort && f > 0) mbar_wait_quiet(&sm.stg_full, (f - 1) & 1, 100000000LL);
}

// ------------------------------------------------------------------ warps 1-2: MMA issuers
// Two issuing warps share the tensor pipe: warp 1 issues every S = Q K^T and warp 2 every
// O += P V, so a tile's P V enters the pipe as soon as its P is written even while the next
// tile's Q K^T is still being issued. Each warp walks the whole tile ring in order, waiting
// for every fill (also those it does not use): a parity wait is only safe when the slot's
// previous fill is known to have landed, and walking in order guarantees it. A slot is
// refilled only when every walker has passed it (each arrives on the slot's empty barrier
// once it has seen the fill) and its consumer has released it (tcgen05.commit for K and V,
// the edge warps for Q), so no walker can miss a fill. A warp's commits track only its own
// MMAs (a commit covers the MMAs its thread issued).
// Ring order per item: Q, K0, then K_j, V_{j-1} for j >= 1, then V_{n-1}, with the gate
// tile of the gated passes right before V_0 (Q and K only in the weights pass).
// With e4m3 caches a fill is ready once the edge warps have widened it (K, V) or seen it (Q).
template <int kMode, bool kPair = false>
struct RingWalk {
  uint32_t cnt = 0;
  // wait for the next fill in ring order (its slot in `slot`) and count this warp as past it
  __device__ __forceinline__ bool next(AttnSmem& sm, volatile int* abort, uint32_t& slot) {
    constexpr uint32_t kRing = (uint32_t)ring_slots<kPair>();
    slot = cnt % kRing;
    const bool ok = kMode == kModeVerify8
                        ? __all_sync(0xffffffffu, mbar_wait<true>(&sm.conv[slot], (cnt / kRing) & 1, abort))
                        : warp_wait(&sm.full[slot], (cnt / kRing) & 1, abort);
    ++cnt;
    if (ok && (threadIdx.x & 31) == 0) mbar_arrive(&sm.empty[slot]);
    return ok;
  }
};

// descriptors advance by constants (addresses in 16-byte units in the low field): K by
// 32 bytes per k-step inside a 64-dim block and 16 KiB per block; P by 32 bytes per k-step
// inside a 64-key block and 16 KiB per block; V by 2 KiB per k-step; a slot is 64 KiB.
template <int kMode, bool kW, bool kPair>
__device__ void qk_loop(AttnSmem& sm, const AttnArgs& a, uint32_t tmem, volatile int* abort) {
  // a pair: M = 256 (both CTAs' rows), each CTA holding 64 of the tile's keys, so a 64-dim
  // block of this CTA's K is 8 KiB
  constexpr uint32_t kIdQK = idesc_bf16(kPair ? 256 : 128, kTileN, false, false);
  constexpr uint32_t kKBlock = kPair ? kChunkBytes / 2 : kChunkBytes;
  constexpr uint32_t kSlotBytes = kPair ? kHalfTileBytes : kTileBytes;
  const uint64_t k_desc0 = sdesc_sw128(smem_u32(sm.tile[0]), 16, 1024);
  const uint64_t qhi_desc0 = sdesc_sw128(smem_u32(sm.qhi[0]), 16, 1024);
  RingWalk<kMode, kPair> ring;
  uint32_t g = 0;         // global key-tile counter: S phases
  uint32_t it_done = 0;
  uint32_t slot;
  ItemWalk<kMode, kPair> walk;
  Item it;
  // V_idx, preceded by the gate tile when idx is 0 (not in a pair's ring)
  auto walk_v = [&](int idx) -> bool {
    if (!kPair && has_gate<kMode, kW>() && idx == 0 && !ring.next(sm, abort, slot)) return false;
    return ring.next(sm, abort, slot);
  };
  while (walk.next(a, it)) {
    if (!kPair && !ring.next(sm, abort, slot)) return;  // the item's Q tile (edge warps)
    if (!warp_wait<kPair>(&sm.q_full, it_done & 1, abort)) return;
    for (int j = 0; j < it.n; ++j, ++g) {
      if (!kW && j >= 2 && !walk_v(j - 2)) return;      // V_{j-2}
      if (!ring.next(sm, abort, slot)) return;          // K_j
      // S is free once the softmax warps have copied the previous tile's S out
      if (g > 0 && !warp_wait<kPair>(&sm.s_free, (g - 1) & 1, abort)) return;
      tc_fence_after();
      const uint64_t kd0 = k_desc0 + (uint64_t)(slot * (kSlotBytes >> 4));
      // dims 0..127 with Q from tensor memory, dims 128..255 with Q from shared memory
#pragma unroll
      for (int kk = 0; kk < kDim / 32; ++kk) {
        const uint64_t bd = kd0 + (uint64_t)((kk >> 2) * (kKBlock >> 4) + (kk & 3) * 2);
        mma_ts<kPair>(tmem + kTmemS, tmem + kTmemQ + kk * 8, bd, kIdQK, kk > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int kk = kDim / 32; kk < kDim / 16; ++kk) {
        const uint32_t blk = (kk >> 2) - 2;
        const uint64_t bd = kd0 + (uint64_t)((kk >> 2) * (kKBlock >> 4) + (kk & 3) * 2);
        const uint64_t ad = qhi_desc0 + (uint64_t)(blk * (kChunkBytes >> 4) + (kk & 3) * 2);
        mma_ss<kPair>(tmem + kTmemS, ad, bd, kIdQK, 1u);
      }
      mma_commit<kPair>(&sm.empty[slot]);
      mma_commit<kPair>(&sm.s_full);
      if (j == it.n - 1) mma_commit<kPair>(&sm.q_empty);
    }
    if (!kW) {
      if (it.n >= 2 && !walk_v(it.n - 2)) return;       // V_{n-2}
      if (!walk_v(it.n - 1)) return;                    // V_{n-1}
    }
    ++it_done;
  }
}

// A pair's V half is its two 64-dim blocks of 128 keys (N = 256 over the pair), at the same
// block stride as a whole tile's.
template <int kMode, bool kPair>
__device__ void pv_loop(AttnSmem& sm, const AttnArgs& a, uint32_t tmem, volatile int* abort) {
  constexpr uint32_t kIdPV = idesc_bf16(kPair ? 256 : 128, kDim, false, true);
  constexpr uint32_t kSlotBytes = kPair ? kHalfTileBytes : kTileBytes;
  const uint64_t v_desc0 = sdesc_sw128(smem_u32(sm.tile[0]), kChunkBytes, 1024);
  RingWalk<kMode, kPair> ring;
  uint32_t g = 0;         // global key-tile counter: P and P V phases
  uint32_t it_done = 0;
  uint32_t slot;
  ItemWalk<kMode, kPair> walk;
  Item it;
  while (walk.next(a, it)) {
    if (!kPair && !ring.next(sm, abort, slot)) return;  // Q
    if (!ring.next(sm, abort, slot)) return;            // K0
    for (int j = 0; j < it.n; ++j, ++g) {
      if (j + 1 < it.n && !ring.next(sm, abort, slot)) return;   // K_{j+1}
      if (!kPair && has_gate<kMode, false>() && j == 0 && !ring.next(sm, abort, slot)) return;   // gate
      if (!ring.next(sm, abort, slot)) return;                   // V_j
      if (j == 0 && it_done > 0 && !warp_wait<kPair>(&sm.o_free, (it_done - 1) & 1, abort)) return;
      const uint64_t bd0 = v_desc0 + (uint64_t)(slot * (kSlotBytes >> 4));
      // The two 64-key halves of P go separately: each softmax warpgroup writes its half
      // of the next tile as soon as this tile's P V has read that half.
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        if (!warp_wait<kPair>(&sm.p_full[hb], g & 1, abort)) return;
        tc_fence_after();
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = 4 * hb + k4;
          mma_ts<kPair>(tmem + kTmemO, tmem + kTmemP + hb * (kHalfKeys / 2) + k4 * 8,
                        bd0 + (uint64_t)(kk * (2048 >> 4)), kIdPV,
                        (j > 0 || kk > 0) ? 1u : 0u);
        }
        // p_empty[1] also tells the softmax that O holds every P V so far
        mma_commit<kPair>(&sm.p_empty[hb]);
      }
      mma_commit<kPair>(&sm.empty[slot]);
    }
    mma_commit<kPair>(&sm.o_done);
    ++it_done;
  }
}

// Issue every MMA, then wait (bounded) until all of them completed, so that tensor
// memory is never released under an MMA in flight.
template <int kMode, bool kW, bool kPair>
__device__ void mma_issuer(AttnSmem& sm, const AttnArgs& a, uint32_t tmem, volatile int* abort,
                           bool pv_warp) {
  uint64_t* drain = pv_warp ? &sm.drain_pv : &sm.drain;
  if (pv_warp) {
    if (kW) return;   // the weights pass has no P V
    pv_loop<kMode, kPair>(sm, a, tmem, abort);
  } else {
    qk_loop<kMode, kW, kPair>(sm, a, tmem, abort);
  }
  if (kPair) umma_commit_pair_local_warp(drain);
  else umma_commit_warp(drain);
  mbar_wait_quiet(drain, 0, 100000000LL);
}

// ------------------------------------------------------------------ shared helpers
__device__ __forceinline__ float lo_f(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hi_f(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return (uint32_t)bf16_bits(a) | ((uint32_t)bf16_bits(b) << 16);
}

// Visibility of the 32 keys kt*128 + 32*ch .. +31 for one row: bit k <-> key +k. `limit`
// is the row's last visible key (causal and verify modes).
template <int kMode>
__device__ __forceinline__ uint32_t chunk_visibility(const AttnArgs& a, int row, int limit, int kt,
                                                     int ch, bool valid) {
  if (!valid) return 0u;
  const int first = kt * kTileN + ch * 32;
  int n = (kMode == kModeBidir) ? (a.T - first) : (limit - first + 1);
  n = max(0, min(32, n));
  return n >= 32 ? 0xFFFFFFFFu : ((1u << n) - 1u);
}

// Stored mask: this row's visibility words of one 64-key half of tile kt (keys 32 apart,
// in the prepass's bit order). Rows past the end of the call lie inside the prepass's
// padded row tile, whose words are zero.
__device__ __forceinline__ uint2 mask_words_half(const AttnArgs& a, int row, int kt, int hf) {
  return __ldg(reinterpret_cast<const uint2*>(a.mask_bits + (size_t)row * a.mask_words +
                                              kt * (kTileN / 32) + 2 * hf));
}

// The bf16 score pairs sb[0..31] of a 64-key half with every hidden key set to -inf, from
// the half's two visibility words. For s = 0..7, word << s holds keys 4s .. 4s+3 in the top
// bits of its bytes (the prepass's bit order), and a byte permute that replicates those
// bits gives each pair's keep mask (0xFFFF per visible key); one three-input logic op then
// keeps the score or puts -inf (0xFF80) in its place.
__device__ __forceinline__ void apply_mask_half(uint32_t (&sb)[kHalfKeys], uint2 vis) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t word = c ? vis.y : vis.x;
#pragma unroll
    for (int s4 = 0; s4 < 8; ++s4) {
      const uint32_t w = word << s4;
      const uint32_t k0 = prmt_b32(w, 0u, 0x9988u);   // keys 4s, 4s+1
      const uint32_t k1 = prmt_b32(w, 0u, 0xBBAAu);   // keys 4s+2, 4s+3
      uint32_t& p0 = sb[16 * c + 2 * s4];
      uint32_t& p1 = sb[16 * c + 2 * s4 + 1];
      p0 = (p0 & k0) | (0xFF80FF80u & ~k0);
      p1 = (p1 & k1) | (0xFF80FF80u & ~k1);
    }
  }
}

// Every key of tile kt visible to every row of row tile mt (no per-key selects needed).
// (Verify: every key visible to every row of the item; the padding lanes past 6 vrows see
// zero queries and are never written out.)
template <int kMode>
__device__ __forceinline__ bool tile_full(const AttnArgs& a, const Item& it, int kt) {
  if (kMode == kModeMask) return false;
  if (is_verify<kMode>()) return (kt + 1) * kTileN - 1 <= a.seq_len[it.seq];
  if ((it.mt + 1) * kTileM > it.rows || (kt + 1) * kTileN > it.T) return false;
  if (is_causal<kMode>()) return (kt + 1) * kTileN - 1 <= it.qb + it.mt * kTileM;
  return true;
}

// ------------------------------------------------------------------ warps 4-11: softmax
// Weights pass: bf16(bf16(2^(t - M)) / l) for the 64 keys of one half tile (bf16 score pairs
// in sb[0 .. 31], hidden ones -inf), with the main pass's final M and l, written to
// weights[h][row][key0 ..].
__device__ __forceinline__ void weights_half(const AttnArgs& a, const uint32_t (&sb)[kHalfKeys],
                                             int h, int row, int key0, int M, float l_final) {
  const float mf = (float)M;
  uint16_t* wrow = a.weights + ((size_t)h * a.rows + row) * (size_t)a.T + (size_t)key0;
  const int ncol = min(kHalfKeys, a.T - key0);
  const bool vec = (ncol == kHalfKeys) && ((a.T & 7) == 0);
#pragma unroll
  for (int ch = 0; ch < kHalfKeys / 32; ++ch) {
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

// Softmax of one 64-key half (hf) of every S tile, one query row per thread.
template <int kMode, bool kW, bool kPair>
__device__ void softmax_worker(AttnSmem& sm, const AttnArgs& a, uint32_t tmem, int hf,
                               volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t s_taddr = tmem + kTmemS + lane_off + kHalfKeys * hf;
  uint32_t g = 0, it_done = 0;
  ItemWalk<kMode, kPair> walk;
  Item it;
  while (walk.next(a, it)) {
    const int row = it.mt * kTileM + r;   // the row within its sequence
    const bool valid = is_verify<kMode>() ? r < kVerifyHeadsPerTile * a.vrows : row < it.rows;
    const int limit = is_verify<kMode>() ? a.seq_len[it.seq] + r / kVerifyHeadsPerTile
                                           : it.qb + row;
    const int h = it.h;
    int M = 0;
    bool hasM = false;
    float l = 0.f;        // this half's sum of the rounded weights
    float l_final = 0.f;  // weights pass: the main pass's l (relative to its final M)
    if (kW && valid) {
      M = (int)a.row_stats[((size_t)h * a.rows + row) * 2];
      l_final = a.row_stats[((size_t)h * a.rows + row) * 2 + 1];
      hasM = l_final > 0.f;
    }
    TileCursor<kMode> cursor(it);
    // stored mask: the next tile's visibility words are loaded a tile ahead, so their
    // latency hides behind this tile's work
    int kt_next = cursor.next(0);
    uint2 vis_next = make_uint2(0u, 0u);
    if (kMode == kModeMask) vis_next = mask_words_half(a, it.mt * kTileM + r, kt_next, hf);
    for (int j = 0; j < it.n; ++j, ++g) {
      const int kt = kt_next;
      const uint2 vis = vis_next;
      if (j + 1 < it.n) {
        kt_next = cursor.next(j + 1);
        if (kMode == kModeMask) vis_next = mask_words_half(a, it.mt * kTileM + r, kt_next, hf);
      }
      if (!warp_wait(&sm.s_full, g & 1, abort)) return;
      tc_fence_after();
      // this half's 64 S columns -> registers, packed in place as bf16 pairs (the score's
      // own rounding); then the columns are released
      uint32_t sb[kHalfKeys];
      tmem_ld32(s_taddr + 0, *reinterpret_cast<uint32_t(*)[32]>(sb));
      tmem_ld32(s_taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(sb + 32));
      tmem_wait_ld(sb);
      tc_fence_before();
      arrive_for_mma<kPair>(&sm.s_free);   // the next S = Q K^T may overwrite S once both halves are out
      if (kMode == kModeMask) {
#pragma unroll
        for (int k = 0; k < kHalfKeys / 2; ++k)
          sb[k] = pack_bf16x2(__uint_as_float(sb[2 * k]), __uint_as_float(sb[2 * k + 1]));
        if (!__all_sync(0xffffffffu, (vis.x & vis.y) == 0xFFFFFFFFu)) apply_mask_half(sb, vis);
      } else if (tile_full<kMode>(a, it, kt)) {
#pragma unroll
        for (int k = 0; k < kHalfKeys / 2; ++k)
          sb[k] = pack_bf16x2(__uint_as_float(sb[2 * k]), __uint_as_float(sb[2 * k + 1]));
      } else {
#pragma unroll
        for (int ch = 0; ch < kHalfKeys / 32; ++ch) {
          const uint32_t vis = chunk_visibility<kMode>(a, row, limit, kt, 2 * hf + ch, valid);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            // hidden keys read as -inf: weight exactly 0, never the maximum
            const int e = ch * 32 + 2 * k;
            const float s0 = ((vis >> (2 * k)) & 1u) ? __uint_as_float(sb[e]) : -INFINITY;
            const float s1 = ((vis >> (2 * k + 1)) & 1u) ? __uint_as_float(sb[e + 1]) : -INFINITY;
            sb[ch * 16 + k] = pack_bf16x2(s0, s1);   // writes an index already read
          }
        }
      }

      if (kW) {
        if (valid && hasM) weights_half(a, sb, h, row, kt * kTileN + kHalfKeys * hf, M, l_final);
        continue;
      }
      // this half's maximum of the bf16 scores, exchanged with the other half's: both halves
      // then take the same decisions on M
      uint32_t m0 = sb[0], m1 = sb[1], m2 = sb[2], m3 = sb[3];
#pragma unroll
      for (int k = 4; k < kHalfKeys / 2; k += 4) {
        m0 = max_bf16x2(m0, sb[k]);
        m1 = max_bf16x2(m1, sb[k + 1]);
        m2 = max_bf16x2(m2, sb[k + 2]);
        m3 = max_bf16x2(m3, sb[k + 3]);
      }
      const uint32_t mm = max_bf16x2(max_bf16x2(m0, m1), max_bf16x2(m2, m3));
      const uint32_t mine = max_bf16x2(mm, mm >> 16) & 0xFFFFu;   // low half: max of both
      sm.mx[g & 1][hf][r] = (uint16_t)mine;
      mbar_arrive(&sm.mx_bar);
      if (!warp_wait(&sm.mx_bar, g & 1, abort)) return;
      const uint32_t other = sm.mx[g & 1][hf ^ 1][r];
      const float mx = fmaxf(__uint_as_float(mine << 16), __uint_as_float(other << 16));
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
        // O must hold every earlier P.V before it is scaled (the PV of global tile g-1, whose
        // completion p_empty[1] marks; the P buffer wait below then passes at once). Each
        // half scales its own 128 of O's 256 columns.
        if (!warp_wait(&sm.p_empty[1], (g - 1) & 1, abort)) return;
        tc_fence_after();
        const float f = rescale ? exp2f((float)(M - newM)) : 1.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < kDim / 2; c0 += 32) {
          const uint32_t ta = tmem + kTmemO + lane_off + (kDim / 2) * hf + c0;
          uint32_t o[32];
          tmem_ld32(ta, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
          tmem_st32(ta, o);
        }
        tmem_wait_st();
        l *= f;
      }
      M = newM;
      const float mf = hasM ? (float)M : 0.f;
      // P = bf16(2^(t - M)), t = bf16(s) * log2(e) / 16, computed in place over the scores
      // (l sums the rounded P), then stored into this half's 64-key block of shared memory
      // once the previous P.V has read it: the exponentials do not wait for the tensor cores
      float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
      for (int k = 0; k < kHalfKeys / 2; ++k) {
        const uint32_t w = sb[k];
        const float t0 = fmaf(lo_f(w), kLog2eOver16, -mf);
        const float t1 = fmaf(hi_f(w), kLog2eOver16, -mf);
        sb[k] = pack_bf16x2(ex2_approx(t0), ex2_approx(t1));
        if (k & 1) add_bf16x2(l2, l3, sb[k]);
        else add_bf16x2(l0, l1, sb[k]);
      }
      l += (l0 + l2) + (l1 + l3);
      // this half's P (word k: keys 2k, 2k+1) into its 32 columns of tensor memory once the
      // previous P V has read them
      if (g > 0 && !warp_wait(&sm.p_empty[hf], (g - 1) & 1, abort)) return;
      tc_fence_after();
      tmem_st32(tmem + kTmemP + lane_off + (kHalfKeys / 2) * hf,
                *reinterpret_cast<uint32_t(*)[32]>(sb));
      tmem_wait_st();
      tc_fence_before();
      arrive_for_mma<kPair>(&sm.p_full[hf]);
    }
    if (!kW) {
      // hand this half's l (and M) of the item to the edge warps
      if (it_done > 0 && !warp_wait(&sm.st_empty, (it_done - 1) & 1, abort)) return;
      sm.stat_l[hf][r] = l;
      if (hf == 0) sm.stat_m[r] = hasM ? (float)M : 0.f;
      mbar_arrive(&sm.st_full);
    }
    ++it_done;
  }
}

// ------------------------------------------------------------------ warps 12-15: edge
// The item's prepared Q tile (a ring slot: four 128-row x 64-dim blocks, 128-byte
// swizzled): dims 0..127 into this thread's TMEM lane at Q (row r, dims 2c and 2c+1 in
// column c), dims 128..255 as they are into the item's Q blocks in shared memory (the same
// swizzled layout, read by the tensor cores). Every lane of the warp runs it
// (warp-collective stores). Lanes with `have` false (verify padding) store zeros.
template <bool kPair>
__device__ __forceinline__ void q_copy(const uint8_t* tile, int r, bool have, uint32_t q_taddr,
                                       uint8_t (&qhi)[2][kChunkBytes]) {
#pragma unroll
  for (int grp = 0; grp < 4; ++grp) {
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const uint8_t* base = tile + grp * kChunkBytes;
      const uint32_t o0 = sw128_offset((uint32_t)r, (uint32_t)j);
      const uint32_t o1 = sw128_offset((uint32_t)r, (uint32_t)j + 1);
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
      if (have) {
        v0 = *reinterpret_cast<const uint4*>(base + o0);
        v1 = *reinterpret_cast<const uint4*>(base + o1);
      }
      if (grp < 2) {
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        tmem_st8(q_taddr + 32 * grp + 4 * j, w);
      } else {
        *reinterpret_cast<uint4*>(qhi[grp - 2] + o0) = v0;
        *reinterpret_cast<uint4*>(qhi[grp - 2] + o1) = v1;
      }
    }
  }
  tmem_wait_st();
  // the tensor cores read the shared-memory half (a pair's: MMAs the peer CTA issues)
  if (kPair) fence_async_smem_cluster();
  else fence_async_smem();
}

// bf16(sigmoid(g)) for every bf16 g (index: g's bits), exact from the double definition;
// filled once per device from the host. Every gate of the epilogue and of the verify
// combine is looked up here: the answer is the definition itself, and a lookup costs the
// edge warps far less than computing it (exponential and reciprocal on the special-function
// unit the softmax needs) while the item's tiles run.
__device__ uint16_t g_sigmoid_bf16[1 << 16];

__device__ __forceinline__ uint32_t sigmoid_pair(uint32_t g) {
  return (uint32_t)g_sigmoid_bf16[g & 0xFFFFu] | ((uint32_t)g_sigmoid_bf16[g >> 16] << 16);
}

// This thread's 256 gates (row r of the item's gate tile in a ring slot: four 128-row x
// 64-value blocks, 128-byte swizzled) into registers, word c holding dims 2c and 2c+1.
// Rows past the end read as zeros; their outputs are never stored.
__device__ __forceinline__ void gate_from_tile(const uint8_t* tile, int r, uint4 (&sg)[kDim / 8]) {
#pragma unroll
  for (int grp = 0; grp < 4; ++grp) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      sg[grp * 8 + j] = *reinterpret_cast<const uint4*>(tile + grp * kChunkBytes +
                                                        sw128_offset((uint32_t)r, (uint32_t)j));
  }
}

// bf16(sigmoid(g)) of the 256 gates in sg, in place, from the table. The table (128 KB) does
// not fit in the L1 left beside the shared memory, so each lookup is an L2 read: the gates
// go 32 at a time (64 independent lookups in flight), through a register queue that moves on
// by 4 entries per round. The loop body stays short: this code shares the instruction cache
// with the softmax loop on the same SM sub-partition.
__device__ void gate_sigmoid(uint4 (&sg)[kDim / 8]) {
  constexpr int kPer = 4;   // queue entries (8 gates each) per round
#pragma unroll 1
  for (int round = 0; round < kDim / 8 / kPer; ++round) {
    uint4 o[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const uint4 g = sg[i];
      o[i] = make_uint4(sigmoid_pair(g.x), sigmoid_pair(g.y), sigmoid_pair(g.z), sigmoid_pair(g.w));
    }
#pragma unroll
    for (int i = 0; i < kDim / 8 - kPer; ++i) sg[i] = sg[i + kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) sg[kDim / 8 - kPer + i] = o[i];
  }
}

// Outputs of a work item none of whose key tiles is visible (mask mode): every row is
// hidden, its output row and statistics are zero.
__device__ void write_hidden_rows(const AttnArgs& a, const Item& it, int r, bool weights_pass) {
  const int row = it.mt * kTileM + r;
  if (row >= a.rows || weights_pass) return;
  uint4* o = reinterpret_cast<uint4*>(a.out + (size_t)row * kOutRow + it.h * kDim);
  for (int i = 0; i < 32; ++i) o[i] = make_uint4(0, 0, 0, 0);
  if (a.row_stats) {
    a.row_stats[((size_t)it.h * a.rows + row) * 2] = 0.f;
    a.row_stats[((size_t)it.h * a.rows + row) * 2 + 1] = 0.f;
  }
  if (a.hidden_rows && it.h == a.head0) atomicAdd(a.hidden_rows, 1);
}

// Gated epilogue of one finished item: out = bf16(bf16(O / l) * s) with s = bf16(sigmoid(
// gate)) already in registers. All of O is read first (64 columns at a time, each gated pair
// of bf16 kept in a register: 128 words for the row, the gate registers freed as they are
// used) and released at once, so the next item's first P V waits only for the reads; the
// row's 512 bytes of stores follow while the next item runs.
// A pair CTA writes its output tile into the staging buffer instead (row r of each 64-dim
// block, in the 128-byte-swizzled layout of the output map's boxes) and one thread stores it
// with four tensor stores: whole 128-byte lines, where each thread's own row stores (32 rows
// 12 KiB apart per warp instruction) hold up the tensor cores' shared-memory reads for their
// whole duration.
template <int kMode, bool kPair>
__device__ bool epilogue(AttnSmem& sm, const AttnArgs& a, const CUtensorMap* tm_o, const Item& it,
                         uint32_t tmem, uint32_t lane_off, int r, uint32_t it_done,
                         uint4 (&sg)[kDim / 8], volatile int* abort) {
  const int row = it.mt * kTileM + r;   // the row within its sequence
  const bool valid = row < it.rows;
  const int h = it.h;
  if (!warp_wait(&sm.st_full, it_done & 1, abort)) return false;
  const float l = sm.stat_l[0][r] + sm.stat_l[1][r];
  const float M = sm.stat_m[r];
  if (!warp_wait(&sm.o_done, it_done & 1, abort)) return false;
  tc_fence_after();
  const float inv = l > 0.f ? 1.0f / l : 0.f;
  uint32_t res[kDim / 2];   // word j: the gated outputs of columns 2j, 2j+1
  // 64 columns per round: two 32-column loads in flight, one wait
#pragma unroll
  for (int c64 = 0; c64 < kDim / 64; ++c64) {
    uint32_t o[64];
    tmem_ld32(tmem + kTmemO + lane_off + 64 * c64, *reinterpret_cast<uint32_t(*)[32]>(o));
    tmem_ld32(tmem + kTmemO + lane_off + 64 * c64 + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
    tmem_wait_ld(o);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 g4 = sg[8 * c64 + i];   // the sigmoids of columns 64 c64 + 8 i .. + 7
      const uint32_t sw[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t ob = pack_bf16x2(__uint_as_float(o[8 * i + 2 * k]) * inv,
                                        __uint_as_float(o[8 * i + 2 * k + 1]) * inv);
        res[32 * c64 + 4 * i + k] = mul_bf16x2(ob, sw[k]);   // bf16(o * s), both bf16
      }
    }
  }
  tc_fence_before();
  arrive_for_mma<kPair>(&sm.o_free);
  mbar_arrive(&sm.st_empty);
  // batch mode: a tile that ends inside its sequence leaves by the rows' own stores (the
  // box's remaining rows belong to the next sequence)
  const bool tma_out = kMode != kModeBatch || (it.mt + 1) * kTileM <= it.rows;
  if (kPair && !tma_out) {
    mbar_arrive(&sm.o_st);   // every row has read the staged Q: the buffer may refill
    if (threadIdx.x == kEdgeThread0) {
      if (!mbar_wait(&sm.o_st, it_done & 1, abort)) return false;
      mbar_arrive(&sm.stg_empty);
    }
  } else if (kPair) {
    uint8_t* stg = staging_ptr(sm);
#pragma unroll
    for (int c64 = 0; c64 < kDim / 64; ++c64)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(stg + c64 * kChunkBytes + sw128_offset((uint32_t)r, (uint32_t)j)) =
            make_uint4(res[32 * c64 + 4 * j], res[32 * c64 + 4 * j + 1], res[32 * c64 + 4 * j + 2],
                       res[32 * c64 + 4 * j + 3]);
    fence_async_smem();   // the tensor stores read what the threads wrote
    mbar_arrive(&sm.o_st);
    if (threadIdx.x == kEdgeThread0) {
      if (!mbar_wait(&sm.o_st, it_done & 1, abort)) return false;
      // rows past the call's end lie outside the map and are not written
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tma_store_3d(tm_o, stg + c * kChunkBytes, c * 64, h, it.row0 + it.mt * kTileM);
      bulk_commit_group();
      bulk_wait_group_read0();
      mbar_arrive(&sm.stg_empty);   // the buffer may take the next gate tile
    }
  }
  if (!valid) return true;
  uint4* op = reinterpret_cast<uint4*>(a.out + (size_t)(it.row0 + row) * kOutRow + h * kDim);
  if (kPair && tma_out) {
  } else if ((reinterpret_cast<uintptr_t>(a.out) & 31u) == 0) {   // rows are 12 KiB apart
#pragma unroll
    for (int q = 0; q < kDim / 16; ++q) {
      const uint32_t w[8] = {res[8 * q], res[8 * q + 1], res[8 * q + 2], res[8 * q + 3],
                             res[8 * q + 4], res[8 * q + 5], res[8 * q + 6], res[8 * q + 7]};
      st_global_v8(op + 2 * q, w);
    }
  } else {
#pragma unroll
    for (int q = 0; q < kDim / 8; ++q)
      op[q] = make_uint4(res[4 * q], res[4 * q + 1], res[4 * q + 2], res[4 * q + 3]);
  }
  if (a.row_stats) {
    a.row_stats[((size_t)h * a.rows + row) * 2] = M;
    a.row_stats[((size_t)h * a.rows + row) * 2 + 1] = l;
  }
  if (a.hidden_rows && h == a.head0 && l == 0.f) atomicAdd(a.hidden_rows, 1);
  return true;
}

// Verify epilogue of one item: the unnormalised O (fp32, relative to 2^M) and M, l of each
// lane's packed row, for the combine kernel; O is released after the copy.
__device__ bool epilogue_partial(AttnSmem& sm, const AttnArgs& a, const Item& it, uint32_t tmem,
                                 uint32_t lane_off, int r, uint32_t it_done, volatile int* abort) {
  const bool valid = r < kVerifyHeadsPerTile * a.vrows;
  if (!warp_wait(&sm.st_full, it_done & 1, abort)) return false;
  const float l = sm.stat_l[0][r] + sm.stat_l[1][r];
  const float M = sm.stat_m[r];
  if (!warp_wait(&sm.o_done, it_done & 1, abort)) return false;
  tc_fence_after();
  const int chunk = it.kt0 / a.chunk_tiles;
  const size_t slot = (((size_t)it.seq * kKvHeads + it.h / kGroup) * 2 + it.half) * a.n_chunks + chunk;
  const size_t prow = slot * kVerifyLanes + (valid ? r : 0);
  float4* op = reinterpret_cast<float4*>(a.part_o + prow * kDim);
#pragma unroll 1
  for (int c = 0; c < kDim / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(tmem + kTmemO + lane_off + c * 32, o);
    tmem_wait_ld(o);
    if (valid) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        op[8 * c + q] = make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                    __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
    }
  }
  tc_fence_before();
  mbar_arrive(&sm.o_free);
  mbar_arrive(&sm.st_empty);
  if (valid) reinterpret_cast<float2*>(a.part_ml)[prow] = make_float2(M, l);
  return true;
}

// e4m3 caches: this CTA's 64 keys of the fill's tile (their codes in eight pieces, each in
// the rows of the edge warp that widens it) become rows 64 rank .. 64 rank + 63 of the bf16
// tile the tensor cores read, bf16(fp32(code * scale)) per element, in this CTA's slot; the
// copy engine then copies them into the same rows of the peer's slot (the peer supplies the
// other 64). Edge warp w widens rows 16w .. 16w+15 of the half, lane l the 16 codes of column
// l % 16 in rows l / 16 + 2k. Each thread reads its codes (its rows' scales loaded during the
// previous fill); once the warp has read (its rows overwrite its own codes, and nothing else
// does) it writes its rows and arrives on this CTA's conv barrier of the slot, which also
// waits for the 32 KiB the peer copies in. Lane 0 of each warp then waits until the peer's
// slot is free for this fill (its producer's signal, normally long given) and copies the
// warp's 16 rows of each 64-dim block (2 KiB, rows contiguous) to the peer. The MMA warps of
// each CTA wait on their conv barrier. The long-prompt page's F8 rows are staged this way:
// loaded a step ahead, widened in the slot.
constexpr uint32_t kPeerCopyBytes = kRawKeys * 128 * 4;   // the peer's 64 rows of 4 blocks
constexpr int kWideRows = 8;   // rows each edge thread widens per fill
// The scales of an edge thread's rows of key tile kt (this CTA's half), for the fill after the
// current one: loaded while the current fill is widened.
__device__ __forceinline__ void load_row_scales(const AttnArgs& a, const float* scale, int seq,
                                                int kvh, int kt, int t, float (&scv)[kWideRows]) {
  const uint32_t rank = blockIdx.x & 1;
  const int rbase = 16 * (t >> 5) + ((t & 31) >> 4);
  const float* srow = scale + (size_t)seq * a.cache_cap * kKvHeads + kvh;
#pragma unroll
  for (int k = 0; k < kWideRows; ++k) {
    const int key = kt * kTileN + kRawKeys * (int)rank + rbase + 2 * k;
    scv[k] = key < a.cache_cap ? __ldg(srow + (size_t)key * kKvHeads) : 0.f;
  }
}
__device__ bool widen_e4m3(AttnSmem& sm, uint32_t pos, const float (&scv)[kWideRows], int t,
                           volatile int* abort) {
  const uint32_t slot = pos % kSlots;
  const uint32_t rank = blockIdx.x & 1, peer = rank ^ 1u;
  const int w = t >> 5, l = t & 31;
  const int c = l & 15;
  const int rbase = 16 * w + (l >> 4);   // this thread's rows: rbase + 2k of the half
  constexpr int kRows = kWideRows;
  if (!warp_wait(&sm.full[slot], (pos / kSlots) & 1, abort)) return false;
  uint4 v[kRows];
#pragma unroll
  for (int k = 0; k < kRows; ++k) {
    const int kk = (l >> 4) + 2 * k;   // the warp's key 0 .. 15: piece kk / 8, row kk % 8
    v[k] = *reinterpret_cast<const uint4*>(sm.tile[slot] + raw_piece_offset(w, kk >> 3, rank) +
                                           (kk & 7) * kDim + c * 16);
  }
  __syncwarp();   // the warp's codes are read before its rows overwrite them
  uint8_t* blk = sm.tile[slot] + (c >> 2) * kChunkBytes;
  const uint32_t j0 = (uint32_t)(c & 3) * 2;
#pragma unroll
  for (int k = 0; k < kRows; ++k) {
    const uint32_t row = (uint32_t)(kRawKeys * rank + rbase + 2 * k);
    const uint32_t wi[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
    uint32_t wd[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // codes of dims 4q .. 4q+3 of this chunk, lowest byte first; fp32(code * scale)
      const float2 lo = e4m3x2_to_float2(wi[q]);
      const float2 hi = e4m3x2_to_float2(wi[q] >> 16);
      wd[2 * q] = pack_bf16x2(lo.x * scv[k], lo.y * scv[k]);
      wd[2 * q + 1] = pack_bf16x2(hi.x * scv[k], hi.y * scv[k]);
    }
    *reinterpret_cast<uint4*>(blk + sw128_offset(row, j0)) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    *reinterpret_cast<uint4*>(blk + sw128_offset(row, j0 + 1)) = make_uint4(wd[4], wd[5], wd[6], wd[7]);
  }
  fence_async_smem();   // this CTA's tensor cores and copy engine read what the threads wrote
  if (t == 0) mbar_arrive_expect_tx(&sm.conv[slot], kPeerCopyBytes);   // the peer's rows
  else mbar_arrive(&sm.conv[slot]);
  __syncwarp();
  if (!__all_sync(0xffffffffu, mbar_wait<true>(&sm.peer_free[slot], (pos / kSlots) & 1, abort)))
    return false;
  if (l == 0) {
    const uint32_t bar_peer = mapa_shared(smem_u32(&sm.conv[slot]), peer);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint8_t* src = sm.tile[slot] + b * kChunkBytes + (kRawKeys * rank + 16 * w) * 128;
      bulk_copy_to_peer(mapa_shared(smem_u32(src), peer), src, 16 * 128, bar_peer);
    }
  }
  return true;
}

template <int kMode, bool kW, bool kPair>
__device__ void edge_worker(AttnSmem& sm, const AttnArgs& a, const CUtensorMap* tm_o, uint32_t tmem,
                            volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t q_taddr = tmem + kTmemQ + lane_off;
  int round = 0;
  // the CTA's next item with key tiles; items without any are answered on the way
  auto next_item = [&](Item& out) -> bool {
    for (;; ++round) {
      const int idx = walk_index<kMode, kPair>(round);
      if (idx >= a.n_items) return false;
      out = make_item<kMode, kPair>(a, idx);
      if (out.n > 0) {
        ++round;
        return true;
      }
      if (!is_verify<kMode>()) write_hidden_rows(a, out, r, kW);
    }
  };
  // Ring position of each item's Q tile: the producer loads Q, then the item's K and V tiles.
  // The slot is handed back once all 128 edge threads have read it (bounded waits only).
  // q_empty(i) comes first: it means the tensor cores have used item i's last K tile, the
  // slot's previous fill, so the slot's full barrier is at most one phase behind the
  // awaited one (a parity wait cannot tell a phase from the one two before it).
  uint32_t q_pos = 0, q_takes = 0;
  uint32_t stg_f = 0;   // pairs: staging fills taken (the CTA's item i: Q 2i, gate tile 2i + 1)
  // A pair's Q comes from the staging buffer, which the item's output tile takes next (it
  // is handed back after the output's tensor stores); only the first item's Q, which no
  // output follows, is handed back at once.
  auto take_q_pair = [&](bool wait_empty, uint32_t it_done) -> bool {
    if (wait_empty && !warp_wait(&sm.q_empty, it_done & 1, abort)) return false;
    if (!warp_wait(&sm.stg_full, stg_f & 1, abort)) return false;
    tc_fence_after();
    q_copy<true>(staging_ptr(sm), r, true, q_taddr, sm.qhi);
    tc_fence_before();
    arrive_for_mma<true, true>(&sm.q_full);
    ++stg_f;
    if (!wait_empty) {
      mbar_arrive(&sm.q_read);
      if (threadIdx.x == kEdgeThread0) {
        if (!mbar_wait(&sm.q_read, q_takes & 1, abort)) return false;
        mbar_arrive(&sm.stg_empty);
      }
      ++q_takes;
    }
    return true;
  };
  auto take_q = [&](const Item& it, bool wait_empty, uint32_t it_done) -> bool {
    if (kPair) return take_q_pair(wait_empty, it_done);
    const uint32_t slot = q_pos % kSlots;
    if (wait_empty && !warp_wait(&sm.q_empty, it_done & 1, abort)) return false;
    if (!warp_wait(&sm.full[slot], (q_pos / kSlots) & 1, abort)) return false;
    if (kMode == kModeVerify8) mbar_arrive(&sm.conv[slot]);
    tc_fence_after();
    q_copy<kPair>(sm.tile[slot], r, !is_verify<kMode>() || r < kVerifyHeadsPerTile * a.vrows,
                  q_taddr, sm.qhi);
    tc_fence_before();
    arrive_for_mma<kPair, true>(&sm.q_full);
    mbar_arrive(&sm.q_read);
    if (threadIdx.x == kEdgeThread0) {
      if (!mbar_wait(&sm.q_read, q_takes & 1, abort)) return false;
      mbar_arrive(&sm.empty[slot]);
    }
    ++q_takes;
    q_pos += (has_gate<kMode, kW>() ? 2 : 1) + (kW ? 1 : 2) * it.n;
    return true;
  };
  // The item's gate tile sits at ring position pos (after Q, K0 and, when the item has two
  // key tiles or more, K1). Its slot's previous fill is the item's own Q tile or the
  // previous item's last V tile, both known to have landed (the previous epilogue waited for
  // its last P V), so the parity wait is safe. The slot is handed back once all 128 edge
  // threads have copied their row.
  uint32_t g_takes = 0;
  auto take_gate = [&](uint32_t pos, uint4 (&sg)[kDim / 8]) -> bool {
    if (kPair) {   // from the staging buffer, handed back once all 128 rows are read
      if (!warp_wait(&sm.stg_full, stg_f & 1, abort)) return false;
      gate_from_tile(staging_ptr(sm), r, sg);
      ++stg_f;
      mbar_arrive(&sm.g_read);
      if (threadIdx.x == kEdgeThread0) {
        if (!mbar_wait(&sm.g_read, g_takes & 1, abort)) return false;
        mbar_arrive(&sm.stg_empty);
      }
      ++g_takes;
      return true;
    }
    const uint32_t slot = pos % kSlots;
    if (!warp_wait(&sm.full[slot], (pos / kSlots) & 1, abort)) return false;
    gate_from_tile(sm.tile[slot], r, sg);
    mbar_arrive(&sm.g_read);
    if (threadIdx.x == kEdgeThread0) {
      if (!mbar_wait(&sm.g_read, g_takes & 1, abort)) return false;
      mbar_arrive(&sm.empty[slot]);
    }
    ++g_takes;
    return true;
  };
  // Item i+1's Q goes into TMEM as soon as item i's last S = Q K^T has read Q; item i's
  // gate sigmoids are computed while its tiles run, and its epilogue once its last P V
  // is done.
  Item cur, nxt;
  if (!next_item(cur)) return;
  uint32_t cur_q = q_pos;   // ring position of the current item's Q tile
  if (!take_q(cur, false, 0)) return;
  uint4 sg[kDim / 8];
  uint32_t it_done = 0;
  // e4m3 caches: the edge warps walk every fill of the ring in order and widen each K and V
  // tile of the item (ring order K0, then K_j, V_{j-1} for j >= 1, then V_{n-1})
  auto widen_item = [&](const Item& it, uint32_t q_at) -> bool {
    const int kvh = it.h / kGroup;
    // fill f (1 .. 2n) after the item's Q: K0, then K_j, V_{j-1} for j >= 1, then V_{n-1}
    auto fill_tile = [&](int f, bool& is_v) -> int {
      if (f == 1) { is_v = false; return 0; }
      if (f == 2 * it.n) { is_v = true; return it.n - 1; }
      is_v = (f & 1) != 0;
      return is_v ? (f - 3) / 2 : f / 2;
    };
    float scv[kWideRows], scv_next[kWideRows];
    bool is_v;
    int tile = fill_tile(1, is_v);
    load_row_scales(a, is_v ? a.v_scale : a.k_scale, it.seq, kvh, it.kt0 + tile, r, scv_next);
    for (int f = 1; f <= 2 * it.n; ++f) {
#pragma unroll
      for (int k = 0; k < kWideRows; ++k) scv[k] = scv_next[k];
      if (f < 2 * it.n) {
        tile = fill_tile(f + 1, is_v);
        load_row_scales(a, is_v ? a.v_scale : a.k_scale, it.seq, kvh, it.kt0 + tile, r, scv_next);
      }
      if (!widen_e4m3(sm, q_at + f, scv, r, abort)) return false;
    }
    return true;
  };
  while (true) {
    if (kMode == kModeVerify8 && !widen_item(cur, cur_q)) return;
    if (has_gate<kMode, kW>()) {
      if (!take_gate(cur_q + (cur.n >= 2 ? 3 : 2), sg)) return;
      // rows past the sequence's end are never stored: their lookups are skipped (whole
      // warps in a ragged last tile, which frees the L1 for the rows that count)
      if (cur.mt * kTileM + r < cur.rows) gate_sigmoid(sg);
    }
    const bool have_next = next_item(nxt);
    const uint32_t nxt_q = q_pos;
    if (have_next && !take_q(nxt, true, it_done)) return;
    if (is_verify<kMode>()) {
      if (!epilogue_partial(sm, a, cur, tmem, lane_off, r, it_done, abort)) return;
    } else if (!kW && !epilogue<kMode, kPair>(sm, a, tm_o, cur, tmem, lane_off, r, it_done, sg, abort)) {
      return;
    }
    ++it_done;
    if (!have_next) break;
    cur = nxt;
    cur_q = nxt_q;
  }
}

// kPair (causal, bidirectional and stored-mask passes): the kernel runs as clusters of two
// CTAs that share each K and V tile. A pair item is one row tile of two neighbouring query
// heads of a KV group (the even CTA's head first); the even CTA issues every MMA for both
// (cta_group::2, M = 256: each CTA's 128 rows of Q, S, P and O stay in its own shared and
// tensor memory), and each CTA loads only its half of every K and V tile, so each SM's
// shared memory carries half the key and value traffic of a single CTA's. The tensor
// cores' commits arrive on the barriers of both CTAs; the odd CTA's softmax and edge warps
// arrive on the even CTA's barriers (one arrival per warp) for the MMA warps there.
template <int kMode, bool kW, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ AttnArgs a) {
  constexpr bool kCluster = kPair || kMode == kModeVerify8;
  // The dynamic shared memory is declared 1024-byte aligned (the 128-byte swizzle of TMA
  // and the MMA descriptors needs it); every thread checks it before using any of it.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0u) {
    if (threadIdx.x == 0) record_abort(a.status, kDevBadLaunch);
    if (kCluster) {   // the peer's cluster barriers (after set-up, [before the release,] at exit)
      cluster_sync_all();
      if (kPair) cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool leader = !kPair || (blockIdx.x & 1) == 0;   // a pair's MMA-issuing CTA
  volatile int* abort = &sm.abort;
  if (threadIdx.x == 0) {
    sm.abort = 0;
    for (int i = 0; i < kMaxSlots; ++i) {   // a pair's ring has four slots
      mbar_init(&sm.full[i], 1);
      // refilled once both MMA warps have passed the fill and its consumer released it
      // (weights pass: the score warp alone walks the ring); in a pair's odd CTA, once the
      // pair's commit released it
      mbar_init(&sm.empty[i], !leader ? 1 : kW ? 2 : 3);
    }
    // barriers the MMA warps wait on: per thread of this CTA, plus in a pair one arrival per
    // warp of the odd CTA
    mbar_init(&sm.q_full, kPair ? 128 + 4 : 128);
    mbar_init(&sm.q_empty, 1);
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_free, kPair ? 256 + 8 : 256);       // both softmax warpgroups
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.p_full[i], kPair ? 128 + 4 : 128);
      mbar_init(&sm.p_empty[i], 1);
    }
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.o_free, kPair ? 128 + 4 : 128);
    mbar_init(&sm.st_full, 256);
    mbar_init(&sm.st_empty, 128);
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.drain_pv, 1);
    mbar_init(&sm.q_read, 128);
    // e4m3 caches: conv counts this CTA's 128 edge threads (and, for a K or V fill, the 32 KiB
    // the peer copies in); peer_free the peer's producer, once per fill of the slot
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sm.conv[i], 128);
      mbar_init(&sm.peer_free[i], 1);
    }
    mbar_init(&sm.g_read, 128);
    mbar_init(&sm.mx_bar, 256);
    mbar_init(&sm.stg_full, 1);
    mbar_init(&sm.stg_empty, 1);
    mbar_init(&sm.o_st, 128);
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if (has_gate<kMode, kW>()) tma_prefetch_desc(&tm_g);
    if (kPair) tma_prefetch_desc(&tm_o);
  }
  if (warp == 1) {
    if (kPair) {
      tmem_alloc_pair(&sm.tmem_base, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&sm.tmem_base, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // the peer arrives on this CTA's barriers (and, in a pair, its MMAs use this CTA's tensor
  // memory): both CTAs' barriers are initialised and their columns allocated before either runs
  if (kCluster) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // a pair's MMAs address both CTAs' tensor memory at the even CTA's column: both CTAs
  // check that the allocation gave the same columns in each (else neither runs)
  bool run = true;
  if (kPair) {
    const uint32_t other =
        ld_shared_cluster_u32(mapa_shared(smem_u32(&sm.tmem_base), (blockIdx.x & 1) ^ 1u));
    if (other != tmem) {
      run = false;
      if (threadIdx.x == 0) record_abort(a.status, kDevBadLaunch);
    }
  }

  if (run) {
    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue));
      if (warp == 0) producer<kMode, kW, kPair>(sm, &tm_q, &tm_k, &tm_v, &tm_g, a, abort);
      if ((warp == 1 || warp == 2) && leader)
        mma_issuer<kMode, kW, kPair>(sm, a, tmem, abort, warp == 2);
      if (kPair && warp == 3) stage_producer<kMode, kPair>(sm, &tm_q, &tm_g, a, abort);
    } else if (warp < 12) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
      softmax_worker<kMode, kW, kPair>(sm, a, tmem, (warp - 4) >> 2, abort);
    } else {
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEdge));
      edge_worker<kMode, kW, kPair>(sm, a, &tm_o, tmem, abort);
      // the output tiles' tensor stores complete before the CTA leaves
      if (kPair && threadIdx.x == kEdgeThread0) bulk_wait_group0();
    }
  }
  tc_fence_before();
  __syncthreads();
  // a pair: the even CTA's MMAs into this CTA's tensor memory have completed (its MMA warps
  // waited for their last commits) and neither CTA arrives on the other's barriers any more
  if (kPair) cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (kPair) tmem_dealloc_pair(tmem, kTmemCols);
    else tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && sm.abort) record_abort(a.status, sm.abort);
  // a CTA of a pair leaves only when its peer no longer writes into its shared memory or
  // arrives on its barriers (every wait before this point is bounded)
  if (kCluster) cluster_sync_all();
}

constexpr int kCombineChunkSlots = 3;   // (M, l) pairs per lane: up to 96 chunks
static_assert(kVerifyChunkCap / 4 <= 32 * kCombineChunkSlots, "a verify row has at most 96 chunks");

// kDpl consecutive floats (8 bytes aligned; 16 when kDpl is a multiple of 4) into v.
template <int kDpl>
__device__ __forceinline__ void load_dims(const float* p, float (&v)[kDpl]) {
  if constexpr (kDpl % 4 == 0) {
#pragma unroll
    for (int i = 0; i < kDpl / 4; ++i) {
      const float4 t = reinterpret_cast<const float4*>(p)[i];
      v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kDpl / 2; ++i) {
      const float2 t = reinterpret_cast<const float2*>(p)[i];
      v[2 * i] = t.x; v[2 * i + 1] = t.y;
    }
  }
}

// Verify combine (TensorFold PR #1080, "qwen CUDA: long-prompt prefill 5.4x faster", the
// attn_partial commit: key chunks processed apart, then merged per row). kSplit warps per
// (sequence, query head, row), warp q taking dims (256 / kSplit) q .. , lane l kDpl = 8 /
// kSplit consecutive dims of them. With M = max_c M_c over the chunks the row saw keys in,
// O = sum_c 2^(M_c - M) O_c and L = sum_c 2^(M_c - M) l_c (exact power-of-two scales, chunks
// in order), o = bf16(O / L), out = bf16(o * bf16(sigmoid(g))). The loads do not wait on one
// another: all (M_c, l_c) are read at once, the partial rows several chunks ahead, and only
// the sums run in chunk order; calls with few rows split each row over more warps so that
// the grid still covers the SMs (the bits do not depend on the split).
template <int kSplit>
__global__ void __launch_bounds__(256) verify_combine_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int kDpl = 8 / kSplit;                 // dims per lane
  constexpr int kBatch = kDpl == 8 ? 4 : 8;        // chunks' partial values in flight
  const int lane = threadIdx.x & 31;
  const int wg = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int w = wg / kSplit, part = wg % kSplit;
  if (w >= a.n_seq * kHeads * a.vrows) return;
  const int rr = w % a.vrows;
  const int h = (w / a.vrows) % kHeads;
  const int b = w / (a.vrows * kHeads);
  const int kvh = h / kGroup, half = (h % kGroup) / kVerifyHeadsPerTile;
  const int lanep = rr * kVerifyHeadsPerTile + h % kVerifyHeadsPerTile;
  const int tiles = (a.seq_len[b] + a.vrows + kTileN - 1) / kTileN;
  const int chunks = (tiles + a.chunk_tiles - 1) / a.chunk_tiles;
  const size_t slot0 = (((size_t)b * kKvHeads + kvh) * 2 + half) * a.n_chunks;
  const int d0 = (kDim / kSplit) * part + kDpl * lane;   // this lane's first dim
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
  // every chunk's (M_c, l_c) at once: lane l holds chunks l, l + 32 and l + 64
  float2 mlv[kCombineChunkSlots];
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kCombineChunkSlots; ++k) {
    const int c = lane + 32 * k;
    mlv[k] = c < chunks ? ml[(slot0 + c) * kVerifyLanes + lanep] : make_float2(0.f, 0.f);
    if (mlv[k].y > 0.f) M = fmaxf(M, mlv[k].x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
  // the chunks in order, kBatch chunks' partial values in flight at a time; chunk c's scale
  // and sum come from lane c % 32
  float o[kDpl];
#pragma unroll
  for (int i = 0; i < kDpl; ++i) o[i] = 0.f;
  float L = 0.f;
  for (int c0 = 0; c0 < chunks; c0 += kBatch) {
    float p[kBatch][kDpl];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (c0 + j < chunks)
        load_dims<kDpl>(a.part_o + ((slot0 + c0 + j) * kVerifyLanes + lanep) * kDim + d0, p[j]);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int c = c0 + j;
      if (c >= chunks) break;
      const int k = c >> 5;   // the same for every lane
      const float2 mine = k == 0 ? mlv[0] : (k == 1 ? mlv[1] : mlv[2]);
      const float mc = __shfl_sync(0xFFFFFFFFu, mine.x, c & 31);
      const float lc = __shfl_sync(0xFFFFFFFFu, mine.y, c & 31);
      if (!(lc > 0.f)) continue;
      const float f = ldexpf(1.0f, (int)(mc - M));   // an exact power of two
      L = fmaf(f, lc, L);
#pragma unroll
      for (int i = 0; i < kDpl; ++i) o[i] = fmaf(f, p[j][i], o[i]);
    }
  }
  const float inv = L > 0.f ? 1.0f / L : 0.f;
  const size_t row = (size_t)b * a.vrows + rr;
  const uint32_t* gp = reinterpret_cast<const uint32_t*>(a.qg + (row * kHeads + h) * kQgStride + kDim + d0);
  uint32_t* op = reinterpret_cast<uint32_t*>(a.out + row * kOutRow + h * kDim + d0);
  uint32_t res[kDpl / 2];
#pragma unroll
  for (int k = 0; k < kDpl / 2; ++k) {
    const uint32_t ob = pack_bf16x2(o[2 * k] * inv, o[2 * k + 1] * inv);
    res[k] = mul_bf16x2(ob, sigmoid_pair(__ldg(gp + k)));
  }
  if constexpr (kDpl == 8) {
    *reinterpret_cast<uint4*>(op) = make_uint4(res[0], res[1], res[2], res[3]);
  } else if constexpr (kDpl == 4) {
    *reinterpret_cast<uint2*>(op) = make_uint2(res[0], res[1]);
  } else {
    op[0] = res[0];
  }
}

// Test hook: one thread waits, with a bound of `limit` cycles, on an mbarrier that nothing
// arrives on, through the same bounded wait and status recording every kernel here uses.
__global__ void wait_timeout_kernel(long long limit, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x != 0) return;
  abort = 0;
  mbar_init(&bar, 1);
  mbar_fence_init();
  volatile int* ab = &abort;
  if (!mbar_wait(&bar, 0, ab, limit)) record_abort(status, abort);
}

}  // namespace

cudaError_t launch_wait_timeout(long long limit, int* status, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(limit, status);
  return cudaGetLastError();
}

size_t attn_smem_bytes() { return sizeof(AttnSmem); }

cudaError_t launch_verify_combine(const AttnArgs& a, int sm_count, cudaStream_t s) {
  // one warp per row when the rows alone fill the SMs (about 24 warps resident per SM),
  // else the row split over 2 or 4 warps
  const int rows = a.n_seq * kHeads * a.vrows;
  const int fill = 24 * (sm_count > 0 ? sm_count : 1);
  if (rows * 2 > fill) {
    verify_combine_kernel<1><<<(rows + 7) / 8, 256, 0, s>>>(a);
  } else if (rows * 4 > fill) {
    verify_combine_kernel<2><<<(rows * 2 + 7) / 8, 256, 0, s>>>(a);
  } else {
    verify_combine_kernel<4><<<(rows * 4 + 7) / 8, 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t attn_upload_sigmoid_table(const uint16_t* host_table) {
  return cudaMemcpyToSymbol(g_sigmoid_bf16, host_table, sizeof(g_sigmoid_bf16));
}

cudaError_t attn_set_smem_attribute() {
  const int bytes = (int)attn_smem_bytes();
  const void* kernels[] = {
      (const void*)attn_kernel<kModeCausal, false, false>,
      (const void*)attn_kernel<kModeBidir, false, false>,
      (const void*)attn_kernel<kModeMask, false, false>,
      (const void*)attn_kernel<kModeVerify, false, false>,
      (const void*)attn_kernel<kModeBatch, false, false>,
      (const void*)attn_kernel<kModeVerify8, false, false>,
      (const void*)attn_kernel<kModeMask, true, false>,
      (const void*)attn_kernel<kModeCausal, false, true>,
      (const void*)attn_kernel<kModeBidir, false, true>,
      (const void*)attn_kernel<kModeMask, false, true>,
      (const void*)attn_kernel<kModeBatch, false, true>,
  };
  for (const void* k : kernels) {
    const cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {
cudaLaunchConfig_t pair_config(unsigned grid, size_t smem, cudaStream_t s,
                               cudaLaunchAttribute (&attr)[1]) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}
}  // namespace

cudaError_t attn_max_pair_clusters(int* n) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(2, attn_smem_bytes(), nullptr, attr);
  return cudaOccupancyMaxActiveClusters(n, attn_kernel<kModeVerify8, false, false>, &cfg);
}

cudaError_t attn_max_gated_pair_clusters(int* n) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(2, attn_smem_bytes(), nullptr, attr);
  return cudaOccupancyMaxActiveClusters(n, attn_kernel<kModeCausal, false, true>, &cfg);
}

cudaError_t launch_attn(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                        const CUtensorMap& tm_g, const CUtensorMap& tm_o, const AttnArgs& a,
                        int grid, cudaStream_t s) {
  const size_t smem = attn_smem_bytes();
  if (a.pair || a.mode == kModeVerify8) {
    // clusters of two CTAs (grid even)
    if (grid < 2 || (grid & 1)) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pair_config((unsigned)grid, smem, s, attr);
    if (a.mode == kModeVerify8)
      return cudaLaunchKernelEx(&cfg, attn_kernel<kModeVerify8, false, false>, tm_q, tm_k, tm_v,
                                tm_g, tm_o, a);
    if (a.weights_pass) return cudaErrorInvalidValue;
    if (a.mode == kModeCausal)
      return cudaLaunchKernelEx(&cfg, attn_kernel<kModeCausal, false, true>, tm_q, tm_k, tm_v,
                                tm_g, tm_o, a);
    if (a.mode == kModeBidir)
      return cudaLaunchKernelEx(&cfg, attn_kernel<kModeBidir, false, true>, tm_q, tm_k, tm_v,
                                tm_g, tm_o, a);
    if (a.mode == kModeMask)
      return cudaLaunchKernelEx(&cfg, attn_kernel<kModeMask, false, true>, tm_q, tm_k, tm_v,
                                tm_g, tm_o, a);
    if (a.mode == kModeBatch)
      return cudaLaunchKernelEx(&cfg, attn_kernel<kModeBatch, false, true>, tm_q, tm_k, tm_v,
                                tm_g, tm_o, a);
    return cudaErrorInvalidValue;
  }
  if (a.weights_pass) {
    if (a.mode != kModeMask) return cudaErrorInvalidValue;
    attn_kernel<kModeMask, true, false><<<grid, kThreads, smem, s>>>(tm_q, tm_k, tm_v, tm_g, tm_o, a);
  } else if (a.mode == kModeCausal) {
    attn_kernel<kModeCausal, false, false><<<grid, kThreads, smem, s>>>(tm_q, tm_k, tm_v, tm_g, tm_o, a);
  } else if (a.mode == kModeBidir) {
    attn_kernel<kModeBidir, false, false><<<grid, kThreads, smem, s>>>(tm_q, tm_k, tm_v, tm_g, tm_o, a);
  } else if (a.mode == kModeVerify) {
    attn_kernel<kModeVerify, false, false><<<grid, kThreads, smem, s>>>(tm_q, tm_k, tm_v, tm_g, tm_o, a);
  } else if (a.mode == kModeBatch) {
    attn_kernel<kModeBatch, false, false><<<grid, kThreads, smem, s>>>(tm_q, tm_k, tm_v, tm_g, tm_o, a);
  } else {
    attn_kernel<kModeMask, false, false><<<grid, kThreads, smem, s>>>(tm_q, tm_k, tm_v, tm_g, tm_o, a);
  }
  return cudaGetLastError();
}

}  // namespace ga
