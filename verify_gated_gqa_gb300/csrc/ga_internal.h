// Internal definitions shared by the library's translation units (not part of the ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ga_attn.h"

namespace ga {

constexpr int kHeads = GA_N_Q_HEADS;          // 24
constexpr int kKvHeads = GA_N_KV_HEADS;       // 2
constexpr int kGroup = kHeads / kKvHeads;     // 12
constexpr int kDim = GA_HEAD_DIM;             // 256
constexpr int kQgStride = 2 * kDim;           // 512: q then gate, per head
constexpr int kRowElems = kHeads * kQgStride; // 12288 bf16 per fused row
constexpr int kOutRow = kHeads * kDim;        // 6144 bf16 per output row
constexpr int kHalfRot = GA_ROPE_DIMS / 2;    // 32
constexpr float kEps = 1e-6f;
constexpr double kEpsD = 1e-6;
constexpr double kRopeBase = 1e7;

constexpr int kTileM = 128;  // query rows per attention tile
constexpr int kTileN = 128;  // keys per attention tile

// Attention kernel variants.
enum AttnMode : int {
  kModeCausal = 0,   // key j visible iff j <= q_base + r
  kModeBidir = 1,    // every key j < T
  kModeMask = 2,     // stored bit mask (from the mask prepass)
  kModeVerify = 3,   // few-row windows over long caches: split-key partials (see below)
  kModeBatch = 4,    // several causal prefills (windows) over paged caches in one launch
  kModeVerify8 = 5,  // verify over e4m3 caches, widened to bf16 in the shared-memory slot
};

// Batch mode: sequence b's rows are packed rows batch_row0[b] .. + batch_rows[b] - 1 (row r
// at position batch_qbase[b] + r, seeing keys 0 .. batch_qbase[b] + r of its own paged
// cache). A work item is (row tile entry, query head); the entries, (b << 16) | mt, are
// sorted by the host so that the tiles with the most keys come first.
constexpr int kBatchMaxEntries = 256;   // 128-row tiles per launch (the host loops over groups)

// Verify mode: a work item is (sequence, KV head, half of the query group, key chunk). Its
// 128-lane row tile packs 6 query heads x vrows rows of one sequence (lane 6 rr + hh for
// row rr, head 12 kvh + 6 half + hh; lanes past 6 vrows are padding). The item writes the
// unnormalised partial O (fp32) and its M, l per lane; a combine kernel merges the chunks.
constexpr int kVerifyHeadsPerTile = 6;
constexpr int kVerifyMaxRows = 16;
constexpr int kVerifyLanes = kVerifyHeadsPerTile * kVerifyMaxRows;   // 96
constexpr int kVerifyMaxSeq = 64;       // sequences per launch (the host loops over groups)
// Work items (chunk x sequence x KV head x half group) of one verify launch at most: the
// partial workspace holds kVerifyChunkCap / (4 n_seq) chunks per sequence, 80 at n_seq = 1.
constexpr int kVerifyChunkCap = 320;

// Stored-mask bits, as the mask prepass writes them for the attention kernel. Key j of a
// 32-key word sits at bit 8 (j % 4) + 7 - j / 4: shifted left by s = 0..7, the word holds
// keys 4s .. 4s+3 in the top bits of its four bytes, from which one byte permute with sign
// replication builds the 16-bit keep masks of the bf16 score pairs (4s, 4s+1) and
// (4s+2, 4s+3).
__host__ __device__ constexpr int mask_bit_pos(int j) { return 8 * (j & 3) + 7 - (j >> 2); }
// Tile flags: one byte per (128-row tile, 128-key tile), rows of this many bytes.
constexpr int kMaskFlagStride = GA_MASKED_MAX_TOKENS / kTileN;   // 64

struct AttnArgs {
  const uint16_t* qg;       // [rows][24][512]
  const uint16_t* w_q;      // [256]
  const uint16_t* cos_tab;  // [table_rows][32]
  const uint16_t* sin_tab;
  uint16_t* out;            // [rows][6144]
  float* row_stats;         // nullable [24][rows][2]
  uint16_t* weights;        // weights pass: [24][rows][T]
  int* hidden_rows;         // nullable
  const uint32_t* mask_bits;  // [rows_pad][mask_words]: word w holds keys 32w .. 32w+31, key
                              // 32w + j at bit mask_bit_pos(j)
  const uint8_t* tile_flags;  // [row_tiles][kMaskFlagStride] (128 rows x 128 keys), 1 = a
                              // visible key
  int* status;              // device status word
  int rows, T, q_base, mode, weights_pass;
  int head0, n_heads;       // causal, bidirectional, stored mask: the query heads processed
  int pair;                 // causal, bidirectional, stored mask: clusters of two CTAs that
                            // share each K/V tile (n_items counts row tiles x head pairs;
                            // tm_k / tm_v hold half tiles: box 64 x 64 x 1 x 4, 64 x 128 x 1 x 2)
  int row_tiles, key_tiles, mask_words;
  int n_items;
  // verify mode
  int n_seq, vrows, chunk_tiles, n_chunks;
  int seq_len[kVerifyMaxSeq];   // L per sequence: row rr sits at position L + rr
  float* part_o;                // [n_seq][2][2][n_chunks][96][256]
  float* part_ml;               // [n_seq][2][2][n_chunks][96][2]: M, l
  // verify over paged caches (page_table null: contiguous caches, one per sequence):
  // key tile kt of sequence b is slot (kt % page_tiles) * 128 of page
  // page_table[b * max_pages + kt / page_tiles] of the page pools
  const int* page_table;
  int page_tiles, max_pages, n_pages;
  // verify over e4m3 caches: scales [n_seq][cache_cap][2] fp32 of the key and value rows
  const float* k_scale;
  const float* v_scale;
  int cache_cap;
  // batch mode (n_seq sequences, n_items = n_entries * 24)
  int n_entries;
  int batch_row0[kVerifyMaxSeq], batch_rows[kVerifyMaxSeq], batch_qbase[kVerifyMaxSeq];
  int batch_seq[kVerifyMaxSeq];     // the page-table row of each sequence (piece) of the launch
  uint32_t batch_entry[kBatchMaxEntries];
};

// Launchers (defined next to their kernels). Return a cudaError_t.
// Launchers of the prologue kernel (ga_prologue.cu); sm_count sizes its persistent grid.
cudaError_t launch_k_prologue(const uint16_t* k_raw, const uint16_t* w_k, const uint16_t* cos_tab,
                              const uint16_t* sin_tab, int n_tok, int pos_base, uint16_t* k_prep,
                              int sm_count, cudaStream_t s);
// Prepared query rows of several sequences: token t of sequence t / rows_per_seq sits at
// position seq_base[t / rows_per_seq] + t % rows_per_seq; or, with row_start set (n_seq
// ascending starts, row_start[n_seq] = the total), token t of the sequence b with
// row_start[b] <= t < row_start[b + 1] sits at seq_base[b] + t - row_start[b].
struct SeqPositions {
  int rows_per_seq;
  int seq_base[kVerifyMaxSeq];
  int n_seq;                        // 0: uniform rows_per_seq
  int row_start[kVerifyMaxSeq + 1];
};
cudaError_t launch_q_prologue_seq(const uint16_t* qg, const uint16_t* w_q, const uint16_t* cos_tab,
                                  const uint16_t* sin_tab, int n_tok, const SeqPositions& sp,
                                  uint16_t* q_prep, int sm_count, cudaStream_t s);
// Merges the verify partials and applies the gate: out[b][rr][h*256 ..].
cudaError_t launch_verify_combine(const AttnArgs& a, int sm_count, cudaStream_t s);
// Prepared query rows: q_prep[r][h][0..255] = rope(norm(qg[r][h][0..255])) at q_base + r,
// for the heads head0 .. head0+n_heads-1 (the other heads' slots are not written).
cudaError_t launch_q_prologue(const uint16_t* qg, const uint16_t* w_q, const uint16_t* cos_tab,
                              const uint16_t* sin_tab, int rows, int q_base, int head0,
                              int n_heads, uint16_t* q_prep, int sm_count, cudaStream_t s);
// Both prologues in one launch: the key rows of n_tok tokens at positions k_pos_base.., then
// the query rows of all 24 heads at q_base.., each with the single launches' results.
cudaError_t launch_qk_prologue(const uint16_t* k_raw, const uint16_t* w_k, int n_tok,
                               int k_pos_base, uint16_t* k_prep, const uint16_t* qg,
                               const uint16_t* w_q, int rows, int q_base, uint16_t* q_prep,
                               const uint16_t* cos_tab, const uint16_t* sin_tab, int sm_count,
                               cudaStream_t s);
// e4m3 cache rows: q[row][0..255] and scale[row] for n_rows rows of 256 bf16 values.
cudaError_t launch_quantize_e4m3(const uint16_t* x, long long n_rows, uint8_t* q, float* scale,
                                 cudaStream_t s);
// The widened bf16 rows out[row][0..255] of n_rows e4m3 rows and their scales.
cudaError_t launch_dequantize_e4m3(const uint8_t* q, const float* scale, long long n_rows,
                                   uint16_t* out, cudaStream_t s);
// Selection mask: mask[r][0..T-1] for rows r < rows from block_scores[r][0..ceil(T/4)-1].
cudaError_t launch_select_mask(const float* scores, long long ld_scores, int rows, int T,
                               int q_base, int top_k, uint8_t* mask, long long ld_mask,
                               cudaStream_t s);
cudaError_t attn_set_smem_attribute();
// Clusters of two attention CTAs (the e4m3 verify variant) that can run at once.
cudaError_t attn_max_pair_clusters(int* n);
// The same for the CTA-pair variants of the causal, bidirectional and stored-mask passes.
cudaError_t attn_max_gated_pair_clusters(int* n);
// Test hook (ga_debug.cu): fp32 tensor-core dot products of n_tiles pairs of 128 x 256 bf16
// tiles, s[n][i][j] = q[n][i] . k[n][j].
cudaError_t probe_set_smem_attribute();
cudaError_t launch_qk_probe(const uint16_t* q, const uint16_t* k, int n_tiles, float* s,
                            int* status, cudaStream_t st);
// Test hook: a bounded wait on a barrier nothing arrives on (records a wait timeout).
cudaError_t launch_wait_timeout(long long limit, int* status, cudaStream_t s);
// Fills the device's table of bf16(sigmoid(g)) for every bf16 g (65536 entries, by bits).
cudaError_t attn_upload_sigmoid_table(const uint16_t* host_table);
size_t attn_smem_bytes();
// tm_q: the prepared queries [rows][24][256] (box 64 dims x 1 head x 128 rows); tm_g: the
// fused rows [rows][24][512], read for their gate halves (box 64 values x 1 head x 128 rows;
// used by the causal, bidirectional and stored-mask passes); tm_o: the output [rows][24][256]
// as a.out (box as tm_q), written by tensor stores in the CTA-pair passes (a.pair).
cudaError_t launch_attn(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                        const CUtensorMap& tm_g, const CUtensorMap& tm_o, const AttnArgs& a,
                        int grid, cudaStream_t s);
cudaError_t launch_mask_prepass(const uint8_t* mask, long long ld_mask, int rows, int T,
                                uint32_t* bits, int mask_words, uint8_t* flags, int key_tiles,
                                cudaStream_t s);

}  // namespace ga
