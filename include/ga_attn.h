/*
 * ga_attn.h -- C ABI of the GB300 (sm_103a) gated grouped-query attention library
 * (libga_attn.so).
 *
 * The operation (pegainfer PR #1151, "feat(qwen4): add the QSA sparse-attention kernel
 * and its golden", §Semantics): split each fused q|gate row, apply (1+w) RMSNorm to q
 * and k (eps 1e-6), rotate dims 0..63 of q and k (rotate-half partial RoPE) from a
 * shared bf16 cos/sin table, score s = bf16(q.k) / 16 over GQA groups of 12 (query
 * head h reads KV head h / 12), softmax in fp32 over the visible keys with the weights
 * rounded to bf16 before the context reduction, reduce P.V, and multiply by
 * bf16(sigmoid(gate)). Output columns are head-major (h * 256 + d).
 *
 * Geometry is compiled in: 24 query heads, 2 KV heads, head_dim 256, 64 rotary dims,
 * eps 1e-6, RoPE base 1e7 (the same page, the commit that replaces the proxy geometry).
 *
 * Conventions for every entry point below:
 *  - Tensor pointers are DEVICE pointers owned by the caller, unless a comment says
 *    HOST. The library never allocates device memory on a call path, and keeps no
 *    pointer after the call returns. bf16 values are passed as their 16-bit patterns
 *    (ga_bf16). All tensors are dense, row-major, without padding unless a leading
 *    dimension argument says otherwise.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *    and is asynchronous: the return value reports argument validation and launch
 *    errors, not the kernels' completion. Calls on different streams are re-entrant.
 *  - Every argument is validated BEFORE any CUDA call (system1-omni PR #99, "run
 *    prompts that share prefixes once per prefix": refusals happen before any
 *    allocation or CUDA call). A zero-row call returns GA_OK without touching the GPU
 *    (pegainfer PR #1151, §What changed: an empty launch is a no-op).
 *  - There is no fallback path: a launch failure is returned as GA_ERR_CUDA with the
 *    CUDA error kept for ga_last_cuda_error() (system1-omni PR #202, "cuda: widen the
 *    attention query tile on sm_89 and sm_120", review §Dispatch/guard: no silent
 *    fallback).
 *  - Kernels never trap. A bounded device-side wait that gives up records an error in
 *    the library's device status word (ga_device_status).
 *  - Pointers that the kernels read or write with 16-byte vector or TMA accesses must be
 *    16-byte aligned (GA_ERR_ALIGN otherwise).
 */
#ifndef GA_ATTN_H
#define GA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GA_ABI_VERSION 1

#define GA_N_Q_HEADS 24
#define GA_N_KV_HEADS 2
#define GA_HEAD_DIM 256
#define GA_ROPE_DIMS 64
#define GA_MASKED_MAX_TOKENS 8192 /* pegainfer PR #1151, §Summary: the 8192-token cap */
#define GA_MAX_TOKENS (1 << 20)   /* index-arithmetic limit of the library */
/* Keys per indexer block (pegainfer PR #1151: a budget of 2048 tokens is 512 blocks). */
#define GA_INDEX_BLOCK_TOKENS 4

typedef uint16_t ga_bf16; /* bfloat16 bit pattern */
typedef void* ga_stream;  /* cudaStream_t */

enum ga_status {
  GA_OK = 0,
  GA_ERR_NULL = -1,      /* a required pointer is NULL */
  GA_ERR_SHAPE = -2,     /* a size is negative or zero where it must be positive */
  GA_ERR_ALIGN = -3,     /* a pointer or leading dimension breaks 16-byte alignment */
  GA_ERR_RANGE = -4,     /* a window, position or size is outside what the call allows */
  GA_ERR_TABLE = -5,     /* the cos/sin table is shorter than the largest position + 1 */
  GA_ERR_WORKSPACE = -6, /* workspace missing, misaligned or smaller than required */
  GA_ERR_DEVICE = -7,    /* current device is not sm_103 or refused the smem opt-in */
  GA_ERR_CUDA = -8,      /* a CUDA call failed; see ga_last_cuda_error() */
  GA_ERR_GEOMETRY = -9   /* ga_check_geometry: not the compiled geometry */
};

/* Geometry a caller expects; ga_check_geometry compares it with the compiled constants
 * (pegainfer PR #1151, §What changed: the wrapper validates its geometry against the
 * compiled constants before sizing any buffer). */
typedef struct ga_geometry {
  int n_q_heads;    /* 24 */
  int n_kv_heads;   /* 2 */
  int head_dim;     /* 256 */
  int rope_dims;    /* 64 */
  float eps;        /* 1e-6 */
  double rope_base; /* 1e7 */
} ga_geometry;

/* GA_ABI_VERSION of the loaded library. */
int ga_abi_version(void);

/* GA_OK if *g equals the compiled geometry, GA_ERR_GEOMETRY if not, GA_ERR_NULL for NULL. */
int ga_check_geometry(const ga_geometry* g);

/* Static English text for a status code (never NULL). */
const char* ga_status_string(int status);

/* The cudaError_t value behind the calling thread's last GA_ERR_CUDA (0 if none). */
int ga_last_cuda_error(void);

/* Number of CUDA runtime calls this library has made in this process (diagnostic: a
 * refused call must not change it). Makes no CUDA call itself. */
unsigned long long ga_debug_cuda_calls(void);

/* Reads the current device's status word, written by kernels whose bounded waits gave
 * up or whose inputs failed a device-side check (0 = no error, 1 = wait timeout, 2 = bad
 * launch configuration, 3 = a page-table entry outside the page pool, see
 * ga_attn_verify_paged). Synchronises the device. clear != 0 resets the word afterwards. */
int ga_device_status(int* status_out, int clear);

/* Test hook for failure detection (no counterpart in the pages): launches a one-thread
 * kernel that waits, bounded by limit_cycles SM clock cycles (1 .. 2e9), on an mbarrier
 * that nothing arrives on. The wait gives up, the kernel records the wait-timeout status
 * (1) in the device status word and returns: the same bounded wait and recording every
 * kernel of the library uses, without a fault, a trap or a hang. Read the result with
 * ga_device_status. Errors: RANGE, DEVICE, CUDA. */
int ga_debug_wait_timeout(long long limit_cycles, ga_stream stream);

/* Selects how the attention passes run (no counterpart in the pages; the results are the
 * same bits either way). mode 2: the causal, bidirectional, stored-mask and batched passes
 * as clusters of two CTAs that share each key and value tile, two query heads of one KV
 * group per pair item, whenever the call's heads come in such pairs (every call through the
 * ABI does: the KV-group entry points take whole groups of 12); the weights pass and the
 * verify passes on single CTAs. mode 1 (the default): the same, except that causal,
 * bidirectional and stored-mask calls over fewer than 2,048 keys run on single CTAs, which
 * are faster there. mode 0: every pass on single CTAs (one CTA per 128-row tile and head).
 * Process-wide; takes effect from the next call. Returns the previous mode (0, 1 or 2).
 * Errors: RANGE (mode outside 0 .. 2). Makes no CUDA call. */
int ga_debug_set_cta_pairs(int mode);

/* Test hook: the fp32 dot products the tensor cores form for the scores, before any
 * rounding. For each of n_tiles tiles, s[n][i][j] = q[n][i] . k[n][j] over 256 dims, computed
 * exactly as the attention kernel computes S = Q K^T (tcgen05.mma kind::f16, M128 N128,
 * sixteen K16 steps accumulating in fp32 in tensor memory, operands in shared memory in the
 * kernel's 128-byte-swizzled layout). The score is the bf16 rounding of this value (pegainfer
 * PR #1151, the commit that adds the attention reader: "the bf16 GEMM result"); the fp32
 * reduction order inside the tensor core is the hardware's, and the tests use this hook to
 * bound its distance from the exact dot product.
 *   q, k   [n_tiles][128][256] bf16, 16-byte aligned
 *   s      [n_tiles][128][128] fp32, 16-byte aligned
 * Rules: 0 <= n_tiles <= 65535 (0 is a no-op).
 * Errors: NULL, SHAPE, RANGE, ALIGN, DEVICE, CUDA. */
int ga_debug_qk_fp32(const ga_bf16* q, const ga_bf16* k, int n_tiles, float* s,
                     ga_stream stream);

/* HOST helper. Fills cos_out and sin_out (HOST arrays of n_pos * 32 values each,
 * [position][pair]) with cos and sin of p * 1e7^(-2i/64) for positions p < n_pos and
 * pairs i < 32, each computed in double and rounded once to bf16 (pegainfer PR #1151,
 * review F4: a double pow, rounded once; §What changed: one shared table, no device
 * trigonometry). Pair i rotates dims i and i + 32. Makes no CUDA call. */
int ga_rope_table_host(int n_pos, ga_bf16* cos_out, ga_bf16* sin_out);

/* K prologue (pegainfer PR #1151, §What changed: one key pass (1+w)-norms and partially
 * rotates every token's two key heads once, because all twelve query heads of a KV head
 * read the same prepared key).
 *   k_raw  [n_tok][2][256]  raw keys of tokens at positions pos_base .. pos_base+n_tok-1
 *   w_k    [256]            key norm weight w (applied as 1 + w)
 *   cos_tab, sin_tab [table_rows][32]; table_rows >= pos_base + n_tok
 *   k_prep [n_tok][2][256]  output: bf16(rope(norm(k))); may not alias k_raw
 * Errors: NULL, SHAPE (n_tok < 0), RANGE (pos_base < 0 or n_tok > GA_MAX_TOKENS), TABLE,
 * ALIGN (k_raw, k_prep, cos_tab, sin_tab, w_k), DEVICE, CUDA. */
int ga_k_prologue(const ga_bf16* k_raw, const ga_bf16* w_k, const ga_bf16* cos_tab,
                  const ga_bf16* sin_tab, int table_rows, int n_tok, int pos_base,
                  ga_bf16* k_prep, ga_stream stream);

/* Query prologue: the same (1+w) RMSNorm and partial RoPE for the q half of every fused
 * row and head (pegainfer PR #1151, §Semantics: q is split from the fused q|gate row,
 * normed and rotated at its own position). ga_attn_prefill runs it itself; it is exposed
 * so that a caller can time or reuse the prepared queries (ga_attn_prefill_prepared).
 *   qg      [rows][24][512]  fused rows of positions q_base .. q_base+rows-1
 *   w_q     [256]            query norm weight w (applied as 1 + w)
 *   cos_tab, sin_tab [table_rows][32]; table_rows >= q_base + rows
 *   q_prep  [rows][24][256]  output: bf16(rope(norm(q))); may not overlap qg
 * Errors: NULL, SHAPE (rows < 0), RANGE (q_base < 0 or rows > GA_MAX_TOKENS), TABLE,
 * ALIGN (qg, w_q, cos_tab, sin_tab, q_prep), DEVICE, CUDA. */
int ga_q_prologue(const ga_bf16* qg, const ga_bf16* w_q, const ga_bf16* cos_tab,
                  const ga_bf16* sin_tab, int table_rows, int rows, int q_base,
                  ga_bf16* q_prep, ga_stream stream);

/* Both prologues in one launch (pegainfer PR #1151, §What changed and §Semantics: the key
 * pass and the query pass take the same (1+w) norm and partial rotation):
 * ga_k_prologue over n_tok key tokens and ga_q_prologue over rows fused query rows, with
 * the same results bit for bit. One persistent grid walks the
 * key rows and then the query rows, so the two share every SM instead of competing as two
 * launches on two streams would.
 *   k_raw, w_k, n_tok, k_pos_base, k_prep: as ga_k_prologue's k_raw, w_k, n_tok, pos_base
 *                            and k_prep
 *   qg, w_q, rows, q_base, q_prep: as ga_q_prologue's; q_prep may not overlap qg, and no
 *                            output may overlap the other call's inputs or output
 *   cos_tab, sin_tab [table_rows][32]; table_rows >= k_pos_base + n_tok and
 *                            table_rows >= q_base + rows
 * Errors: NULL, SHAPE (n_tok < 0 or rows < 0), RANGE, TABLE, ALIGN (every pointer),
 * DEVICE, CUDA; all checked before anything is launched. */
int ga_qk_prologue(const ga_bf16* k_raw, const ga_bf16* w_k, int n_tok, int k_pos_base,
                   ga_bf16* k_prep, const ga_bf16* qg, const ga_bf16* w_q, int rows, int q_base,
                   ga_bf16* q_prep, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                   int table_rows, ga_stream stream);

/* Causal / prefix-window / bidirectional gated GQA attention (system1-omni PR #202,
 * §Scope: full pass, causal or bidirectional, and causal prefix windows at q_base).
 *   qg      [rows][24][512]  fused rows of query positions q_base .. q_base+rows-1; per
 *                            head the first 256 values are q, the last 256 the gate
 *   k_prep  [T][2][256]      prepared keys (ga_k_prologue) of positions 0 .. T-1
 *   v       [T][2][256]      values
 *   w_q     [256]            query norm weight w (applied as 1 + w)
 *   cos_tab, sin_tab [table_rows][32]; table_rows >= q_base + rows
 *   causal  1: row r sees keys j <= q_base + r;  0: bidirectional, every key j < T
 *           (q_base must then be 0)
 *   out     [rows][24 * 256] bf16, head-major columns. It may not overlap any input;
 *           the call also uses it as scratch (each (row, head) slot holds that row's
 *           prepared query before its output), so its contents are unspecified until
 *           the call has completed on the stream.
 *   row_stats NULL or [24][rows][2] float: per (head, row) the final running maximum M
 *           (an integer, base-2 units) and the sum l of the rounded weights relative to
 *           2^M, so that the row's weights are bf16(2^(t - M)) / l with t = s * log2(e).
 * Rules (review §Dispatch/guard of the same page): q_base % 64 == 0, q_base >= 0,
 * q_base + rows <= T <= GA_MAX_TOKENS.
 * Errors: NULL, SHAPE, RANGE, TABLE, ALIGN (qg, k_prep, v, out, w_q, tables, row_stats),
 * DEVICE, CUDA. */
int ga_attn_prefill(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                    const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                    int table_rows, int rows, int T, int q_base, int causal, ga_bf16* out,
                    float* row_stats, ga_stream stream);

/* ga_attn_prefill for one group of KV heads: the query heads 12 * kv_first ..
 * 12 * (kv_first + kv_count) - 1 (each KV head with the 12 query heads that read it) and
 * nothing else. This is how the pass shards over GPUs with no exchange between them: GPU g
 * takes KV head g, reads only that head's keys and values and its query heads' halves of the
 * fused rows, and writes only their output columns h * 256 .. h * 256 + 255; the other
 * columns of out (and of row_stats) are left as they were. The results are the bits of
 * ga_attn_prefill in those columns.
 *   kv_first, kv_count: 0 <= kv_first, 1 <= kv_count, kv_first + kv_count <= 2
 *   every other argument as in ga_attn_prefill (out doubles as scratch only in the columns
 *   of the heads processed)
 * Errors: as ga_attn_prefill (RANGE also for the KV-head group). */
int ga_attn_prefill_kv(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                       const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                       int table_rows, int rows, int T, int q_base, int causal, int kv_first,
                       int kv_count, ga_bf16* out, float* row_stats, ga_stream stream);

/* ga_attn_prefill from prepared queries (ga_q_prologue's output): the attention kernel
 * alone. qg still supplies the gates (its last 256 values per head).
 *   q_prep  [rows][24][256]  prepared queries; may be the same buffer as out (each
 *                            (row, head) slot is read before its output is written there)
 *   qg, k_prep, v, rows, T, q_base, causal, out, row_stats: as in ga_attn_prefill
 * Errors: NULL, SHAPE, RANGE, ALIGN (q_prep, qg, k_prep, v, out, row_stats), DEVICE, CUDA. */
int ga_attn_prefill_prepared(const ga_bf16* q_prep, const ga_bf16* qg, const ga_bf16* k_prep,
                             const ga_bf16* v, int rows, int T, int q_base, int causal,
                             ga_bf16* out, float* row_stats, ga_stream stream);

/* Bytes of workspace ga_attn_masked needs for (rows, T); 0 for invalid sizes. */
size_t ga_masked_workspace_bytes(int rows, int T);

/* Stored-mask gated GQA attention (pegainfer PR #1151, §Semantics: the kernel consumes
 * the selection mask as given, non-zero = visible; it is not ANDed with causality here).
 *   qg, k_prep, v, w_q, cos_tab, sin_tab, table_rows, q_base: as in ga_attn_prefill
 *   mask    [rows][ld_mask] uint8; row r is query position q_base + r, column j key j
 *   out     [rows][24 * 256] (scratch during the call, as in ga_attn_prefill)
 *   weights NULL or [24][rows][T] bf16: the normalised weights bf16(w_hat / L), exactly
 *           0 where a key is hidden
 *   hidden_rows NULL or one device int; receives the number of rows with no visible key
 *           (their outputs and weights are 0; the page leaves such rows outside its
 *           contract)
 *   workspace >= ga_masked_workspace_bytes(rows, T) bytes of device memory, 256-byte
 *           aligned, owned by the caller, not shared with a concurrent call
 * Rules: T <= GA_MASKED_MAX_TOKENS, ld_mask >= T, ld_mask % 16 == 0, q_base % 64 == 0,
 * q_base + rows <= T.
 * Errors: NULL, SHAPE, RANGE, TABLE, ALIGN (mask also), WORKSPACE, DEVICE, CUDA. */
int ga_attn_masked(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                   const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                   int table_rows, int rows, int T, int q_base, const uint8_t* mask,
                   long long ld_mask, ga_bf16* out, ga_bf16* weights, int* hidden_rows,
                   void* workspace, size_t ws_bytes, ga_stream stream);

/* ga_attn_masked for one group of KV heads (see ga_attn_prefill_kv): the query heads
 * 12 * kv_first .. 12 * (kv_first + kv_count) - 1 only. Their output columns (and, when
 * weights is given, their [12 * kv_count][rows][T] slice of weights, zeroed first) are
 * written; everything else is left as it was. hidden_rows counts each hidden row once.
 *   kv_first, kv_count: 0 <= kv_first, 1 <= kv_count, kv_first + kv_count <= 2
 *   every other argument as in ga_attn_masked
 * Errors: as ga_attn_masked (RANGE also for the KV-head group). */
int ga_attn_masked_kv(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                      const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                      int table_rows, int rows, int T, int q_base, const uint8_t* mask,
                      long long ld_mask, int kv_first, int kv_count, ga_bf16* out,
                      ga_bf16* weights, int* hidden_rows, void* workspace, size_t ws_bytes,
                      ga_stream stream);

/* ga_attn_masked from prepared queries (ga_q_prologue's output): the mask prepass and the
 * attention kernel (and the weights pass) without the query prologue, exposed so that a
 * caller can time or reuse the prepared queries, as ga_attn_prefill_prepared does for the
 * causal pass.
 *   q_prep  [rows][24][256]  prepared queries of positions q_base .. q_base+rows-1, 16-byte
 *                            aligned; may not overlap out
 *   qg, k_prep, v, rows, T, q_base, mask, ld_mask, out, weights, hidden_rows, workspace,
 *           ws_bytes: as in ga_attn_masked (the workspace's query area is not used)
 * Rules and errors: as ga_attn_masked (NULL also for q_prep), without the table checks. */
int ga_attn_masked_prepared(const ga_bf16* q_prep, const ga_bf16* qg, const ga_bf16* k_prep,
                            const ga_bf16* v, int rows, int T, int q_base, const uint8_t* mask,
                            long long ld_mask, ga_bf16* out, ga_bf16* weights,
                            int* hidden_rows, void* workspace, size_t ws_bytes,
                            ga_stream stream);

/* Allocation-free variant of ga_attn_masked. The pages have no counterpart: this is an
 * addition of the library for callers that may not allocate device memory at call time,
 * such as a server step that runs under a fixed memory budget, or a framework that
 * forbids allocation inside a step (an allocation can synchronise the device, and can
 * fail when memory is fragmented). The scratch that ga_attn_masked takes as `workspace`
 * comes instead from one static device array of GA_STATIC_SCRATCH_BYTES per device,
 * reserved when the library is loaded; nothing is allocated by the call.
 *   Arguments, layouts and results: as in ga_attn_masked, without workspace/ws_bytes.
 *   Limit: the call runs when ga_masked_workspace_bytes(rows, T) <=
 *           GA_STATIC_SCRATCH_BYTES: up to 1,239 rows at T = 8192, 1,286 at T = 4096,
 *           1,315 at T = 2048. Larger calls are refused with GA_ERR_WORKSPACE before any
 *           CUDA call.
 *   The first call on a device looks up the array's address (one CUDA runtime query,
 *           once per device, with that device current); make a first call before any
 *           stream capture. The address is kept per device index for the life of the
 *           process: the library assumes each device's primary context (the runtime's
 *           default) and no cudaDeviceReset between calls, the same assumption as its
 *           other per-device set-up.
 *   The scratch needs no initial contents (every call writes all of it that it reads).
 *   The array is shared by all calls on a device: calls that may overlap in time (other
 *           streams, other host threads) race on it and must be serialised by the caller.
 * Errors: as ga_attn_masked. */
#define GA_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
int ga_attn_masked_static(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                          const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                          int table_rows, int rows, int T, int q_base, const uint8_t* mask,
                          long long ld_mask, ga_bf16* out, ga_bf16* weights, int* hidden_rows,
                          ga_stream stream);

/* The widened rows of e4m3 cache rows: out = bf16(fp32(code * scale)) per element, the
 * values ga_attn_verify_e4m3 attends over (TensorFold PR #1080: e4m3 cache rows with an
 * fp32 scale each, widened to bf16).
 *   q      [n_tok][2][256] uint8 e4m3 codes, as ga_kv_quantize_e4m3 writes them, 8-byte aligned
 *   scale  [n_tok][2] fp32, 4-byte aligned
 *   out    [n_tok][2][256] bf16, 16-byte aligned
 * Rules: 0 <= n_tok <= 64 * GA_MAX_TOKENS; n_tok == 0 is a no-op.
 * Errors: NULL, SHAPE, RANGE, ALIGN, DEVICE, CUDA. */
int ga_kv_dequantize_e4m3(const uint8_t* q, const float* scale, long long n_tok, ga_bf16* out,
                          ga_stream stream);

/* Bytes of workspace ga_attn_prefill_e4m3 needs for T keys (the widened K and V); 0 for
 * T outside 1 .. GA_MAX_TOKENS. */
size_t ga_prefill_e4m3_workspace_bytes(int T);

/* ga_attn_prefill over e4m3 caches of prepared keys and values (TensorFold PR #1080: e4m3
 * cache rows with an fp32 scale each, read by the prompt chain). Prefill reads every key
 * tile once per 128-row tile of queries, so the rows are widened once, into the workspace,
 * by ga_kv_dequantize_e4m3's kernel, and the bf16 pass then runs over them: the results
 * are the bits of ga_attn_prefill over the widened rows.
 *   k_codes, v_codes [T][2][256] uint8, 16-byte aligned; k_scale, v_scale [T][2] fp32
 *   qg, w_q, cos_tab, sin_tab, table_rows, rows, T, q_base, causal, out, row_stats: as in
 *           ga_attn_prefill
 *   workspace >= ga_prefill_e4m3_workspace_bytes(T) bytes, 256-byte aligned, owned by the
 *           caller and not shared with a concurrent call; it holds the widened K then V
 * Errors: NULL, SHAPE, RANGE, TABLE, ALIGN, WORKSPACE, DEVICE, CUDA. */
int ga_attn_prefill_e4m3(const ga_bf16* qg, const uint8_t* k_codes, const float* k_scale,
                         const uint8_t* v_codes, const float* v_scale, const ga_bf16* w_q,
                         const ga_bf16* cos_tab, const ga_bf16* sin_tab, int table_rows,
                         int rows, int T, int q_base, int causal, ga_bf16* out,
                         float* row_stats, void* workspace, size_t ws_bytes, ga_stream stream);

/* The selection mask ga_attn_masked reads, from the indexer's per-block scores (pegainfer
 * PR #1151, "feat(qwen4): add the QSA sparse-attention kernel and its golden": the mask is
 * the indexer's selection AND causality; a budget of 2048 tokens keeps 512 blocks of 4 keys,
 * a budget of 16 keeps 4). The scores themselves come from the indexer, which the pages
 * do not specify; this call does the selection and writes the mask.
 *   block_scores [rows][ld_scores] fp32, 4-byte aligned: row r scores block b (keys
 *           4b .. 4b+3) at r * ld_scores + b for b < ceil(T / 4). Scores may be +-inf
 *           and -0 equals +0; a NaN score gives an unspecified selection for its row.
 *   rows, T, q_base: row r is query position p = q_base + r; the keys are 0 .. T-1
 *   block_topk  blocks kept per row (budget / GA_INDEX_BLOCK_TOKENS)
 *   mask    [rows][ld_mask] uint8, written for columns 0 .. T-1 (later columns untouched):
 *           1 iff j <= p and block j / 4 is among the row's block_topk highest-scoring
 *           candidates (the blocks b <= p / 4), a tie going to the lower block index;
 *           every candidate when there are fewer. A row always sees at least one key.
 * Rules: T <= GA_MASKED_MAX_TOKENS, q_base + rows <= T, ld_scores >= ceil(T / 4),
 * ld_mask >= T, ld_mask % 16 == 0, mask 16-byte aligned, both leading dimensions <= 2^31.
 * Nothing is allocated; the call keeps no pointer. rows == 0 is a no-op.
 * Errors: NULL, SHAPE, RANGE, ALIGN, DEVICE, CUDA. */
int ga_select_mask(const float* block_scores, long long ld_scores, int rows, int T, int q_base,
                   int block_topk, uint8_t* mask, long long ld_mask, ga_stream stream);

/* Bytes of workspace ga_attn_verify needs; max_len is the largest L over the sequences. */
size_t ga_verify_workspace_bytes(int n_seq, int rows, int max_len);

/* Few-row verify windows over long caches, split over key chunks with a log-sum-exp
 * combine (TensorFold PR #1080, "qwen CUDA: long-prompt prefill 5.4x faster", the
 * attn_partial commit: keys split into chunks, partial rows combined afterwards).
 *   qg       [n_seq][rows][24][512] fused rows; sequence b's row r is position L_b + r
 *   k_cache  [n_seq][cap][2][256] PREPARED keys of positions 0 .. L_b+rows-1 (the
 *            window's own keys included; fill with ga_k_prologue)
 *   v_cache  [n_seq][cap][2][256] values
 *   seq_len  HOST array of n_seq ints: L_b, with L_b >= 0 and L_b + rows <= cap
 *   out      [n_seq][rows][24 * 256] (scratch during the call, as in ga_attn_prefill)
 *   workspace >= ga_verify_workspace_bytes(n_seq, rows, max L_b), 256-byte aligned
 * Row r of sequence b sees keys 0 .. L_b + r. Cache positions from L_b + rows up to the
 * end of the 128-key tile that holds position L_b + rows - 1 are read and hidden, so they
 * must hold finite values (a hidden value still meets the tensor cores with weight 0).
 * Rules: 1 <= rows <= 16, cap <= GA_MAX_TOKENS, table_rows >= max L_b + rows.
 * Errors: NULL, SHAPE, RANGE, TABLE, ALIGN, WORKSPACE, DEVICE, CUDA. */
int ga_attn_verify(const ga_bf16* qg, const ga_bf16* k_cache, const ga_bf16* v_cache,
                   int cap, const int* seq_len, int n_seq, int rows, const ga_bf16* w_q,
                   const ga_bf16* cos_tab, const ga_bf16* sin_tab, int table_rows,
                   ga_bf16* out, void* workspace, size_t ws_bytes, ga_stream stream);

/* ga_attn_verify over e4m3 caches (TensorFold PR #1080, "qwen CUDA: long-prompt prefill 5.4x
 * faster": e4m3 cache rows with an fp32 scale each, staged a step ahead and widened to bf16
 * in the shared-memory slot). The caches hold what ga_kv_quantize_e4m3 writes:
 *   k_codes, v_codes  [n_seq][cap][2][256] uint8 e4m3 codes, 16-byte aligned
 *   k_scale, v_scale  [n_seq][cap][2] fp32 row scales, 4-byte aligned
 * Each row is widened to bf16(fp32(code * scale)) and the call then computes exactly what
 * ga_attn_verify computes over those bf16 rows: the same bits. It reads half the cache bytes.
 * Positions read but hidden (past L_b + rows inside the last 128-key tile, below cap) must
 * hold codes other than NaN (0x7F, 0xFF) and finite scales. Everything else, the rules and
 * the errors are those of ga_attn_verify, with the same workspace size. */
int ga_attn_verify_e4m3(const ga_bf16* qg, const uint8_t* k_codes, const float* k_scale,
                        const uint8_t* v_codes, const float* v_scale, int cap, const int* seq_len,
                        int n_seq, int rows, const ga_bf16* w_q, const ga_bf16* cos_tab,
                        const ga_bf16* sin_tab, int table_rows, ga_bf16* out, void* workspace,
                        size_t ws_bytes, ga_stream stream);

/* ga_attn_verify over PAGED caches, and decode (rows = 1). pegainfer PR #1151, "feat(qwen4):
 * add the QSA sparse-attention kernel and its golden", §Summary and §Limits name paged KV
 * and decode as the next steps after its contiguous key array; the layout is the plain
 * reading of a page table. Each sequence's positions live in fixed-size pages of two pools:
 *   k_pages   [n_pages][page_size][2][256] PREPARED keys (as ga_k_prologue writes them)
 *   v_pages   [n_pages][page_size][2][256] values
 *   page_table DEVICE int32 [n_seq][max_pages]: position t of sequence b lives on page
 *             page_table[b * max_pages + t / page_size], slot t % page_size. Only the
 *             entries that cover positions 0 .. L_b + rows - 1 are read; each must lie in
 *             [0, n_pages). An entry outside that range is not a fault: the kernel records
 *             status 3 in the device status word (ga_device_status) and reads zeros for
 *             that tile, so the call's outputs are then meaningless.
 *   page_size a multiple of 128 (one or more 128-key tiles per page)
 * Everything else (qg, seq_len on the HOST, rows, the tables, out, the workspace from
 * ga_verify_workspace_bytes, the finite-values rule for hidden positions) is as in
 * ga_attn_verify, and so are the results: the same sequence gives the same bits whether
 * its caches are contiguous or paged. Pages may be shared between sequences (a common
 * prefix) and need not be in any order. Nothing is allocated; the call keeps no pointer.
 * Rules: 1 <= rows <= 16, L_b + rows <= max_pages * page_size and <= GA_MAX_TOKENS,
 * table_rows >= max L_b + rows, page_table 4-byte aligned.
 * Errors: NULL, SHAPE, RANGE, TABLE, ALIGN, WORKSPACE, DEVICE, CUDA. */
int ga_attn_verify_paged(const ga_bf16* qg, const ga_bf16* k_pages, const ga_bf16* v_pages,
                         int n_pages, int page_size, const int* page_table, int max_pages,
                         const int* seq_len, int n_seq, int rows, const ga_bf16* w_q,
                         const ga_bf16* cos_tab, const ga_bf16* sin_tab, int table_rows,
                         ga_bf16* out, void* workspace, size_t ws_bytes, ga_stream stream);

/* e4m3 cache rows with one fp32 scale each (TensorFold PR #1080, "qwen CUDA: long-prompt
 * prefill 5.4x faster": its prompt chain reads e4m3 cache rows with an fp32 scale each and
 * widens them to bf16 in the shared-memory slot; its rope kernels compute the e4m3 scales by
 * reductions over the row). For every (token, head) row of 256 bf16 values x:
 *   scale = fp32(max|x| / 448),  q = e4m3(fp32(x / scale))
 * with IEEE divisions rounded to nearest and the OCP FP8 E4M3 conversion rounding to nearest
 * (ties to even) and saturating at +-448; a row of zeros gives scale 0 and q 0. The widened
 * row that ga_attn_verify_e4m3 attends over is bf16(fp32(q * scale)).
 *   x      [n_tok][2][256] bf16: prepared keys (as ga_k_prologue writes them) or values
 *   q      [n_tok][2][256] uint8 e4m3 codes (byte d of a row is dim d)
 *   scale  [n_tok][2] fp32
 * Rules: x 8-byte aligned, q 4-byte aligned, scale 4-byte aligned, 0 <= n_tok <= GA_MAX_TOKENS
 * x 64 (sequences laid end to end count as one long run). n_tok = 0 is a no-op.
 * Errors: NULL, SHAPE, RANGE, ALIGN, DEVICE, CUDA. */
int ga_kv_quantize_e4m3(const ga_bf16* x, long long n_tok, uint8_t* q, float* scale,
                        ga_stream stream);

/* Several causal prefills in one call: sequences (or branches) of different lengths, each a
 * window of rows at its own q_base over its own paged cache. system1-omni PR #99, "run
 * prompts that share prefixes once per prefix", and PR #196, "perf(open-jev): optimize 9B
 * prefill while preserving native outputs" (its batched gated-attention entry points,
 * checked bit for bit against the one-sequence path): prompts that share a prefix run the
 * prefix once and continue each branch from it. Here a branch is a sequence whose page-table
 * row lists the prefix's pages (whole pages, shared) and then its own; its rows are its
 * positions after the prefix (q_base = the prefix length).
 *   qg          [total_rows][24][512] fused rows of all sequences, packed: sequence b's row r
 *               is packed row row_start[b] + r, at position q_base[b] + r
 *   row_start   HOST int[n_seq + 1], ascending, row_start[0] >= 0; sequence b has
 *               row_start[b + 1] - row_start[b] >= 0 rows
 *   q_base      HOST int[n_seq], multiples of 64
 *   k_pages, v_pages, n_pages, page_size, page_table, max_pages: as in ga_attn_verify_paged;
 *               sequence b's keys 0 .. q_base[b] + rows_b - 1 are read through page-table
 *               row b (they must be prepared and present, the window's own keys included)
 *   out         [total_rows][24 * 256] (scratch during the call, as in ga_attn_prefill)
 * Row r of sequence b sees keys 0 .. q_base[b] + r. Every sequence's rows come out with the
 * same bits as ga_attn_prefill gives for them over the same keys (causal, window q_base[b],
 * T = q_base[b] + rows_b). The kernels handle up to 64 sequences and 256 row tiles of 128
 * rows per launch and the call launches as many times as needed; nothing is allocated and
 * no pointer is kept. Hidden positions read inside a window's last key tile must be finite.
 * Rules: page_size a multiple of 128, q_base[b] + rows_b <= max_pages * page_size and
 * <= GA_MAX_TOKENS, row_start[n_seq] <= GA_MAX_TOKENS, table_rows >= max q_base[b] + rows_b,
 * page_table 4-byte aligned. A call with no rows returns GA_OK without a CUDA call.
 * Errors: NULL, SHAPE, RANGE, TABLE, ALIGN, DEVICE, CUDA. */
int ga_attn_prefill_batch(const ga_bf16* qg, const int* row_start, const int* q_base, int n_seq,
                          const ga_bf16* k_pages, const ga_bf16* v_pages, int n_pages,
                          int page_size, const int* page_table, int max_pages,
                          const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                          int table_rows, ga_bf16* out, ga_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* GA_ATTN_H */
