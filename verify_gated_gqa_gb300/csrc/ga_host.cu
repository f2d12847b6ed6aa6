// Host side of libga_attn.so: argument validation (before any CUDA call), per-device
// set-up, TMA descriptor encoding, launches, status codes.
#include <atomic>
#include <cmath>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <vector>

#include "ga_internal.h"

namespace ga {
namespace {

std::atomic<unsigned long long> g_cuda_calls{0};
thread_local int t_last_cuda_error = 0;

// Every CUDA runtime or driver call of the library goes through here (so that tests can
// prove a refused call made none).
template <typename T>
inline T counted(T r) {
  return r;
}
#define GA_CUDA(expr) (g_cuda_calls.fetch_add(1, std::memory_order_relaxed), counted(expr))

__device__ int g_device_status;  // written by kernels whose bounded waits gave up

constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready = false;
  int status = GA_OK;  // GA_OK or GA_ERR_DEVICE / GA_ERR_CUDA from set-up
  int sm_count = 0;
  int pair_clusters = 0;  // clusters of two attention CTAs that fit at once (e4m3 verify)
  int gated_pair_clusters = 0;  // the same for the CTA-pair gated passes
  int* status_word = nullptr;
};
DeviceState g_devices[kMaxDevices];
std::mutex g_device_mutex;

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return GA_ERR_CUDA;
}

uint16_t bf16_rne(double x);

// bf16(1 / (1 + e^-g)) for every bf16 g, indexed by g's bits, from the definition in double
// (pegainfer PR #1151, §Semantics: the gate's sigmoid is rounded to bf16 before the final
// product). NaN gates give a quiet NaN.
const uint16_t* sigmoid_table() {
  static uint16_t table[1 << 16];
  static std::once_flag once;
  std::call_once(once, [] {
    for (uint32_t b = 0; b < (1u << 16); ++b) {
      const uint32_t bits = b << 16;
      float g;
      std::memcpy(&g, &bits, 4);
      if (std::isnan(g)) {
        table[b] = 0x7FC0u;
        continue;
      }
      table[b] = bf16_rne(1.0 / (1.0 + std::exp(-(double)g)));
    }
  });
  return table;
}

// Capability check, shared-memory opt-in, sigmoid table and status-word address, once
// per device
// (system1-omni PR #202, "cuda: widen the attention query tile on sm_89 and sm_120",
// second review and the author's fix: the decision and the opt-in are kept per device).
int current_device(DeviceState** out) {
  int dev = 0;
  cudaError_t e = GA_CUDA(cudaGetDevice(&dev));
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return GA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_device_mutex);
  DeviceState& d = g_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = GA_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev))) != cudaSuccess ||
        (e = GA_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev))) != cudaSuccess ||
        (e = GA_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) != cudaSuccess)
      return fail_cuda(e);
    if (major != 10 || minor != 3) {
      d.ready = true;
      d.status = GA_ERR_DEVICE;
    } else {
      void* sw = nullptr;
      if ((e = GA_CUDA(attn_set_smem_attribute())) != cudaSuccess) return fail_cuda(e);
      if ((e = GA_CUDA(probe_set_smem_attribute())) != cudaSuccess) return fail_cuda(e);
      if ((e = GA_CUDA(attn_max_pair_clusters(&d.pair_clusters))) != cudaSuccess) return fail_cuda(e);
      if ((e = GA_CUDA(attn_max_gated_pair_clusters(&d.gated_pair_clusters))) != cudaSuccess)
        return fail_cuda(e);
      if (d.pair_clusters < 1 || d.gated_pair_clusters < 1) {
        d.ready = true;
        d.status = GA_ERR_DEVICE;
        *out = &d;
        return d.status;
      }
      if ((e = GA_CUDA(attn_upload_sigmoid_table(sigmoid_table()))) != cudaSuccess)
        return fail_cuda(e);
      if ((e = GA_CUDA(cudaGetSymbolAddress(&sw, g_device_status))) != cudaSuccess) return fail_cuda(e);
      d.status_word = static_cast<int*>(sw);
      d.sm_count = sms;
      d.status = GA_OK;
      d.ready = true;
    }
  }
  *out = &d;
  return d.status;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

int get_encode(EncodeTiledFn* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (GA_CUDA(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                 cudaEnableDefault, &q)) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(p);
  });
  *fn = g_encode;
  return g_encode ? GA_OK : GA_ERR_DEVICE;
}

// [n_outer][n_tok][2][256] bf16 keys or values as a TMA tensor: box = 64 dims x box_tok
// tokens x 1 head x box_blocks blocks of 64 dims (a whole tile: 128 x 4; a CTA pair's
// halves: 64 x 4 for K, 128 x 2 for V), 128-byte swizzle; tokens past the end read as zeros.
// With seq_dim the sequence is the fifth coordinate (verify caches, n_outer >= 1 sequences);
// without it the map has four dimensions (n_outer must be 1).
int encode_kv_map(CUtensorMap* map, const void* base, long long n_tok, long long n_outer,
                  bool seq_dim, int box_tok = kTileN, int box_blocks = kDim / 64) {
  EncodeTiledFn enc;
  int st = get_encode(&enc);
  if (st != GA_OK) return st;
  // dims (64 dims of a block, token, head, block of 64 dims[, sequence]): the block index
  // is listed after the token so one box of 64 x 128 x 1 x 4 lands as four consecutive
  // [128 keys][64 dims] blocks, the layout the tensor cores read
  cuuint64_t dims[5] = {64, (cuuint64_t)n_tok, (cuuint64_t)kKvHeads, (cuuint64_t)(kDim / 64),
                        (cuuint64_t)n_outer};
  cuuint64_t strides[4] = {(cuuint64_t)kKvHeads * kDim * 2, (cuuint64_t)kDim * 2, 64 * 2,
                           (cuuint64_t)n_tok * kKvHeads * kDim * 2};
  cuuint32_t box[5] = {64, (cuuint32_t)box_tok, 1, (cuuint32_t)box_blocks, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  const cuuint32_t rank = seq_dim ? 5 : 4;
  CUresult r = GA_CUDA(enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base),
                           dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = (int)r;
    return GA_ERR_CUDA;
  }
  return GA_OK;
}

// [rows][24][256] bf16 prepared queries as a TMA tensor: box = 64 dims x box_heads heads x
// box_rows rows (1 x 128 for the prefill row tiles, 6 x rows for a verify tile), 128-byte
// swizzle; rows past the end read as zeros.
int encode_q_map(CUtensorMap* map, const void* base, long long rows, int box_heads = 1,
                 int box_rows = kTileM) {
  EncodeTiledFn enc;
  int st = get_encode(&enc);
  if (st != GA_OK) return st;
  cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)kHeads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kDim * 2, (cuuint64_t)kOutRow * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = GA_CUDA(enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                           strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = (int)r;
    return GA_ERR_CUDA;
  }
  return GA_OK;
}

// [n_seq][cap][2][256] e4m3 key or value rows as a TMA tensor: box = one head's 256 codes x
// 8 tokens of one sequence (an eighth of one CTA's 64 keys of a 128-key tile), unswizzled
// (the edge warps widen it to the swizzled bf16 tile); tokens past the cache read as zeros.
int encode_kv8_map(CUtensorMap* map, const void* base, long long cap, long long n_seq) {
  EncodeTiledFn enc;
  int st = get_encode(&enc);
  if (st != GA_OK) return st;
  cuuint64_t dims[4] = {(cuuint64_t)kDim, (cuuint64_t)kKvHeads, (cuuint64_t)cap, (cuuint64_t)n_seq};
  cuuint64_t strides[3] = {(cuuint64_t)kDim, (cuuint64_t)kKvHeads * kDim,
                           (cuuint64_t)cap * kKvHeads * kDim};
  cuuint32_t box[4] = {(cuuint32_t)kDim, 1, 8, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = GA_CUDA(enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims,
                           strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = (int)r;
    return GA_ERR_CUDA;
  }
  return GA_OK;
}

// [rows][24][512] bf16 fused q|gate rows as a TMA tensor, read for the gate halves: box =
// 64 values x 1 head x 128 rows at x = 256 + 64c, 128-byte swizzle; rows past the end read
// as zeros.
int encode_gate_map(CUtensorMap* map, const void* base, long long rows) {
  EncodeTiledFn enc;
  int st = get_encode(&enc);
  if (st != GA_OK) return st;
  cuuint64_t dims[3] = {(cuuint64_t)kQgStride, (cuuint64_t)kHeads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kQgStride * 2, (cuuint64_t)kHeads * kQgStride * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kTileM};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = GA_CUDA(enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                           strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = (int)r;
    return GA_ERR_CUDA;
  }
  return GA_OK;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// bf16 (nearest, ties to even) of a double.
uint16_t bf16_rne(double x) {
  if (x == 0.0) return std::signbit(x) ? 0x8000u : 0u;
  int e = 0;
  std::frexp(x, &e);
  if (e < -125) e = -125;
  const double q = std::ldexp(std::nearbyint(std::ldexp(x, 8 - e)), e - 8);
  const float f = (float)q;  // exact: q holds a bf16 value
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

// Shared checks of the attention entry points (no CUDA call).
int check_attention_args(const void* qg, const void* k_prep, const void* v, const void* w_q,
                         const void* cos_tab, const void* sin_tab, int table_rows, int rows,
                         int T, int q_base, const void* out) {
  if (!qg || !k_prep || !v || !w_q || !cos_tab || !sin_tab || !out) return GA_ERR_NULL;
  if (rows < 0 || T < 1 || table_rows < 0) return GA_ERR_SHAPE;
  if (T > GA_MAX_TOKENS || q_base < 0 || q_base % 64 != 0 || (long long)q_base + rows > T)
    return GA_ERR_RANGE;
  if ((long long)table_rows < (long long)q_base + rows) return GA_ERR_TABLE;
  if (!aligned(qg, 16) || !aligned(k_prep, 16) || !aligned(v, 16) || !aligned(w_q, 16) ||
      !aligned(cos_tab, 16) || !aligned(sin_tab, 16) || !aligned(out, 16))
    return GA_ERR_ALIGN;
  return GA_OK;
}

struct MaskedLayout {
  size_t bits_off, flags_off, stats_off, q_off, total;
  int row_tiles, key_tiles, mask_words;
};
MaskedLayout masked_layout(int rows, int T) {
  MaskedLayout L;
  L.row_tiles = (rows + kTileM - 1) / kTileM;
  L.key_tiles = (T + kTileN - 1) / kTileN;
  L.mask_words = L.key_tiles * (kTileN / 32);
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  L.bits_off = 0;
  L.flags_off = up(L.bits_off + (size_t)L.row_tiles * kTileM * L.mask_words * 4);
  L.stats_off = up(L.flags_off + (size_t)L.row_tiles * kMaskFlagStride);
  L.q_off = up(L.stats_off + (size_t)kHeads * rows * 2 * sizeof(float));
  L.total = up(L.q_off + (size_t)rows * kOutRow * sizeof(uint16_t));
  return L;
}

// Verify split: sequences in groups of up to kVerifyMaxSeq per launch; per group, the keys
// of each sequence in n_chunks chunks of chunk_tiles 128-key tiles, with about two work
// items (chunk x sequence x KV head x half group) per SM. The workspace holds one group's
// partials; its size does not depend on the device (at most kVerifyChunkCap / n_seq chunks).
struct VerifyPlan {
  int n_seq_group, n_tiles_max, n_chunks_cap;
};
VerifyPlan verify_plan(int n_seq, int rows, int max_len) {
  VerifyPlan p;
  p.n_seq_group = n_seq < kVerifyMaxSeq ? n_seq : kVerifyMaxSeq;
  p.n_tiles_max = (max_len + rows + kTileN - 1) / kTileN;
  const int by_items = kVerifyChunkCap / (4 * (p.n_seq_group > 0 ? p.n_seq_group : 1));
  p.n_chunks_cap = by_items < 1 ? 1 : by_items;
  if (p.n_chunks_cap > p.n_tiles_max) p.n_chunks_cap = p.n_tiles_max > 0 ? p.n_tiles_max : 1;
  return p;
}
size_t verify_part_o_bytes(const VerifyPlan& p) {
  return (size_t)p.n_seq_group * 4 * p.n_chunks_cap * kVerifyLanes * kDim * sizeof(float);
}
size_t verify_ws_bytes(const VerifyPlan& p) {
  return verify_part_o_bytes(p) +
         (size_t)p.n_seq_group * 4 * p.n_chunks_cap * kVerifyLanes * 2 * sizeof(float);
}

// The query prologue (unless q_ready: q_prep already holds this call's prepared queries)
// and the attention kernel. q_prep [rows][24][256] may be the output buffer itself: each
// (row, head) slot is read by the work item that later writes its output there.
// ga_debug_set_cta_pairs: 0 single CTAs; 1 CTA pairs where they pay (below); 2 CTA pairs
// wherever the heads allow them
std::atomic<int> g_cta_pairs{1};
// Keys below which a single-sequence pass runs on single CTAs under mode 1: measured on one
// box from a flushed L2, causal and bidirectional, the pairs' cluster set-up and staging
// chain cost about 2 us per call up to 1,024 keys (S = 64: 17.1 against 15.0 us; S = 1024
// causal: 31.4 against 29.3 us) and win from 2,048 keys on (53.9 against 55.9 us; at
// 4,096: 135.8 against 144.1 us).
constexpr int kPairMinKeys = 2048;

int launch_attention(const AttnArgs& a0, uint16_t* q_prep, bool q_ready, const void* k_prep,
                     const void* v, long long n_tok, DeviceState* dev, cudaStream_t s) {
  AttnArgs a = a0;
  a.status = dev->status_word;
  if (a.n_heads == 0) {   // every query head unless the caller chose a KV-head group
    a.head0 = 0;
    a.n_heads = kHeads;
  }
  // The causal, bidirectional and stored-mask passes run as CTA pairs (two query heads of
  // one KV group per pair item) whenever the heads come in such pairs and the keys are
  // many enough for the pairs to pay (kPairMinKeys); the weights pass runs on single CTAs.
  const int pair_mode = g_cta_pairs.load();
  const bool pair = (pair_mode == 2 || (pair_mode == 1 && a.T >= kPairMinKeys)) &&
                    !a.weights_pass &&
                    (a.mode == kModeCausal || a.mode == kModeBidir || a.mode == kModeMask) &&
                    a.head0 % 2 == 0 && a.n_heads % 2 == 0;
  a.pair = pair ? 1 : 0;
  CUtensorMap tm_q, tm_k, tm_v, tm_g, tm_o;
  int st = encode_q_map(&tm_q, q_prep, a0.rows);
  if (st != GA_OK) return st;
  st = encode_gate_map(&tm_g, a0.qg, a0.rows);
  if (st != GA_OK) return st;
  st = pair ? encode_q_map(&tm_o, a0.out, a0.rows) : encode_q_map(&tm_o, q_prep, a0.rows);
  if (st != GA_OK) return st;
  st = pair ? encode_kv_map(&tm_k, k_prep, n_tok, 1, false, kTileN / 2, kDim / 64)
            : encode_kv_map(&tm_k, k_prep, n_tok, 1, false);
  if (st != GA_OK) return st;
  st = pair ? encode_kv_map(&tm_v, v, n_tok, 1, false, kTileN, kDim / 128)
            : encode_kv_map(&tm_v, v, n_tok, 1, false);
  if (st != GA_OK) return st;
  a.row_tiles = (a.rows + kTileM - 1) / kTileM;
  a.n_items = a.row_tiles * (pair ? a.n_heads / 2 : a.n_heads);
  cudaError_t e;
  if (!q_ready &&
      (e = GA_CUDA(launch_q_prologue(a.qg, a.w_q, a.cos_tab, a.sin_tab, a.rows, a.q_base, a.head0,
                                     a.n_heads, q_prep, dev->sm_count, s))) != cudaSuccess)
    return fail_cuda(e);
  const int cap = pair ? dev->gated_pair_clusters : dev->sm_count;
  const int grid = (pair ? 2 : 1) * (a.n_items < cap ? a.n_items : cap);
  e = GA_CUDA(launch_attn(tm_q, tm_k, tm_v, tm_g, tm_o, a, grid, s));
  if (e != cudaSuccess) return fail_cuda(e);
  return GA_OK;
}

// The verify call over contiguous caches (one [cap][2][256] cache per sequence) or paged
// caches (page pools and a page table); the callers have checked the arguments that differ.
struct VerifyCaches {
  const ga_bf16* k;
  const ga_bf16* v;
  const uint8_t* k8;        // e4m3 caches (k, v null): [n_seq][cap][2][256] codes
  const uint8_t* v8;
  const float* k_scale;     // and their row scales [n_seq][cap][2]
  const float* v_scale;
  int cap;                  // contiguous: positions per sequence's cache
  const int* page_table;    // paged: [n_seq][max_pages] device array, else null
  int page_size, max_pages, n_pages;
};

int verify_run(const ga_bf16* qg, const VerifyCaches& c, const int* seq_len, int n_seq, int rows,
               const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
               int table_rows, ga_bf16* out, void* workspace, size_t ws_bytes, ga_stream stream) {
  int max_len = 0;
  for (int b = 0; b < n_seq; ++b)
    if (seq_len[b] > max_len) max_len = seq_len[b];
  if ((long long)table_rows < (long long)max_len + rows) return GA_ERR_TABLE;
  const bool fp8 = c.k8 != nullptr;
  if (!aligned(qg, 16) || !aligned(fp8 ? (const void*)c.k8 : c.k, 16) ||
      !aligned(fp8 ? (const void*)c.v8 : c.v, 16) || !aligned(w_q, 16) || !aligned(cos_tab, 16) ||
      !aligned(sin_tab, 16) || !aligned(out, 16))
    return GA_ERR_ALIGN;
  if (fp8 && (!aligned(c.k_scale, 4) || !aligned(c.v_scale, 4))) return GA_ERR_ALIGN;
  if (n_seq == 0 || rows == 0) return GA_OK;
  if (!workspace || !aligned(workspace, 256) ||
      ws_bytes < ga_verify_workspace_bytes(n_seq, rows, max_len))
    return GA_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const VerifyPlan plan = verify_plan(n_seq, rows, max_len);
  const size_t seq_elems = (size_t)c.cap * kKvHeads * kDim;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  for (int g0 = 0; g0 < n_seq; g0 += kVerifyMaxSeq) {
    const int n = n_seq - g0 < kVerifyMaxSeq ? n_seq - g0 : kVerifyMaxSeq;
    AttnArgs a{};
    a.qg = qg + (size_t)g0 * rows * kRowElems;
    a.out = out + (size_t)g0 * rows * kOutRow;
    a.mode = fp8 ? kModeVerify8 : kModeVerify;
    a.n_seq = n;
    a.vrows = rows;
    SeqPositions sp{};
    sp.rows_per_seq = rows;
    int tiles_max = 1;
    for (int b = 0; b < n; ++b) {
      a.seq_len[b] = seq_len[g0 + b];
      sp.seq_base[b] = seq_len[g0 + b];
      const int t = (seq_len[g0 + b] + rows + kTileN - 1) / kTileN;
      if (t > tiles_max) tiles_max = t;
    }
    // The chunk count (at most the workspace's) that minimises the busiest SM's key tiles:
    // ceil(items / SMs) items of chunk_tiles tiles each, ties to fewer chunks (fewer partials).
    int best_nc = 1;
    long long best_cost = -1;
    for (int nc = 1; nc <= plan.n_chunks_cap && nc <= tiles_max; ++nc) {
      const int ct = (tiles_max + nc - 1) / nc;
      const long long items = 4LL * n * ((tiles_max + ct - 1) / ct);
      const long long cost = (items + dev->sm_count - 1) / dev->sm_count * ct;
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best_nc = nc;
      }
    }
    a.chunk_tiles = (tiles_max + best_nc - 1) / best_nc;
    a.n_chunks = (tiles_max + a.chunk_tiles - 1) / a.chunk_tiles;
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_ml = reinterpret_cast<float*>(ws + verify_part_o_bytes(plan));
    a.n_items = a.n_chunks * n * 4;
    a.status = dev->status_word;
    a.rows = n * rows;
    cudaError_t e;
    if ((e = GA_CUDA(launch_q_prologue_seq(a.qg, w_q, cos_tab, sin_tab, n * rows, sp, a.out,
                                           dev->sm_count, s))) !=
        cudaSuccess)
      return fail_cuda(e);
    CUtensorMap tm_q, tm_k, tm_v;
    st = encode_q_map(&tm_q, a.out, (long long)n * rows, kVerifyHeadsPerTile, rows);
    if (st != GA_OK) return st;
    if (fp8) {
      const size_t seq_codes = (size_t)c.cap * kKvHeads * kDim;
      st = encode_kv8_map(&tm_k, c.k8 + (size_t)g0 * seq_codes, c.cap, n);
      if (st != GA_OK) return st;
      st = encode_kv8_map(&tm_v, c.v8 + (size_t)g0 * seq_codes, c.cap, n);
      if (st != GA_OK) return st;
      a.k_scale = c.k_scale + (size_t)g0 * c.cap * kKvHeads;
      a.v_scale = c.v_scale + (size_t)g0 * c.cap * kKvHeads;
      a.cache_cap = c.cap;
    } else if (c.page_table) {
      // the whole pools, the page as the outer coordinate
      st = encode_kv_map(&tm_k, c.k, c.page_size, c.n_pages, true);
      if (st != GA_OK) return st;
      st = encode_kv_map(&tm_v, c.v, c.page_size, c.n_pages, true);
      if (st != GA_OK) return st;
      a.page_table = c.page_table + (size_t)g0 * c.max_pages;
      a.page_tiles = c.page_size / kTileN;
      a.max_pages = c.max_pages;
      a.n_pages = c.n_pages;
    } else {
      st = encode_kv_map(&tm_k, c.k + (size_t)g0 * seq_elems, c.cap, n, true);
      if (st != GA_OK) return st;
      st = encode_kv_map(&tm_v, c.v + (size_t)g0 * seq_elems, c.cap, n, true);
      if (st != GA_OK) return st;
    }
    int grid = a.n_items < dev->sm_count ? a.n_items : dev->sm_count;
    if (fp8) {   // clusters of two CTAs (the two halves of a query group), as many as fit
      const int pairs = a.n_items / 2;
      grid = 2 * (pairs < dev->pair_clusters ? pairs : dev->pair_clusters);
    }
    // the verify partials have no gated epilogue: tm_q stands in for the unused gate map
    if ((e = GA_CUDA(launch_attn(tm_q, tm_k, tm_v, tm_q, tm_q, a, grid, s))) != cudaSuccess)
      return fail_cuda(e);
    if ((e = GA_CUDA(launch_verify_combine(a, dev->sm_count, s))) != cudaSuccess) return fail_cuda(e);
  }
  return GA_OK;
}

// Several causal prefills (each a window of rows at its own q_base over its own paged
// cache) in as few launches as the per-launch tables allow. A sequence of more than
// kBatchMaxEntries row tiles is cut into windows of that many tiles, each a piece of its own.
struct BatchPiece {
  int seq, row0, rows, qbase;
};

int batch_run(const ga_bf16* qg, const BatchPiece* pieces, int n_pieces, const ga_bf16* k_pages,
              const ga_bf16* v_pages, int n_pages, int page_size, const int* page_table,
              int max_pages, const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
              ga_bf16* out, ga_stream stream) {
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  // CTA pairs (two query heads of a KV group per pair item, each CTA holding half of every
  // K and V tile: maps of half boxes) unless switched off: a batch of prompts walks enough
  // key tiles for them in every size measured (16 prompts of 512 to 4,096 tokens: 1.09
  // against 1.29 ms)
  const bool pair = g_cta_pairs.load() > 0;
  CUtensorMap tm_k, tm_v;
  st = pair ? encode_kv_map(&tm_k, k_pages, page_size, n_pages, true, kTileN / 2, kDim / 64)
            : encode_kv_map(&tm_k, k_pages, page_size, n_pages, true);
  if (st != GA_OK) return st;
  st = pair ? encode_kv_map(&tm_v, v_pages, page_size, n_pages, true, kTileN, kDim / 128)
            : encode_kv_map(&tm_v, v_pages, page_size, n_pages, true);
  if (st != GA_OK) return st;
  int p0 = 0;
  while (p0 < n_pieces) {
    // the next group: consecutive pieces, at most kVerifyMaxSeq of them and kBatchMaxEntries
    // row tiles in all (every piece has at most kBatchMaxEntries tiles)
    int p1 = p0, entries = 0;
    while (p1 < n_pieces && p1 - p0 < kVerifyMaxSeq) {
      const int t = (pieces[p1].rows + kTileM - 1) / kTileM;
      if (entries + t > kBatchMaxEntries) break;
      entries += t;
      ++p1;
    }
    AttnArgs a{};
    const int grp_row0 = pieces[p0].row0;
    const int grp_rows = pieces[p1 - 1].row0 + pieces[p1 - 1].rows - grp_row0;
    a.qg = qg + (size_t)grp_row0 * kRowElems;
    a.out = out + (size_t)grp_row0 * kOutRow;
    a.mode = kModeBatch;
    a.rows = grp_rows;
    a.n_seq = p1 - p0;
    a.page_table = page_table;
    a.page_tiles = page_size / kTileN;
    a.max_pages = max_pages;
    a.n_pages = n_pages;
    a.status = dev->status_word;
    SeqPositions sp{};
    sp.n_seq = p1 - p0;
    std::vector<std::pair<int, uint32_t>> order;   // (key tiles, entry)
    for (int p = p0; p < p1; ++p) {
      const int i = p - p0;
      a.batch_seq[i] = pieces[p].seq;
      a.batch_row0[i] = pieces[p].row0 - grp_row0;
      a.batch_rows[i] = pieces[p].rows;
      a.batch_qbase[i] = pieces[p].qbase;
      sp.row_start[i] = pieces[p].row0 - grp_row0;
      sp.seq_base[i] = pieces[p].qbase;
      const int tiles = (pieces[p].rows + kTileM - 1) / kTileM;
      for (int mt = 0; mt < tiles; ++mt) {
        const int last_row = std::min(pieces[p].rows, (mt + 1) * kTileM) - 1;
        const int n = (pieces[p].qbase + last_row + 1 + kTileN - 1) / kTileN;
        order.push_back({n, ((uint32_t)i << 16) | (uint32_t)mt});
      }
    }
    sp.row_start[p1 - p0] = grp_rows;
    // the tiles with the most keys first, so each CTA's share of the work evens out
    std::stable_sort(order.begin(), order.end(),
                     [](const std::pair<int, uint32_t>& x, const std::pair<int, uint32_t>& y) {
                       return x.first > y.first;
                     });
    a.n_entries = (int)order.size();
    for (int i = 0; i < a.n_entries; ++i) a.batch_entry[i] = order[i].second;
    a.pair = pair ? 1 : 0;
    a.n_items = a.n_entries * (pair ? kHeads / 2 : kHeads);
    cudaError_t e;
    if ((e = GA_CUDA(launch_q_prologue_seq(a.qg, w_q, cos_tab, sin_tab, grp_rows, sp, a.out,
                                           dev->sm_count, s))) !=
        cudaSuccess)
      return fail_cuda(e);
    CUtensorMap tm_q, tm_g;
    st = encode_q_map(&tm_q, a.out, grp_rows);
    if (st != GA_OK) return st;
    st = encode_gate_map(&tm_g, a.qg, grp_rows);
    if (st != GA_OK) return st;
    // the output map is the prepared-query map: the attention writes each row tile over the
    // queries it has read
    const int cap = pair ? dev->gated_pair_clusters : dev->sm_count;
    const int grid = (pair ? 2 : 1) * (a.n_items < cap ? a.n_items : cap);
    if ((e = GA_CUDA(launch_attn(tm_q, tm_k, tm_v, tm_g, tm_q, a, grid, s))) != cudaSuccess)
      return fail_cuda(e);
    p0 = p1;
  }
  return GA_OK;
}

}  // namespace
}  // namespace ga

using namespace ga;

extern "C" {

int ga_abi_version(void) { return GA_ABI_VERSION; }

int ga_check_geometry(const ga_geometry* g) {
  if (!g) return GA_ERR_NULL;
  if (g->n_q_heads != GA_N_Q_HEADS || g->n_kv_heads != GA_N_KV_HEADS ||
      g->head_dim != GA_HEAD_DIM || g->rope_dims != GA_ROPE_DIMS || g->eps != 1e-6f ||
      g->rope_base != 1e7)
    return GA_ERR_GEOMETRY;
  return GA_OK;
}

const char* ga_status_string(int status) {
  switch (status) {
    case GA_OK: return "ok";
    case GA_ERR_NULL: return "a required pointer is NULL";
    case GA_ERR_SHAPE: return "a size is negative or zero where it must be positive";
    case GA_ERR_ALIGN: return "a pointer or leading dimension is not 16-byte aligned";
    case GA_ERR_RANGE: return "a window, position or size is out of range";
    case GA_ERR_TABLE: return "the cos/sin table is shorter than the largest position + 1";
    case GA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case GA_ERR_DEVICE: return "the current device is not sm_103 or refused set-up";
    case GA_ERR_CUDA: return "a CUDA call failed (see ga_last_cuda_error)";
    case GA_ERR_GEOMETRY: return "geometry differs from the compiled 24/2/256/64/1e-6/1e7";
    default: return "unknown status";
  }
}

int ga_last_cuda_error(void) { return t_last_cuda_error; }

unsigned long long ga_debug_cuda_calls(void) { return g_cuda_calls.load(); }

int ga_device_status(int* status_out, int clear) {
  if (!status_out) return GA_ERR_NULL;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaError_t e = GA_CUDA(cudaDeviceSynchronize());
  if (e != cudaSuccess) return fail_cuda(e);
  if ((e = GA_CUDA(cudaMemcpy(status_out, dev->status_word, sizeof(int), cudaMemcpyDeviceToHost))) != cudaSuccess)
    return fail_cuda(e);
  if (clear && (e = GA_CUDA(cudaMemset(dev->status_word, 0, sizeof(int)))) != cudaSuccess)
    return fail_cuda(e);
  return GA_OK;
}

int ga_debug_wait_timeout(long long limit_cycles, ga_stream stream) {
  if (limit_cycles < 1 || limit_cycles > 2000000000LL) return GA_ERR_RANGE;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaError_t e = GA_CUDA(launch_wait_timeout(limit_cycles, dev->status_word, (cudaStream_t)stream));
  return e == cudaSuccess ? GA_OK : fail_cuda(e);
}

int ga_debug_set_cta_pairs(int mode) {
  if (mode < 0 || mode > 2) return GA_ERR_RANGE;
  return g_cta_pairs.exchange(mode);
}

int ga_debug_qk_fp32(const ga_bf16* q, const ga_bf16* k, int n_tiles, float* s,
                     ga_stream stream) {
  if (!q || !k || !s) return GA_ERR_NULL;
  if (n_tiles < 0) return GA_ERR_SHAPE;
  if (n_tiles > 65535) return GA_ERR_RANGE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(s, 16)) return GA_ERR_ALIGN;
  if (n_tiles == 0) return GA_OK;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaError_t e = GA_CUDA(launch_qk_probe(q, k, n_tiles, s, dev->status_word, (cudaStream_t)stream));
  return e == cudaSuccess ? GA_OK : fail_cuda(e);
}

int ga_rope_table_host(int n_pos, ga_bf16* cos_out, ga_bf16* sin_out) {
  if (!cos_out || !sin_out) return GA_ERR_NULL;
  if (n_pos < 0) return GA_ERR_SHAPE;
  if (n_pos > GA_MAX_TOKENS) return GA_ERR_RANGE;
  double inv_freq[kHalfRot];
  for (int i = 0; i < kHalfRot; ++i) inv_freq[i] = std::pow(kRopeBase, -(2.0 * i) / 64.0);
  for (int p = 0; p < n_pos; ++p)
    for (int i = 0; i < kHalfRot; ++i) {
      const double ang = (double)p * inv_freq[i];
      cos_out[(size_t)p * kHalfRot + i] = bf16_rne(std::cos(ang));
      sin_out[(size_t)p * kHalfRot + i] = bf16_rne(std::sin(ang));
    }
  return GA_OK;
}

int ga_k_prologue(const ga_bf16* k_raw, const ga_bf16* w_k, const ga_bf16* cos_tab,
                  const ga_bf16* sin_tab, int table_rows, int n_tok, int pos_base,
                  ga_bf16* k_prep, ga_stream stream) {
  if (!k_raw || !w_k || !cos_tab || !sin_tab || !k_prep) return GA_ERR_NULL;
  if (n_tok < 0 || table_rows < 0) return GA_ERR_SHAPE;
  if (pos_base < 0 || n_tok > GA_MAX_TOKENS || pos_base > GA_MAX_TOKENS) return GA_ERR_RANGE;
  if ((long long)table_rows < (long long)pos_base + n_tok) return GA_ERR_TABLE;
  if (!aligned(k_raw, 16) || !aligned(k_prep, 16) || !aligned(w_k, 16) || !aligned(cos_tab, 16) ||
      !aligned(sin_tab, 16))
    return GA_ERR_ALIGN;
  if (n_tok == 0) return GA_OK;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaError_t e = GA_CUDA(launch_k_prologue(k_raw, w_k, cos_tab, sin_tab, n_tok, pos_base, k_prep,
                                            dev->sm_count, (cudaStream_t)stream));
  return e == cudaSuccess ? GA_OK : fail_cuda(e);
}

int ga_q_prologue(const ga_bf16* qg, const ga_bf16* w_q, const ga_bf16* cos_tab,
                  const ga_bf16* sin_tab, int table_rows, int rows, int q_base,
                  ga_bf16* q_prep, ga_stream stream) {
  if (!qg || !w_q || !cos_tab || !sin_tab || !q_prep) return GA_ERR_NULL;
  if (rows < 0 || table_rows < 0) return GA_ERR_SHAPE;
  if (q_base < 0 || rows > GA_MAX_TOKENS || q_base > GA_MAX_TOKENS) return GA_ERR_RANGE;
  if ((long long)table_rows < (long long)q_base + rows) return GA_ERR_TABLE;
  if (!aligned(qg, 16) || !aligned(q_prep, 16) || !aligned(w_q, 16) || !aligned(cos_tab, 16) ||
      !aligned(sin_tab, 16))
    return GA_ERR_ALIGN;
  if (rows == 0) return GA_OK;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaError_t e = GA_CUDA(launch_q_prologue(qg, w_q, cos_tab, sin_tab, rows, q_base, 0, kHeads,
                                            q_prep, dev->sm_count, (cudaStream_t)stream));
  return e == cudaSuccess ? GA_OK : fail_cuda(e);
}

int ga_qk_prologue(const ga_bf16* k_raw, const ga_bf16* w_k, int n_tok, int k_pos_base,
                   ga_bf16* k_prep, const ga_bf16* qg, const ga_bf16* w_q, int rows, int q_base,
                   ga_bf16* q_prep, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                   int table_rows, ga_stream stream) {
  if (!k_raw || !w_k || !k_prep || !qg || !w_q || !q_prep || !cos_tab || !sin_tab)
    return GA_ERR_NULL;
  if (n_tok < 0 || rows < 0 || table_rows < 0) return GA_ERR_SHAPE;
  if (k_pos_base < 0 || n_tok > GA_MAX_TOKENS || k_pos_base > GA_MAX_TOKENS || q_base < 0 ||
      rows > GA_MAX_TOKENS || q_base > GA_MAX_TOKENS)
    return GA_ERR_RANGE;
  if ((long long)table_rows < (long long)k_pos_base + n_tok ||
      (long long)table_rows < (long long)q_base + rows)
    return GA_ERR_TABLE;
  if (!aligned(k_raw, 16) || !aligned(k_prep, 16) || !aligned(w_k, 16) || !aligned(qg, 16) ||
      !aligned(q_prep, 16) || !aligned(w_q, 16) || !aligned(cos_tab, 16) || !aligned(sin_tab, 16))
    return GA_ERR_ALIGN;
  if (n_tok == 0 && rows == 0) return GA_OK;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaError_t e = GA_CUDA(launch_qk_prologue(k_raw, w_k, n_tok, k_pos_base, k_prep, qg, w_q, rows,
                                             q_base, q_prep, cos_tab, sin_tab, dev->sm_count,
                                             (cudaStream_t)stream));
  return e == cudaSuccess ? GA_OK : fail_cuda(e);
}

int ga_attn_prefill_prepared(const ga_bf16* q_prep, const ga_bf16* qg, const ga_bf16* k_prep,
                             const ga_bf16* v, int rows, int T, int q_base, int causal,
                             ga_bf16* out, float* row_stats, ga_stream stream) {
  if (!q_prep || !qg || !k_prep || !v || !out) return GA_ERR_NULL;
  if (rows < 0 || T < 1) return GA_ERR_SHAPE;
  if (T > GA_MAX_TOKENS || q_base < 0 || q_base % 64 != 0 || (long long)q_base + rows > T)
    return GA_ERR_RANGE;
  if (causal != 0 && causal != 1) return GA_ERR_RANGE;
  if (!causal && q_base != 0) return GA_ERR_RANGE;
  if (!aligned(q_prep, 16) || !aligned(qg, 16) || !aligned(k_prep, 16) || !aligned(v, 16) ||
      !aligned(out, 16) || (row_stats && !aligned(row_stats, 4)))
    return GA_ERR_ALIGN;
  if (rows == 0) return GA_OK;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  AttnArgs a{};
  a.qg = qg;
  a.out = out; a.row_stats = row_stats;
  a.rows = rows; a.T = T; a.q_base = q_base;
  a.mode = causal ? kModeCausal : kModeBidir;
  return launch_attention(a, const_cast<uint16_t*>(q_prep), true, k_prep, v, T, dev,
                          (cudaStream_t)stream);
}

int ga_attn_prefill_kv(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                       const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                       int table_rows, int rows, int T, int q_base, int causal, int kv_first,
                       int kv_count, ga_bf16* out, float* row_stats, ga_stream stream) {
  int st = check_attention_args(qg, k_prep, v, w_q, cos_tab, sin_tab, table_rows, rows, T,
                                q_base, out);
  if (st != GA_OK) return st;
  if (causal != 0 && causal != 1) return GA_ERR_RANGE;
  if (!causal && q_base != 0) return GA_ERR_RANGE;  // bidirectional passes start at 0
  if (kv_first < 0 || kv_count < 1 || kv_first + kv_count > kKvHeads) return GA_ERR_RANGE;
  if (row_stats && !aligned(row_stats, 4)) return GA_ERR_ALIGN;
  if (rows == 0) return GA_OK;
  DeviceState* dev = nullptr;
  st = current_device(&dev);
  if (st != GA_OK) return st;
  AttnArgs a{};
  a.qg = qg; a.w_q = w_q; a.cos_tab = cos_tab; a.sin_tab = sin_tab;
  a.out = out; a.row_stats = row_stats;
  a.rows = rows; a.T = T; a.q_base = q_base;
  a.mode = causal ? kModeCausal : kModeBidir;
  a.head0 = kv_first * kGroup;
  a.n_heads = kv_count * kGroup;
  return launch_attention(a, out, false, k_prep, v, T, dev, (cudaStream_t)stream);
}

int ga_attn_prefill(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                    const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                    int table_rows, int rows, int T, int q_base, int causal, ga_bf16* out,
                    float* row_stats, ga_stream stream) {
  return ga_attn_prefill_kv(qg, k_prep, v, w_q, cos_tab, sin_tab, table_rows, rows, T, q_base,
                            causal, 0, kKvHeads, out, row_stats, stream);
}

size_t ga_masked_workspace_bytes(int rows, int T) {
  if (rows < 0 || T < 1 || T > GA_MASKED_MAX_TOKENS) return 0;
  return masked_layout(rows, T).total;
}

}  // extern "C"

namespace ga {
namespace {
// Every check of a stored-mask call except the workspace's (no CUDA call); shared by
// ga_attn_masked and ga_attn_masked_static.
int masked_check_args(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                      const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                      int table_rows, int rows, int T, int q_base, const uint8_t* mask,
                      long long ld_mask, const ga_bf16* out, const ga_bf16* weights,
                      const int* hidden_rows) {
  int st = check_attention_args(qg, k_prep, v, w_q, cos_tab, sin_tab, table_rows, rows, T,
                                q_base, out);
  if (st != GA_OK) return st;
  if (!mask) return GA_ERR_NULL;
  if (T > GA_MASKED_MAX_TOKENS || ld_mask < T) return GA_ERR_RANGE;
  if (!aligned(mask, 16) || ld_mask % 16 != 0) return GA_ERR_ALIGN;
  if ((weights && !aligned(weights, 16)) || (hidden_rows && !aligned(hidden_rows, 4)))
    return GA_ERR_ALIGN;
  return GA_OK;
}
}  // namespace
}  // namespace ga

extern "C" {

}  // extern "C"

namespace ga {
namespace {
// The stored-mask call after its checks: zero hidden_rows, the mask prepass into the
// workspace, the query prologue into the workspace (unless q_prep already holds the
// prepared queries), the attention, and the weights pass when weights are wanted.
int masked_run(const ga_bf16* q_prep_in, const ga_bf16* qg, const ga_bf16* k_prep,
               const ga_bf16* v, const ga_bf16* w_q, const ga_bf16* cos_tab,
               const ga_bf16* sin_tab, int rows, int T, int q_base, const uint8_t* mask,
               long long ld_mask, int kv_first, int kv_count, ga_bf16* out, ga_bf16* weights,
               int* hidden_rows, void* workspace, ga_stream stream) {
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  const MaskedLayout L = masked_layout(rows, T);
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* bits = reinterpret_cast<uint32_t*>(ws + L.bits_off);
  uint8_t* flags = ws + L.flags_off;
  float* stats = reinterpret_cast<float*>(ws + L.stats_off);
  uint16_t* q_prep = q_prep_in ? const_cast<uint16_t*>(q_prep_in)
                               : reinterpret_cast<uint16_t*>(ws + L.q_off);
  cudaError_t e;
  if (hidden_rows && (e = GA_CUDA(cudaMemsetAsync(hidden_rows, 0, sizeof(int), s))) != cudaSuccess)
    return fail_cuda(e);
  if ((e = GA_CUDA(launch_mask_prepass(mask, ld_mask, rows, T, bits, L.mask_words, flags,
                                       L.key_tiles, s))) != cudaSuccess)
    return fail_cuda(e);
  AttnArgs a{};
  a.qg = qg; a.w_q = w_q; a.cos_tab = cos_tab; a.sin_tab = sin_tab;
  a.out = out; a.row_stats = stats; a.hidden_rows = hidden_rows;
  a.mask_bits = bits; a.tile_flags = flags;
  a.key_tiles = L.key_tiles; a.mask_words = L.mask_words;
  a.rows = rows; a.T = T; a.q_base = q_base; a.mode = kModeMask;
  a.head0 = kv_first * kGroup;
  a.n_heads = kv_count * kGroup;
  st = launch_attention(a, q_prep, q_prep_in != nullptr, k_prep, v, T, dev, s);
  if (st != GA_OK || !weights) return st;
  // the weights of the heads processed: zero first (hidden keys stay 0), then the pass
  const size_t head_elems = (size_t)rows * T;
  if ((e = GA_CUDA(cudaMemsetAsync(weights + (size_t)a.head0 * head_elems, 0,
                                   (size_t)a.n_heads * head_elems * sizeof(uint16_t), s))) != cudaSuccess)
    return fail_cuda(e);
  a.weights = weights;
  a.weights_pass = 1;
  a.hidden_rows = nullptr;
  return launch_attention(a, q_prep, true, k_prep, v, T, dev, s);
}
}  // namespace
}  // namespace ga

extern "C" {

int ga_attn_masked_kv(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                      const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                      int table_rows, int rows, int T, int q_base, const uint8_t* mask,
                      long long ld_mask, int kv_first, int kv_count, ga_bf16* out,
                      ga_bf16* weights, int* hidden_rows, void* workspace, size_t ws_bytes,
                      ga_stream stream) {
  int st = masked_check_args(qg, k_prep, v, w_q, cos_tab, sin_tab, table_rows, rows, T, q_base,
                             mask, ld_mask, out, weights, hidden_rows);
  if (st != GA_OK) return st;
  if (kv_first < 0 || kv_count < 1 || kv_first + kv_count > kKvHeads) return GA_ERR_RANGE;
  if (!workspace || !aligned(workspace, 256) || ws_bytes < masked_layout(rows, T).total)
    return GA_ERR_WORKSPACE;
  if (rows == 0) return GA_OK;
  return masked_run(nullptr, qg, k_prep, v, w_q, cos_tab, sin_tab, rows, T, q_base, mask,
                    ld_mask, kv_first, kv_count, out, weights, hidden_rows, workspace, stream);
}

int ga_attn_masked(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                   const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                   int table_rows, int rows, int T, int q_base, const uint8_t* mask,
                   long long ld_mask, ga_bf16* out, ga_bf16* weights, int* hidden_rows,
                   void* workspace, size_t ws_bytes, ga_stream stream) {
  return ga_attn_masked_kv(qg, k_prep, v, w_q, cos_tab, sin_tab, table_rows, rows, T, q_base,
                           mask, ld_mask, 0, kKvHeads, out, weights, hidden_rows, workspace,
                           ws_bytes, stream);
}

int ga_attn_masked_prepared(const ga_bf16* q_prep, const ga_bf16* qg, const ga_bf16* k_prep,
                            const ga_bf16* v, int rows, int T, int q_base, const uint8_t* mask,
                            long long ld_mask, ga_bf16* out, ga_bf16* weights,
                            int* hidden_rows, void* workspace, size_t ws_bytes,
                            ga_stream stream) {
  if (!q_prep) return GA_ERR_NULL;
  // the prepared queries stand in for w_q and the tables in the shared checks (no
  // table is read; table_rows is the largest position + 1)
  int st = masked_check_args(qg, k_prep, v, q_prep, q_prep, q_prep, q_base + rows, rows, T,
                             q_base, mask, ld_mask, out, weights, hidden_rows);
  if (st != GA_OK) return st;
  if (!workspace || !aligned(workspace, 256) || ws_bytes < masked_layout(rows, T).total)
    return GA_ERR_WORKSPACE;
  if (rows == 0) return GA_OK;
  return masked_run(q_prep, qg, k_prep, v, nullptr, nullptr, nullptr, rows, T, q_base, mask,
                    ld_mask, 0, kKvHeads, out, weights, hidden_rows, workspace, stream);
}

size_t ga_verify_workspace_bytes(int n_seq, int rows, int max_len) {
  if (n_seq < 1 || rows < 1 || rows > kVerifyMaxRows || max_len < 0 || max_len > GA_MAX_TOKENS)
    return 0;
  return verify_ws_bytes(verify_plan(n_seq, rows, max_len));
}

int ga_attn_verify(const ga_bf16* qg, const ga_bf16* k_cache, const ga_bf16* v_cache, int cap,
                   const int* seq_len, int n_seq, int rows, const ga_bf16* w_q,
                   const ga_bf16* cos_tab, const ga_bf16* sin_tab, int table_rows,
                   ga_bf16* out, void* workspace, size_t ws_bytes, ga_stream stream) {
  if (!qg || !k_cache || !v_cache || !seq_len || !w_q || !cos_tab || !sin_tab || !out)
    return GA_ERR_NULL;
  if (n_seq < 0 || rows < 0 || cap < 1 || table_rows < 0) return GA_ERR_SHAPE;
  if (rows > 16 || cap > GA_MAX_TOKENS) return GA_ERR_RANGE;
  for (int b = 0; b < n_seq; ++b)
    if (seq_len[b] < 0 || (long long)seq_len[b] + rows > cap) return GA_ERR_RANGE;
  VerifyCaches c{};
  c.k = k_cache;
  c.v = v_cache;
  c.cap = cap;
  return verify_run(qg, c, seq_len, n_seq, rows, w_q, cos_tab, sin_tab, table_rows, out,
                    workspace, ws_bytes, stream);
}

int ga_attn_verify_e4m3(const ga_bf16* qg, const uint8_t* k_codes, const float* k_scale,
                        const uint8_t* v_codes, const float* v_scale, int cap, const int* seq_len,
                        int n_seq, int rows, const ga_bf16* w_q, const ga_bf16* cos_tab,
                        const ga_bf16* sin_tab, int table_rows, ga_bf16* out, void* workspace,
                        size_t ws_bytes, ga_stream stream) {
  if (!qg || !k_codes || !k_scale || !v_codes || !v_scale || !seq_len || !w_q || !cos_tab ||
      !sin_tab || !out)
    return GA_ERR_NULL;
  if (n_seq < 0 || rows < 0 || cap < 1 || table_rows < 0) return GA_ERR_SHAPE;
  if (rows > 16 || cap > GA_MAX_TOKENS) return GA_ERR_RANGE;
  for (int b = 0; b < n_seq; ++b)
    if (seq_len[b] < 0 || (long long)seq_len[b] + rows > cap) return GA_ERR_RANGE;
  VerifyCaches c{};
  c.k8 = k_codes;
  c.v8 = v_codes;
  c.k_scale = k_scale;
  c.v_scale = v_scale;
  c.cap = cap;
  return verify_run(qg, c, seq_len, n_seq, rows, w_q, cos_tab, sin_tab, table_rows, out,
                    workspace, ws_bytes, stream);
}

int ga_attn_verify_paged(const ga_bf16* qg, const ga_bf16* k_pages, const ga_bf16* v_pages,
                         int n_pages, int page_size, const int* page_table, int max_pages,
                         const int* seq_len, int n_seq, int rows, const ga_bf16* w_q,
                         const ga_bf16* cos_tab, const ga_bf16* sin_tab, int table_rows,
                         ga_bf16* out, void* workspace, size_t ws_bytes, ga_stream stream) {
  if (!qg || !k_pages || !v_pages || !page_table || !seq_len || !w_q || !cos_tab || !sin_tab ||
      !out)
    return GA_ERR_NULL;
  if (n_seq < 0 || rows < 0 || n_pages < 1 || page_size < 1 || max_pages < 1 || table_rows < 0)
    return GA_ERR_SHAPE;
  if (rows > 16 || page_size % kTileN != 0 || page_size > GA_MAX_TOKENS) return GA_ERR_RANGE;
  for (int b = 0; b < n_seq; ++b)
    if (seq_len[b] < 0 || (long long)seq_len[b] + rows > (long long)max_pages * page_size ||
        (long long)seq_len[b] + rows > GA_MAX_TOKENS)
      return GA_ERR_RANGE;
  if (!aligned(page_table, 4)) return GA_ERR_ALIGN;
  VerifyCaches c{};
  c.k = k_pages;
  c.v = v_pages;
  c.page_table = page_table;
  c.page_size = page_size;
  c.max_pages = max_pages;
  c.n_pages = n_pages;
  return verify_run(qg, c, seq_len, n_seq, rows, w_q, cos_tab, sin_tab, table_rows, out,
                    workspace, ws_bytes, stream);
}

int ga_attn_prefill_batch(const ga_bf16* qg, const int* row_start, const int* q_base, int n_seq,
                          const ga_bf16* k_pages, const ga_bf16* v_pages, int n_pages,
                          int page_size, const int* page_table, int max_pages, const ga_bf16* w_q,
                          const ga_bf16* cos_tab, const ga_bf16* sin_tab, int table_rows,
                          ga_bf16* out, ga_stream stream) {
  if (!qg || !row_start || !q_base || !k_pages || !v_pages || !page_table || !w_q || !cos_tab ||
      !sin_tab || !out)
    return GA_ERR_NULL;
  if (n_seq < 0 || n_pages < 1 || page_size < 1 || max_pages < 1 || table_rows < 0 ||
      row_start[0] < 0)
    return GA_ERR_SHAPE;
  if (page_size % kTileN != 0 || page_size > GA_MAX_TOKENS) return GA_ERR_RANGE;
  long long max_T = 0;
  for (int b = 0; b < n_seq; ++b) {
    const long long rows = (long long)row_start[b + 1] - row_start[b];
    if (rows < 0) return GA_ERR_SHAPE;
    if (q_base[b] < 0 || q_base[b] % 64 != 0) return GA_ERR_RANGE;
    const long long T = (long long)q_base[b] + rows;
    if (T > (long long)max_pages * page_size || T > GA_MAX_TOKENS) return GA_ERR_RANGE;
    if (T > max_T) max_T = T;
  }
  if (row_start[n_seq] > GA_MAX_TOKENS) return GA_ERR_RANGE;
  if ((long long)table_rows < max_T) return GA_ERR_TABLE;
  if (!aligned(qg, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(w_q, 16) ||
      !aligned(cos_tab, 16) || !aligned(sin_tab, 16) || !aligned(out, 16) ||
      !aligned(page_table, 4))
    return GA_ERR_ALIGN;
  std::vector<BatchPiece> pieces;
  for (int b = 0; b < n_seq; ++b) {
    const int rows = row_start[b + 1] - row_start[b];
    for (int r0 = 0; r0 < rows; r0 += kBatchMaxEntries * kTileM) {
      const int n = std::min(rows - r0, kBatchMaxEntries * kTileM);
      pieces.push_back({b, row_start[b] + r0, n, q_base[b] + r0});
    }
  }
  if (pieces.empty()) return GA_OK;
  return batch_run(qg, pieces.data(), (int)pieces.size(), k_pages, v_pages, n_pages, page_size,
                   page_table, max_pages, w_q, cos_tab, sin_tab, out, stream);
}

int ga_kv_quantize_e4m3(const ga_bf16* x, long long n_tok, uint8_t* q, float* scale,
                        ga_stream stream) {
  if (!x || !q || !scale) return GA_ERR_NULL;
  if (n_tok < 0) return GA_ERR_SHAPE;
  if (n_tok > (long long)GA_MAX_TOKENS * 64) return GA_ERR_RANGE;
  if (!aligned(x, 8) || !aligned(q, 4) || !aligned(scale, 4)) return GA_ERR_ALIGN;
  if (n_tok == 0) return GA_OK;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaError_t e = GA_CUDA(launch_quantize_e4m3(x, n_tok * kKvHeads, q, scale, (cudaStream_t)stream));
  if (e != cudaSuccess) return fail_cuda(e);
  return GA_OK;
}

int ga_kv_dequantize_e4m3(const uint8_t* q, const float* scale, long long n_tok, ga_bf16* out,
                          ga_stream stream) {
  if (!q || !scale || !out) return GA_ERR_NULL;
  if (n_tok < 0) return GA_ERR_SHAPE;
  if (n_tok > (long long)GA_MAX_TOKENS * 64) return GA_ERR_RANGE;
  if (!aligned(q, 8) || !aligned(scale, 4) || !aligned(out, 16)) return GA_ERR_ALIGN;
  if (n_tok == 0) return GA_OK;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaError_t e = GA_CUDA(launch_dequantize_e4m3(q, scale, n_tok * kKvHeads,
                                                 reinterpret_cast<uint16_t*>(out),
                                                 (cudaStream_t)stream));
  if (e != cudaSuccess) return fail_cuda(e);
  return GA_OK;
}

size_t ga_prefill_e4m3_workspace_bytes(int T) {
  if (T < 1 || T > GA_MAX_TOKENS) return 0;
  return 2 * (size_t)T * kKvHeads * kDim * sizeof(uint16_t);
}

int ga_attn_prefill_e4m3(const ga_bf16* qg, const uint8_t* k_codes, const float* k_scale,
                         const uint8_t* v_codes, const float* v_scale, const ga_bf16* w_q,
                         const ga_bf16* cos_tab, const ga_bf16* sin_tab, int table_rows,
                         int rows, int T, int q_base, int causal, ga_bf16* out,
                         float* row_stats, void* workspace, size_t ws_bytes, ga_stream stream) {
  // the code arrays stand in for the bf16 caches in the shared checks (16-byte aligned)
  int st = check_attention_args(qg, k_codes, v_codes, w_q, cos_tab, sin_tab, table_rows, rows,
                                T, q_base, out);
  if (st != GA_OK) return st;
  if (!k_scale || !v_scale) return GA_ERR_NULL;
  if (causal != 0 && causal != 1) return GA_ERR_RANGE;
  if (!causal && q_base != 0) return GA_ERR_RANGE;   // bidirectional passes start at 0
  if (!aligned(k_scale, 4) || !aligned(v_scale, 4) || (row_stats && !aligned(row_stats, 4)))
    return GA_ERR_ALIGN;
  if (!workspace || !aligned(workspace, 256) || ws_bytes < ga_prefill_e4m3_workspace_bytes(T))
    return GA_ERR_WORKSPACE;
  if (rows == 0) return GA_OK;
  // the widened K and V live in the workspace: [T][2][256] bf16 each
  ga_bf16* k_wide = static_cast<ga_bf16*>(workspace);
  ga_bf16* v_wide = k_wide + (size_t)T * kKvHeads * kDim;
  DeviceState* dev = nullptr;
  st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if ((e = GA_CUDA(launch_dequantize_e4m3(k_codes, k_scale, (long long)T * kKvHeads,
                                          reinterpret_cast<uint16_t*>(k_wide), s))) != cudaSuccess)
    return fail_cuda(e);
  if ((e = GA_CUDA(launch_dequantize_e4m3(v_codes, v_scale, (long long)T * kKvHeads,
                                          reinterpret_cast<uint16_t*>(v_wide), s))) != cudaSuccess)
    return fail_cuda(e);
  AttnArgs a{};
  a.qg = qg; a.w_q = w_q; a.cos_tab = cos_tab; a.sin_tab = sin_tab;
  a.out = out; a.row_stats = row_stats;
  a.rows = rows; a.T = T; a.q_base = q_base;
  a.mode = causal ? kModeCausal : kModeBidir;
  return launch_attention(a, out, false, k_wide, v_wide, T, dev, s);
}

int ga_select_mask(const float* block_scores, long long ld_scores, int rows, int T, int q_base,
                   int block_topk, uint8_t* mask, long long ld_mask, ga_stream stream) {
  if (!block_scores || !mask) return GA_ERR_NULL;
  if (rows < 0 || T < 1 || q_base < 0 || block_topk < 1) return GA_ERR_SHAPE;
  if (T > GA_MASKED_MAX_TOKENS || (long long)q_base + rows > T) return GA_ERR_RANGE;
  const long long n_blocks = (T + GA_INDEX_BLOCK_TOKENS - 1) / GA_INDEX_BLOCK_TOKENS;
  if (ld_scores < n_blocks || ld_mask < T || ld_scores > (1LL << 31) || ld_mask > (1LL << 31))
    return GA_ERR_RANGE;
  if (!aligned(block_scores, 4) || !aligned(mask, 16) || ld_mask % 16 != 0) return GA_ERR_ALIGN;
  if (rows == 0) return GA_OK;
  DeviceState* dev = nullptr;
  int st = current_device(&dev);
  if (st != GA_OK) return st;
  cudaError_t e = GA_CUDA(launch_select_mask(block_scores, ld_scores, rows, T, q_base, block_topk,
                                             mask, ld_mask, (cudaStream_t)stream));
  if (e != cudaSuccess) return fail_cuda(e);
  return GA_OK;
}

// ------------------------------------------------------------------ allocation-free masked call
// The scratch of ga_attn_masked_static: one static array per device, reserved at module
// load, its address looked up once per device on the first call (with that device current).
}  // extern "C"

namespace ga {
namespace {
__device__ __align__(256) uint8_t g_static_scratch[GA_STATIC_SCRATCH_BYTES];
void* g_static_scratch_ptr[kMaxDevices];
std::mutex g_static_mutex;
}  // namespace
}  // namespace ga

extern "C" {

int ga_attn_masked_static(const ga_bf16* qg, const ga_bf16* k_prep, const ga_bf16* v,
                          const ga_bf16* w_q, const ga_bf16* cos_tab, const ga_bf16* sin_tab,
                          int table_rows, int rows, int T, int q_base, const uint8_t* mask,
                          long long ld_mask, ga_bf16* out, ga_bf16* weights, int* hidden_rows,
                          ga_stream stream) {
  // Every argument check first, with no CUDA call (the same checks as ga_attn_masked),
  // then the size limit of the static scratch.
  int st = masked_check_args(qg, k_prep, v, w_q, cos_tab, sin_tab, table_rows, rows, T, q_base,
                             mask, ld_mask, out, weights, hidden_rows);
  if (st != GA_OK) return st;
  if (masked_layout(rows, T).total > GA_STATIC_SCRATCH_BYTES) return GA_ERR_WORKSPACE;
  if (rows == 0) return GA_OK;
  int dev = 0;
  cudaError_t e = GA_CUDA(cudaGetDevice(&dev));
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return GA_ERR_DEVICE;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!g_static_scratch_ptr[dev]) {
      void* p = nullptr;
      if ((e = GA_CUDA(cudaGetSymbolAddress(&p, g_static_scratch))) != cudaSuccess)
        return fail_cuda(e);
      g_static_scratch_ptr[dev] = p;
    }
    scratch = g_static_scratch_ptr[dev];
  }
  return masked_run(nullptr, qg, k_prep, v, w_q, cos_tab, sin_tab, rows, T, q_base, mask,
                    ld_mask, 0, kKvHeads, out, weights, hidden_rows, scratch, stream);
}

}  // extern "C"
