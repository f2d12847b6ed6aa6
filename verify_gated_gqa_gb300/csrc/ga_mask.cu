// Mask prepass for stored-mask attention (pegainfer PR #1151, "feat(qwen4): add the QSA
// sparse-attention kernel and its golden", §Semantics: the kernel consumes the selection
// mask as given, non-zero = visible).
//
// Reads the uint8 mask once and writes (a) one bit per (row, key) -- word w of a row holds
// keys 32w .. 32w+31, key 32w + j at bit mask_bit_pos(j), the order in which the attention
// kernel's softmax turns bits into score masks -- and (b) one flag per (128-row tile,
// 128-key tile) that says whether any key of the tile is visible to any row of the tile,
// so the attention kernel skips all-hidden tiles without loading them. Rows >= rows and
// keys >= T read as hidden.
#include "ga_internal.h"

namespace ga {
namespace {

// One CTA of 256 threads per (128-row tile, four 128-key tiles): warp w takes rows 16w ..
// 16w+15 of the tile, one row per instruction, lane l the 16 keys 16l .. 16l+15 of the 512
// (a 16-byte load; the warp reads 512 contiguous bytes of the row). A byte is visible when
// it is non-zero: ((x & 0x7F..) + 0x7F..) | x has bit 7 of each byte set exactly then (no
// carry crosses a byte). Key j of a 32-key word belongs at bit 8 (j % 4) + 7 - j / 4: for the
// lane's bytes 4i .. 4i+3 of word half h that is bit 7 - (4h + i) of the byte's own
// position, one shift of those top bits. The two lanes of a word combine by one shuffle; a
// tile's flag is the OR over its 8 lanes and the 8 warps. At most 32 registers a thread, so
// eight CTAs fit an SM and the 1,024 CTAs of an 8192 x 8192 mask run as one wave.
constexpr int kPrepThreads = 256;
constexpr int kPrepKeyTiles = 4;

__global__ void __launch_bounds__(kPrepThreads, 8) mask_prepass_kernel(
    const uint8_t* __restrict__ mask, long long ld_mask, int rows, int T,
    uint32_t* __restrict__ bits, int mask_words, uint8_t* __restrict__ flags, int key_tiles) {
  const int kt0 = blockIdx.x * kPrepKeyTiles, mt = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int key = kt0 * kTileN + 16 * lane;   // this lane's first key
  const bool tile_ok = kt0 + (lane >> 3) < key_tiles;
  const uint32_t h = (uint32_t)(lane & 1);     // the lane's half of its 32-key word
  uint32_t any = 0u;
#pragma unroll 2
  for (int i = 0; i < 16; ++i) {
    const int row = mt * kTileM + warp * 16 + i;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < rows && key < T) {
      const uint8_t* src = mask + (long long)row * ld_mask + key;
      if (key + 16 <= T) {
        v = __ldg(reinterpret_cast<const uint4*>(src));
      } else {   // the row's last keys: byte by byte, the rest hidden
        uint32_t w4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (key + e < T) w4[e >> 2] |= (uint32_t)src[e] << (8 * (e & 3));
        v = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t nz = (((x[q] & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | x[q]) & 0x80808080u;
      m |= nz >> (4u * h + (uint32_t)q);
    }
    any |= m;
    const uint32_t word = m | __shfl_xor_sync(0xffffffffu, m, 1);
    if ((lane & 1) == 0 && tile_ok)   // rows past the call's end get zero words
      bits[(size_t)row * mask_words + (size_t)kt0 * (kTileN / 32) + (lane >> 1)] = word;
  }
  any |= __shfl_xor_sync(0xffffffffu, any, 1);
  any |= __shfl_xor_sync(0xffffffffu, any, 2);
  any |= __shfl_xor_sync(0xffffffffu, any, 4);
  __shared__ uint32_t tile_any[kPrepThreads / 32][kPrepKeyTiles];
  if ((lane & 7) == 0) tile_any[warp][lane >> 3] = any;
  __syncthreads();
  if (threadIdx.x < kPrepKeyTiles && kt0 + (int)threadIdx.x < key_tiles) {
    uint32_t o = 0u;
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) o |= tile_any[w][threadIdx.x];
    flags[(size_t)mt * kMaskFlagStride + kt0 + threadIdx.x] = o ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_mask_prepass(const uint8_t* mask, long long ld_mask, int rows, int T,
                                uint32_t* bits, int mask_words, uint8_t* flags, int key_tiles,
                                cudaStream_t s) {
  const int row_tiles = (rows + kTileM - 1) / kTileM;
  dim3 grid((unsigned)((key_tiles + kPrepKeyTiles - 1) / kPrepKeyTiles), (unsigned)row_tiles);
  mask_prepass_kernel<<<grid, kPrepThreads, 0, s>>>(mask, ld_mask, rows, T, bits, mask_words,
                                                    flags, key_tiles);
  return cudaGetLastError();
}

}  // namespace ga
