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

__global__ void __launch_bounds__(128) mask_prepass_kernel(const uint8_t* __restrict__ mask,
                                                           long long ld_mask, int rows, int T,
                                                           uint32_t* __restrict__ bits,
                                                           int mask_words,
                                                           uint8_t* __restrict__ flags,
                                                           int key_tiles) {
  const int kt = blockIdx.x, mt = blockIdx.y;
  const int r = threadIdx.x;
  const int row = mt * kTileM + r;
  const int k0 = kt * kTileN;
  constexpr int kWords = kTileN / 32;
  uint32_t w[kWords];
#pragma unroll
  for (int i = 0; i < kWords; ++i) w[i] = 0u;
  if (row < rows) {
    const uint8_t* src = mask + (long long)row * ld_mask + k0;
#pragma unroll
    for (int c = 0; c < kTileN / 16; ++c) {  // 16-byte chunks of the row's keys
      const int j0 = k0 + 16 * c;
      uint8_t b[16];
      if (j0 + 16 <= T) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + 16 * c));
        *reinterpret_cast<uint4*>(b) = v;
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) b[e] = (j0 + e < T) ? src[16 * c + e] : 0;
      }
      uint32_t m = 0;
#pragma unroll
      for (int e = 0; e < 16; ++e) m |= (b[e] != 0 ? 1u : 0u) << mask_bit_pos(16 * (c & 1) + e);
      w[c >> 1] |= m;
    }
  }
  uint32_t any_bit = 0u;
  uint32_t* dst = bits + (size_t)row * mask_words + (size_t)kt * kWords;
#pragma unroll
  for (int i = 0; i < kWords; ++i) {
    dst[i] = w[i];
    any_bit |= w[i];
  }
  const int any = __syncthreads_or(any_bit != 0u);
  if (r == 0) flags[(size_t)mt * kMaskFlagStride + kt] = any ? 1 : 0;
}

}  // namespace

cudaError_t launch_mask_prepass(const uint8_t* mask, long long ld_mask, int rows, int T,
                                uint32_t* bits, int mask_words, uint8_t* flags, int key_tiles,
                                cudaStream_t s) {
  const int row_tiles = (rows + kTileM - 1) / kTileM;
  dim3 grid((unsigned)key_tiles, (unsigned)row_tiles);
  mask_prepass_kernel<<<grid, 128, 0, s>>>(mask, ld_mask, rows, T, bits, mask_words, flags,
                                           key_tiles);
  return cudaGetLastError();
}

}  // namespace ga
