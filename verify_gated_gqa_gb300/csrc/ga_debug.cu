// Test hook: the tensor cores' fp32 dot products of bf16 rows, formed exactly as the
// attention kernel forms its scores (S = Q K^T with tcgen05.mma kind::f16, M128 N128 K256
// as sixteen K16 steps accumulating in tensor memory, both operands in shared memory in
// the 128-byte-swizzled K-major layout of the kernel's tiles). The score is "the bf16
// GEMM result" (pegainfer PR #1151, the commit that adds the attention reader); the fp32
// reduction order inside the tensor core is the hardware's own, and this hook lets the
// tests measure how far it lies from the exact dot product.
#include "ga_internal.h"
#include "ga_sm100.cuh"

namespace ga {
namespace {

constexpr int kBlockBytes = 128 * 128;   // [128 rows][64 bf16] swizzled block
constexpr uint32_t kProbeCols = 128;

struct ProbeSmem {
  uint8_t q[4][kBlockBytes];   // dims 64b .. 64b+63 of the 128 query rows, block b
  uint8_t k[4][kBlockBytes];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
};

// One CTA per 128 x 128 tile: q, k [n][128][256] bf16 -> s [n][128][128] fp32.
__global__ void __launch_bounds__(128, 1) qk_probe_kernel(const uint16_t* __restrict__ q,
                                                          const uint16_t* __restrict__ k,
                                                          float* __restrict__ s, int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(status, 0, (int)kDevBadLaunch);
    return;
  }
  ProbeSmem& sm = *reinterpret_cast<ProbeSmem*>(smem_raw);
  const int t = threadIdx.x, warp = t >> 5;
  const size_t tile = blockIdx.x;
  // thread t copies row t of both operands: 16-byte chunk c holds dims 8c .. 8c+7
  const uint4* qr = reinterpret_cast<const uint4*>(q + (tile * 128 + t) * kDim);
  const uint4* kr = reinterpret_cast<const uint4*>(k + (tile * 128 + t) * kDim);
#pragma unroll 4
  for (int c = 0; c < kDim / 8; ++c) {
    const uint32_t off = sw128_offset((uint32_t)t, (uint32_t)(c & 7));
    *reinterpret_cast<uint4*>(sm.q[c >> 3] + off) = __ldg(qr + c);
    *reinterpret_cast<uint4*>(sm.k[c >> 3] + off) = __ldg(kr + c);
  }
  fence_async_smem();   // the tensor cores read what the threads wrote
  if (t == 0) {
    sm.abort = 0;
    mbar_init(&sm.done, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, kProbeCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (warp == 0) {
    constexpr uint32_t kId = idesc_bf16(128, 128, false, false);
    const uint64_t qd0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
    const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
#pragma unroll
    for (int kk = 0; kk < kDim / 16; ++kk) {
      const uint64_t step = (uint64_t)((kk >> 2) * (kBlockBytes >> 4) + (kk & 3) * 2);
      umma_ss_warp(tmem, qd0 + step, kd0 + step, kId, kk > 0 ? 1u : 0u);
    }
    umma_commit_warp(&sm.done);
  }
  volatile int* abort = &sm.abort;
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.done, 0, abort));
  if (ok) {
    tc_fence_after();
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float4* dst = reinterpret_cast<float4*>(s + (tile * 128 + t) * 128);
#pragma unroll 1
    for (int c0 = 0; c0 < 4; ++c0) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + 32 * c0, r);
      tmem_wait_ld(r);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[8 * c0 + i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                      __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    }
  } else if (warp == 0) {
    // the MMAs may still be in flight: let them finish before tensor memory is released
    mbar_wait_quiet(&sm.done, 0, 100000000LL);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kProbeCols);
  }
  if (t == 0 && sm.abort) atomicCAS(status, 0, sm.abort);
}

}  // namespace

cudaError_t probe_set_smem_attribute() {
  return cudaFuncSetAttribute(qk_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sizeof(ProbeSmem));
}

cudaError_t launch_qk_probe(const uint16_t* q, const uint16_t* k, int n_tiles, float* s,
                            int* status, cudaStream_t st) {
  qk_probe_kernel<<<n_tiles, 128, sizeof(ProbeSmem), st>>>(q, k, s, status);
  return cudaGetLastError();
}

}  // namespace ga
