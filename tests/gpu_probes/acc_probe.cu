// Accumulator-precision probe of the E4M3 tensor-core MMA (kind::f8f6f4) on
// sm_103a, after the SageAttention2 summary's finding that Hopper's FP8 MMA
// accumulates in fewer bits than FP32 (the reason for its two-level
// accumulation): D (128 x 64 fp32) is preset in TMEM, D += A B^T runs with A
// (128 x 128) and B (64 x 128) E4M3 tiles in the 128-byte swizzled K-major
// layout the attention kernel uses, and D comes back.  With A or B zero, D must
// come back unchanged; with A = 2^-9 in column 0 and B = 2^-(k-9) in column 0
// of row n, D[m][n] = D0 + 2^-k shows how many bits the accumulation keeps.
// Test code: one CTA of 128 threads, every wait bounded.
#include <stdint.h>

#include "sm103.cuh"

using namespace sage;

namespace {
__device__ __forceinline__ uint32_t swz128(int r, int c) {  // 16-byte chunk c of row r, 128-byte rows
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(128, 1) acc_probe_kernel(const uint8_t *a, const uint8_t *b, const float *d0,
                                                           float *out, int *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sA = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);  // 128 x 128 bytes
  uint8_t *sB = sA + 128 * 128;                                                // 64 x 128 bytes
  uint64_t *bar = (uint64_t *)(sB + 64 * 128);
  uint32_t *s_tmem = (uint32_t *)(bar + 1);
  const int t = threadIdx.x, warp = t >> 5;
  for (int i = t; i < 128 * 8; i += 128)
    *reinterpret_cast<uint4 *>(sA + swz128(i >> 3, i & 7)) = reinterpret_cast<const uint4 *>(a)[i];
  for (int i = t; i < 64 * 8; i += 128)
    *reinterpret_cast<uint4 *>(sB + swz128(i >> 3, i & 7)) = reinterpret_cast<const uint4 *>(b)[i];
  fence_proxy_async_smem();
  if (t == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane = tmem + ((uint32_t)(warp * 32) << 16);
  for (int h = 0; h < 2; ++h) {
    uint32_t r[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(d0[t * 64 + h * 32 + e]);
    tmem_st32(lane + h * 32, r);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    if (elect_one()) {
      constexpr uint32_t idesc = instr_desc(kFmtF32, kFmtE4M3, kFmtE4M3, 64, 128);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f8(tmem, smem_desc(smem_u32(sA) + kk * 32, 1024, kSwizzle128),
               smem_desc(smem_u32(sB) + kk * 32, 1024, kSwizzle128), idesc, 1);
      mma_commit(bar);
    }
    __syncwarp();
  }
  volatile int no_abort = 0;
  const bool ok = mbar_wait(bar, 0, status, 1, &no_abort, 2000000000LL);
  tc_fence_after();
  if (__all_sync(0xffffffffu, ok)) {
    for (int h = 0; h < 2; ++h) {
      uint32_t r[32];
      tmem_ld32(lane + h * 32, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) out[t * 64 + h * 32 + e] = __uint_as_float(r[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}
}  // namespace

// a: 128 x 128 E4M3 bytes, b: 64 x 128, d0 and out: 128 x 64 fp32 (row major,
// device pointers), status: int[2] zeroed by the caller.  Returns the launch error.
extern "C" int acc_probe(const void *a, const void *b, const void *d0, void *out, void *status) {
  const int smem = 1024 + 128 * 128 + 64 * 128 + 64;
  acc_probe_kernel<<<1, 128, smem>>>((const uint8_t *)a, (const uint8_t *)b, (const float *)d0, (float *)out,
                                     (int *)status);
  return (int)cudaGetLastError();
}
