// Operand-layout probe for the backward's MMAs on sm_103a: D = A B with A
// K-major (128 rows x K fp16, 128-byte swizzled rows, in 64-element chunks)
// and B given MN-major, i.e. stored as K rows of N contiguous fp16 values in
// the same 128-byte swizzled chunks a K-major tile of those rows would use
// (how a [keys][d] tile loaded by TMA looks when the MMA reduces over keys).
// The descriptor of such a B: the 8-row groups along K are 1024 bytes apart
// (stride field) and the 64-element chunks along N are one chunk apart
// (leading field), transpose-B set in the instruction descriptor.
// Test code: one CTA of 128 threads, every wait bounded; the tiles sit at the
// start of a shared-memory block four times their size, so any stride read
// past them stays inside the block.
#include <stdint.h>

#include "sm103.cuh"

using namespace sage;

namespace {
constexpr int kRows = 128;                 // rows of A, K rows of B
constexpr int kTileBytes = kRows * 256;    // 128 rows x 128 fp16 (two 128-byte chunks)

__device__ __forceinline__ uint32_t swz128(int r, int c16) {  // 16-byte chunk c16 of row r in one chunk
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c16 ^ (r & 7)) << 4));
}

// global row-major [128][128] fp16 -> two swizzled 64-column chunks
__device__ void stage(uint8_t *dst, const uint16_t *src, int t) {
  for (int i = t; i < kRows * 16; i += 128) {
    const int r = i >> 4, c16 = i & 15;  // 16 sixteen-byte pieces per 256-byte row
    const int chunk = c16 >> 3;
    *reinterpret_cast<uint4 *>(dst + chunk * (kRows * 128) + swz128(r, c16 & 7)) =
        reinterpret_cast<const uint4 *>(src)[i];
  }
}

// mode 0: D[128 x 128] = A[:, 0:128] B[0:128, :]  (K = 128: both A chunks, all B rows)
// mode 1: D[128 x 128] = A[:, 64:128] B[64:128, :] (K = 64: A's second chunk, B rows 64..127)
// mode 2: D[128 x 64]  = A[:, 0:64] B[0:64, 0:64]  (N = 64: one chunk of B)
__global__ void __launch_bounds__(128, 1) mn_probe_kernel(const uint16_t *a, const uint16_t *b, float *out, int mode,
                                                          int *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sA = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sB = sA + kTileBytes;
  uint64_t *bar = (uint64_t *)(sB + 3 * kTileBytes);  // after a guard of two tiles
  uint32_t *s_tmem = (uint32_t *)(bar + 1);
  const int t = threadIdx.x, warp = t >> 5;
  for (int i = t; i < 3 * kTileBytes / 16; i += 128) reinterpret_cast<uint4 *>(sB)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  stage(sA, a, t);
  stage(sB, b, t);
  fence_proxy_async_smem();
  if (t == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int n = mode == 2 ? 64 : 128;
  if (warp == 0) {
    if (elect_one()) {
      // kind::f16, f16 x f16 -> f32, B transposed (MN-major): bit 16
      const uint32_t idesc = instr_desc(kFmtF32, kFmtF16, kFmtF16, n, 128) | (1u << 16);
      const int k0 = mode == 1 ? 64 : 0, kn = mode == 0 ? 128 : 64;
      for (int kk = 0; kk < kn / 16; ++kk) {
        const int k = k0 + kk * 16;
        // A: K-major, chunk k / 64, 32 bytes per 16-element step inside the 128-byte row
        const uint32_t aa = smem_u32(sA) + (k / 64) * (kRows * 128) + (k % 64) * 2;
        // B: MN-major, K rows k..k+15 = two 8-row groups starting at group k / 8
        const uint32_t ba = smem_u32(sB) + (k / 8) * 1024;
        uint64_t bd = smem_desc(ba, 1024, kSwizzle128);
        bd = (bd & ~((uint64_t)0x3FFF << 16)) | ((uint64_t)((kRows * 128) >> 4) << 16);  // chunk stride along N
        mma_f16(tmem, smem_desc(aa, 1024, kSwizzle128), bd, idesc, kk > 0);
      }
      mma_commit(bar);
    }
    __syncwarp();
  }
  volatile int no_abort = 0;
  const bool ok = mbar_wait(bar, 0, status, 1, &no_abort, 2000000000LL);
  tc_fence_after();
  if (__all_sync(0xffffffffu, ok)) {
    const uint32_t lane = tmem + ((uint32_t)(warp * 32) << 16);
    for (int h = 0; h < n / 32; ++h) {
      uint32_t r[32];
      tmem_ld32(lane + h * 32, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) out[t * 128 + h * 32 + e] = __uint_as_float(r[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}
}  // namespace

// a, b: [128][128] fp16 row major (device); out: [128][128] fp32 (device);
// status: int[2] zeroed by the caller.  Returns the launch error.
extern "C" int mn_probe(const void *a, const void *b, void *out, int mode, void *status) {
  const int smem = 1024 + 4 * kTileBytes + 64;
  if (cudaFuncSetAttribute(mn_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -1;
  mn_probe_kernel<<<1, 128, smem>>>((const uint16_t *)a, (const uint16_t *)b, (float *)out, mode, (int *)status);
  return (int)cudaGetLastError();
}
