// SageBwd backward on sm_103a (SageAttention3 summary, "SageBwd Backward Pass
// and the Critical dOV^T Decision", eq. 8 and Algorithm 3).
//
// Per (query block i of 128 rows, key block j of 64 keys), with S recomputed
// from the forward's INT8 codes and the row statistics the forward wrote:
//   S_ij  = delta_Q,i delta_K,j Q^_i K^_j^T (+ dS_ij = q_bar_i deq(K^_j)^T)
//   P_ij  = exp(S_ij sm_scale - lse_i)
//   P^_ij = rint(P_ij / s_P), s_P = max(P_ij) / 127      (INT8 per tile)
//   dV_j += P^_ij^T dO^_i s_P s_dO,i                       (dO^ INT8 per block)
//   dP_ij = dO_i V_j^T                                     (16-bit operands)
//   dS_ij = P_ij o (dP_ij - D_i),  D_i = rowsum(dO_i o O_i)
//   dS^_ij = rint(dS_ij / s_dS), s_dS = max|dS_ij| / 127  (INT8 per tile)
//   dQ_i += dS^_ij K^_j s_dS delta_K,j + rowsum(dS_ij) k_bar^T
//   dK_j += dS^_ij^T Q^_i s_dS delta_Q,i (+ colsum(dS_ij) q_bar_i^T)
//   dQ, dK times sm_scale.
// The smoothing corrections take the unquantized dS; rowsum and colsum are
// exact sums of the fp32 values the thread holds.
//
// GB300 mapping: two kernels, so that every gradient is a plain sum without
// atomics (deterministic).  Both keep 128 tokens per TMEM lane group and run
// four INT8-code products on the tensor core as kind::f16 on codes held as
// exact fp16 integers (sm_103a has no INT8 tensor path) and dO V^T as
// kind::f16 on the bf16 inputs:
//   bwd_dkdv_kernel  one CTA per (batch, kv-head, 128 keys = two 64-key
//                    blocks): for every query head of the group and every
//                    query block with a visible pair, S^T = K^ Q^T and
//                    dP^T = V dO^T (keys in TMEM lanes), P^T and dS^T per key
//                    row, then R_V = P^^T dO^ and R_K = dS^^T Q^ (the token
//                    operand read MN-major out of the same tiles) added into
//                    fp32 accumulators in TMEM with the tile's scales;
//   bwd_dq_kernel    one CTA per (batch, q-head, query block): for every key
//                    block, S = Q^ K^T and dP = dO V^T (queries in lanes), dS
//                    per query row, then R = dS^ K^ per 64-key half (K^ read
//                    MN-major) added into an fp32 accumulator in TMEM.
// Warps: 0-3 the token rows (one per thread, its TMEM lane), 4 the TMA
// producer, 5 the MMA issuer.  TMEM: S (or S^T) in columns 0-127, dP in
// 128-255 (each tile's products R overwrite them once they are read),
// accumulators from column 256.  The P / dS tile maxima are the one
// cross-thread step (a warp shuffle and a shared-memory exchange).
// Waits are bounded as in the forward kernels; on timeout the CTA drains its
// own copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.h"
#include "launch.h"
#include "sm103.cuh"

namespace sage {
namespace {

constexpr int kBwdThreads = 192;
constexpr int kBwdProducer = 4, kBwdMma = 5;
constexpr int kBarRows = 1;  // named barrier of the four row warps
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int CH = D / 64;            // 128-byte chunks of a 16-bit d row
  static constexpr int T128 = 128 * D * 2;     // a 128-row tile of 16-bit values
  static constexpr int PT = 128 * 128 * 2;     // a 128 x 128 tile of fp16 codes (two chunks)
  static constexpr int CHUNK = 128 * 128;      // bytes of one 128-byte chunk of 128 rows
  static constexpr int C_S = 0, C_DP = 128, C_ACC = 256;
  static constexpr uint32_t ID_F16 = instr_desc(kFmtF32, kFmtF16, kFmtF16, 128, 128);
  static constexpr uint32_t ID_BF16 = instr_desc(kFmtF32, 1, 1, 128, 128);
  // R = A (K-major codes) x B (the token operand, MN-major): transpose-B bit 16
  static constexpr uint32_t ID_MN = instr_desc(kFmtF32, kFmtF16, kFmtF16, D, 128) | (1u << 16);
};

struct BwdParams {
  int N, M, N_pad, M_pad, Tm, Tn, Hq, Hkv, causal, smooth_q;
  float sm_scale, sm_log2;
  const float *dq, *qbar, *dk, *kbar, *lse, *dos, *drow;
  float *gdq, *gdk, *gdv;
  int *status;
  long long spin;
};

// byte offset of 16-byte piece c16 of row r inside one 128-byte-swizzled chunk
__device__ __forceinline__ uint32_t swz(int r, int c16) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c16 ^ (r & 7)) << 4));
}

// D[128 x 128] (+)= A B^T with A and B K-major 128-row tiles over K = kd
// elements of 16 bits (kd / 64 chunks of 128 rows x 128 bytes)
__device__ __forceinline__ void mma_kmajor(uint32_t d_tmem, uint32_t a_base, uint32_t b_base, int kd, uint32_t idesc) {
  for (int kk = 0; kk < kd / 16; ++kk) {
    const int byte = kk * 32;
    const uint32_t off = (uint32_t)((byte / 128) * (128 * 128) + (byte % 128));
    mma_f16(d_tmem, smem_desc(a_base + off, 1024, kSwizzle128), smem_desc(b_base + off, 1024, kSwizzle128), idesc,
            kk > 0);
  }
}

// D[128 x D] = A B over tokens k0 .. k0 + kn - 1: A a K-major 128 x 128 code
// tile (tokens along K, two chunks), B a 128-token tile of D 16-bit values per
// token read MN-major (8-token groups 1024 bytes apart, 64-value chunks one
// chunk of 128 tokens apart)
template <int D>
__device__ __forceinline__ void mma_tokens(uint32_t d_tmem, uint32_t a_base, uint32_t b_base, int k0, int kn) {
  for (int kk = 0; kk < kn / 16; ++kk) {
    const int k = k0 + kk * 16;
    const uint32_t a = a_base + (uint32_t)((k / 64) * (128 * 128) + (k % 64) * 2);
    uint64_t bd = smem_desc(b_base + (uint32_t)((k / 8) * 1024), 1024, kSwizzle128);
    bd = (bd & ~((uint64_t)0x3FFF << 16)) | ((uint64_t)((128 * 128) >> 4) << 16);
    mma_f16(d_tmem, smem_desc(a, 1024, kSwizzle128), bd, BwdCfg<D>::ID_MN, kk > 0);
  }
}

// q_bar . K^ row r of a K-major fp16 code tile in shared memory (q_bar in shared memory)
template <int D>
__device__ __forceinline__ float qbar_dot_row(const uint8_t *tile, const float *qb, int r) {
  float2 acc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll 4
  for (int p = 0; p < D / 8; ++p) {
    const uint4 w = *reinterpret_cast<const uint4 *>(tile + (p / 8) * (128 * 128) + swz(r, p % 8));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 kv = __half22float2(*reinterpret_cast<const __half2 *>(&ww[e]));
      acc[e & 1] = __ffma2_rn(kv, make_float2(qb[p * 8 + 2 * e], qb[p * 8 + 2 * e + 1]), acc[e & 1]);
    }
  }
  return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// 32 codes rint(x * inv) clamped to +-127 as fp16 values, four 16-byte pieces
__device__ __forceinline__ void codes32(const uint32_t (&x)[32], float inv, uint4 (&out)[4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = fminf(fmaxf(rintf(__uint_as_float(x[u * 8 + 2 * e]) * inv), -127.0f), 127.0f);
      const float b = fminf(fmaxf(rintf(__uint_as_float(x[u * 8 + 2 * e + 1]) * inv), -127.0f), 127.0f);
      const __half2 h = __floats2half2_rn(a, b);
      w[e] = *reinterpret_cast<const uint32_t *>(&h);
    }
    out[u] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------------------- dK, dV
// kSmoothQ: Q smoothing on (its corrections are an instance of their own, so
// the other instance carries none of their code in its loops)
template <int D, bool kSmoothQ>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_doc,
                    const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sK = base, *sV = sK + C::T128, *sQ = sV + C::T128, *sDOC = sQ + C::T128, *sDO = sDOC + C::T128;
  uint8_t *sP = sDO + C::T128, *sDS = sP + C::PT;
  // per query block: lse in base 2, D, q_bar; read only before the tile-maxima
  // barrier, so the next block may overwrite them once every warp is past it
  float *s_lse = (float *)(sDS + C::PT);  // [128]
  float *s_D = s_lse + 128;               // [128]
  float *s_qb = s_D + 128;                // [D]
  float *s_red = s_qb + D;                // [4 warps][2]
  uint64_t *bars = (uint64_t *)(s_red + 8);
  uint64_t *kv_full = bars, *q_full = bars + 1, *do_full = bars + 2, *q_free = bars + 3, *do_free = bars + 4;
  uint64_t *s_full = bars + 5, *r_full = bars + 6, *p_full = bars + 7, *tm_free = bars + 8, *mma_done = bars + 9;
  uint32_t *s_tmem = (uint32_t *)(bars + 10);
  volatile int *s_abort = (volatile int *)(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = p.M_pad / 128;
  const int hk = blockIdx.x / nkb, jb = blockIdx.x % nkb;
  const int b = hk / p.Hkv, g = hk % p.Hkv, G = p.Hq / p.Hkv;
  const int c0 = jb * 128;
  // query blocks with a visible pair: key c is seen by queries q >= c - (M - N)
  int i0 = 0, ni = p.Tm;
  if (p.causal) {
    const int qmin = c0 - (p.M - p.N);
    i0 = qmin <= 0 ? 0 : qmin / 128;
    ni = qmin >= p.N ? 0 : p.Tm - i0;
  }
  const int niter = G * ni;
  int *status = p.status;

  if (threadIdx.x == 0) {
    for (int x = 0; x < 10; ++x) mbar_init(&bars[x], (x == 7 || x == 8) ? 128 : 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kBwdMma) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == kBwdProducer) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_doc);
      tma_prefetch_desc(&tm_do);
      mbar_expect_tx(kv_full, 2 * C::T128);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_load_2d(sK + c * C::CHUNK, &tm_k, kv_full, c * 128, hk * p.M_pad + c0);
        tma_load_2d(sV + c * C::CHUNK, &tm_v, kv_full, c * 128, hk * p.M + c0);
      }
      int n_do = 0, n_q = 0;
      for (int n = 0; n < niter; ++n) {
        const int bh = b * p.Hq + g * G + n / ni, i = i0 + n % ni;
        if (n > 0 && !mbar_wait(do_free, (n - 1) & 1, status, 60, s_abort, p.spin)) break;
        mbar_expect_tx(do_full, C::T128);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) tma_load_2d(sDO + c * C::CHUNK, &tm_do, do_full, c * 128, bh * p.N + i * 128);
        n_do = n + 1;
        if (n > 0 && !mbar_wait(q_free, (n - 1) & 1, status, 61, s_abort, p.spin)) break;
        mbar_expect_tx(q_full, 2 * C::T128);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_2d(sQ + c * C::CHUNK, &tm_q, q_full, c * 128, bh * p.N_pad + i * 128);
          tma_load_2d(sDOC + c * C::CHUNK, &tm_doc, q_full, c * 128, bh * p.N_pad + i * 128);
        }
        n_q = n + 1;
      }
      // every copy this thread issued lands before the CTA leaves
      volatile int no_abort = 0;
      mbar_wait(kv_full, 0, status, 62, &no_abort, kDrainSpin);
      if (n_do > 0) mbar_wait(do_full, (n_do - 1) & 1, status, 62, &no_abort, kDrainSpin);
      if (n_q > 0) mbar_wait(q_full, (n_q - 1) & 1, status, 62, &no_abort, kDrainSpin);
    }
  } else if (warp == kBwdMma) {
    const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), aDOC = smem_u32(sDOC),
                   aDO = smem_u32(sDO), aP = smem_u32(sP), aDS = smem_u32(sDS);
    bool ok = niter == 0 || __all_sync(0xffffffffu, mbar_wait(kv_full, 0, status, 63, s_abort, p.spin));
    for (int n = 0; ok && n < niter; ++n) {
      const bool w = mbar_wait(q_full, n & 1, status, 64, s_abort, p.spin) &&
                     mbar_wait(do_full, n & 1, status, 65, s_abort, p.spin) &&
                     (n == 0 || mbar_wait(tm_free, (n - 1) & 1, status, 66, s_abort, p.spin));
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      if (elect_one()) {
        mma_kmajor(tmem + C::C_S, aK, aQ, D, C::ID_F16);     // S^T = K^ Q^T
        mma_kmajor(tmem + C::C_DP, aV, aDO, D, C::ID_BF16);  // dP^T = V dO^T
        mma_commit(s_full);
        mma_commit(do_free);
      }
      __syncwarp();
      if (!__all_sync(0xffffffffu, mbar_wait(p_full, n & 1, status, 67, s_abort, p.spin))) break;
      tc_fence_after();
      if (elect_one()) {
        mma_tokens<D>(tmem + C::C_S, aP, aDOC, 0, 128);   // R_V = P^^T dO^
        mma_tokens<D>(tmem + C::C_DP, aDS, aQ, 0, 128);   // R_K = dS^^T Q^
        mma_commit(r_full);
        mma_commit(q_free);
      }
      __syncwarp();
    }
    if (elect_one()) mma_commit(mma_done);
    __syncwarp();
    volatile int no_abort = 0;
    mbar_wait(mma_done, 0, status, 68, &no_abort, kDrainSpin);
  } else {
    // ------------------------------------------------------------------ key rows
    const int c = threadIdx.x;  // key c0 + c, TMEM lane c
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int key = c0 + c;
    const bool key_ok = key < p.M;
    const int half = c >> 6;
    const int blk = 2 * jb + half;
    const float dkc = blk < p.Tn ? p.dk[(size_t)hk * p.Tn + blk] : 0.0f;
    const int qlo = key - (p.M - p.N);  // first query that sees this key (causal)
    bool any = false;
    // the K^ tile (read below for dS) has landed
    bool ok = !kSmoothQ || niter == 0 || __all_sync(0xffffffffu, mbar_wait(kv_full, 0, status, 69, s_abort, p.spin));
    // The four row warps meet at named barriers; each barrier also ORs a
    // failure flag, so after a wait that gave up they all leave the loop
    // together (a warp leaving alone would strand the others at a barrier).
    for (int n = 0; n < niter; ++n) {
      const int bh = b * p.Hq + g * G + n / ni, i = i0 + n % ni;
      const float *qbar_i = p.qbar + ((size_t)bh * p.Tm + i) * D;
      {
        const int q = i * 128 + c;
        s_lse[c] = q < p.N ? p.lse[(size_t)bh * p.N_pad + q] * kLog2e : 0.0f;
        s_D[c] = q < p.N ? p.drow[(size_t)bh * p.N_pad + q] : 0.0f;
        if (kSmoothQ && c < D) s_qb[c] = qbar_i[c];
      }
      if (named_bar_any(kBarRows, 128, !ok || *s_abort)) break;
      const float dqs = p.dq[(size_t)bh * p.Tm + i], sdo = p.dos[(size_t)bh * p.Tm + i];
      const float k1 = dqs * dkc * p.sm_log2;
      const float ds2 = kSmoothQ ? qbar_dot_row<D>(sK, s_qb, c) * dkc * p.sm_log2 : 0.0f;
      ok = __all_sync(0xffffffffu, mbar_wait(s_full, n & 1, status, 70, s_abort, p.spin));
      tc_fence_after();
      float pm = 0.0f, sm = 0.0f, cs = 0.0f;
#pragma unroll 1
      for (int ch = 0; ok && ch < 4; ++ch) {
        uint32_t v[32], w[32];
        tmem_ld32(tmem + lane_off + C::C_S + ch * 32, v);
        tmem_ld32(tmem + lane_off + C::C_DP + ch * 32, w);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int q = i * 128 + ch * 32 + e;
          const bool vis = key_ok && q < p.N && (!p.causal || q >= qlo);
          const float t2 = fmaf(__uint_as_float(v[e]), k1, ds2) - s_lse[ch * 32 + e];
          const float pr = vis ? ex2_approx(t2) : 0.0f;
          const float dsv = vis ? pr * (__uint_as_float(w[e]) - s_D[ch * 32 + e]) : 0.0f;
          pm = fmaxf(pm, pr);
          sm = fmaxf(sm, fabsf(dsv));
          cs += dsv;
          v[e] = __float_as_uint(pr);
          w[e] = __float_as_uint(dsv);
        }
        tmem_st32(tmem + lane_off + C::C_S + ch * 32, v);
        tmem_st32(tmem + lane_off + C::C_DP + ch * 32, w);
      }
      tmem_wait_st();
      pm = warp_max(pm);
      sm = warp_max(sm);
      if (lane == 0) {
        s_red[warp * 2] = pm;
        s_red[warp * 2 + 1] = sm;
      }
      if (named_bar_any(kBarRows, 128, !ok)) break;
      // the tile (128 queries x this 64-key block) maxima
      const float Pm = fmaxf(s_red[(2 * half) * 2], s_red[(2 * half + 1) * 2]);
      const float Sm = fmaxf(s_red[(2 * half) * 2 + 1], s_red[(2 * half + 1) * 2 + 1]);
      const float invP = Pm > 0.0f ? 127.0f / Pm : 0.0f, invS = Sm > 0.0f ? 127.0f / Sm : 0.0f;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32];
        uint4 pk[4];
        tmem_ld32(tmem + lane_off + C::C_S + ch * 32, v);
        tmem_wait_ld();
        codes32(v, invP, pk);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4 *>(sP + (ch >> 1) * C::CHUNK + swz(c, (ch & 1) * 4 + u)) = pk[u];
        tmem_ld32(tmem + lane_off + C::C_DP + ch * 32, v);
        tmem_wait_ld();
        codes32(v, invS, pk);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4 *>(sDS + (ch >> 1) * C::CHUNK + swz(c, (ch & 1) * 4 + u)) = pk[u];
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
      // a failed wait here sets the abort flag, which the next iteration's
      // first barrier reads
      ok = __all_sync(0xffffffffu, mbar_wait(r_full, n & 1, status, 71, s_abort, p.spin));
      if (!ok) continue;
      tc_fence_after();
      const float sv = (Pm / 127.0f) * sdo, sk = (Sm / 127.0f) * dqs;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32], a[32];
        tmem_ld32(tmem + lane_off + C::C_S + ch * 32, r);
        if (any) tmem_ld32(tmem + lane_off + C::C_ACC + ch * 32, a);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          a[e] = __float_as_uint(any ? fmaf(__uint_as_float(r[e]), sv, __uint_as_float(a[e]))
                                     : __uint_as_float(r[e]) * sv);
        tmem_st32(tmem + lane_off + C::C_ACC + ch * 32, a);
        tmem_ld32(tmem + lane_off + C::C_DP + ch * 32, r);
        if (any) tmem_ld32(tmem + lane_off + C::C_ACC + D + ch * 32, a);
        tmem_wait_ld();
        // q_bar from global memory here (the shared copy may already hold the next block's)
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 qb4 = kSmoothQ ? __ldg(reinterpret_cast<const float4 *>(qbar_i + ch * 32 + e))
                                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          const float qv[4] = {qb4.x, qb4.y, qb4.z, qb4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
            a[e + u] = __float_as_uint(
                fmaf(__uint_as_float(r[e + u]), sk, (any ? __uint_as_float(a[e + u]) : 0.0f) + cs * qv[u]));
        }
        tmem_st32(tmem + lane_off + C::C_ACC + D + ch * 32, a);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(tm_free);
      any = true;
    }
    // dV = the accumulator, dK = the accumulator times sm_scale (keys < M)
    if (__all_sync(0xffffffffu, !*s_abort)) {
      tc_fence_after();
      float *dv = p.gdv + ((size_t)hk * p.M + key) * D, *dk = p.gdk + ((size_t)hk * p.M + key) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t a[32], k[32];
        if (any) {
          tmem_ld32(tmem + lane_off + C::C_ACC + ch * 32, a);
          tmem_ld32(tmem + lane_off + C::C_ACC + D + ch * 32, k);
          tmem_wait_ld();
        }
        if (key_ok) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float4 x = any ? make_float4(__uint_as_float(a[e]), __uint_as_float(a[e + 1]), __uint_as_float(a[e + 2]),
                                         __uint_as_float(a[e + 3]))
                           : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            float4 y = any ? make_float4(__uint_as_float(k[e]) * p.sm_scale, __uint_as_float(k[e + 1]) * p.sm_scale,
                                         __uint_as_float(k[e + 2]) * p.sm_scale, __uint_as_float(k[e + 3]) * p.sm_scale)
                           : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            *reinterpret_cast<float4 *>(dv + ch * 32 + e) = x;
            *reinterpret_cast<float4 *>(dk + ch * 32 + e) = y;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kBwdMma) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------- dQ
template <int D, bool kSmoothQ>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = base, *sDO = sQ + C::T128, *sK = sDO + C::T128;  // sK[2], then sV[2]
  uint8_t *sV = sK + 2 * C::T128, *sDS = sV + 2 * C::T128;
  float *s_ds = (float *)(sDS + C::PT);  // [2][128] dS of each key in base-2 units
  float *s_qb = s_ds + 256;              // [D]
  float *s_red = s_qb + D;               // [4 warps][2 halves]
  uint64_t *bars = (uint64_t *)(s_red + 8);
  uint64_t *q_full = bars, *kv_full = bars + 1 /*[2]*/, *kv_free = bars + 3 /*[2]*/, *s_full = bars + 5;
  uint64_t *p_full = bars + 6, *r_full = bars + 7, *tm_free = bars + 8, *mma_done = bars + 9;
  uint32_t *s_tmem = (uint32_t *)(bars + 10);
  volatile int *s_abort = (volatile int *)(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x / p.Tm, i = p.Tm - 1 - blockIdx.x % p.Tm;  // longest causal rows first
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int hk = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int last_q = min(p.N, i * 128 + 128) - 1;
  const int nkb = p.M_pad / 128;
  const int nj = p.causal ? min(nkb, (last_q + p.M - p.N) / 128 + 1) : nkb;
  int *status = p.status;

  if (threadIdx.x == 0) {
    for (int x = 0; x < 10; ++x) mbar_init(&bars[x], (x == 6 || x == 8) ? 128 : 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kBwdMma) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  if (kSmoothQ && threadIdx.x < D) s_qb[threadIdx.x] = p.qbar[((size_t)bh * p.Tm + i) * D + threadIdx.x];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == kBwdProducer) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_expect_tx(q_full, 2 * C::T128);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_load_2d(sQ + c * C::CHUNK, &tm_q, q_full, c * 128, bh * p.N_pad + i * 128);
        tma_load_2d(sDO + c * C::CHUNK, &tm_do, q_full, c * 128, bh * p.N + i * 128);
      }
      int issued = 0;
      for (int j = 0; j < nj; ++j) {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(&kv_free[s], ((j - 2) >> 1) & 1, status, 80, s_abort, p.spin)) break;
        mbar_expect_tx(&kv_full[s], 2 * C::T128);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_2d(sK + s * C::T128 + c * C::CHUNK, &tm_k, &kv_full[s], c * 128, hk * p.M_pad + j * 128);
          tma_load_2d(sV + s * C::T128 + c * C::CHUNK, &tm_v, &kv_full[s], c * 128, hk * p.M + j * 128);
        }
        issued = j + 1;
      }
      volatile int no_abort = 0;
      mbar_wait(q_full, 0, status, 81, &no_abort, kDrainSpin);
      for (int j = max(0, issued - 2); j < issued; ++j)
        mbar_wait(&kv_full[j & 1], (j >> 1) & 1, status, 81, &no_abort, kDrainSpin);
    }
  } else if (warp == kBwdMma) {
    const uint32_t aQ = smem_u32(sQ), aDO = smem_u32(sDO), aK = smem_u32(sK), aV = smem_u32(sV), aDS = smem_u32(sDS);
    bool ok = nj == 0 || __all_sync(0xffffffffu, mbar_wait(q_full, 0, status, 82, s_abort, p.spin));
    for (int j = 0; ok && j < nj; ++j) {
      const int s = j & 1;
      const bool w = mbar_wait(&kv_full[s], (j >> 1) & 1, status, 83, s_abort, p.spin) &&
                     (j == 0 || mbar_wait(tm_free, (j - 1) & 1, status, 84, s_abort, p.spin));
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      if (elect_one()) {
        mma_kmajor(tmem + C::C_S, aQ, aK + s * C::T128, D, C::ID_F16);    // S = Q^ K^T
        mma_kmajor(tmem + C::C_DP, aDO, aV + s * C::T128, D, C::ID_BF16); // dP = dO V^T
        mma_commit(s_full);
      }
      __syncwarp();
      if (!__all_sync(0xffffffffu, mbar_wait(p_full, j & 1, status, 85, s_abort, p.spin))) break;
      tc_fence_after();
      if (elect_one()) {
        mma_tokens<D>(tmem + C::C_S, aDS, aK + s * C::T128, 0, 64);    // R0 = dS^[:, 0:64] K^[0:64]
        mma_tokens<D>(tmem + C::C_DP, aDS, aK + s * C::T128, 64, 64);  // R1 = dS^[:, 64:128] K^[64:128]
        mma_commit(r_full);
        mma_commit(&kv_free[s]);
      }
      __syncwarp();
    }
    if (elect_one()) mma_commit(mma_done);
    __syncwarp();
    volatile int no_abort = 0;
    mbar_wait(mma_done, 0, status, 86, &no_abort, kDrainSpin);
  } else {
    // ------------------------------------------------------------------ query rows
    const int r = threadIdx.x;  // query i*128 + r, TMEM lane r
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int q = i * 128 + r;
    const bool q_ok = q < p.N;
    const float lse2 = q_ok ? p.lse[(size_t)bh * p.N_pad + q] * kLog2e : 0.0f;
    const float Dq = q_ok ? p.drow[(size_t)bh * p.N_pad + q] : 0.0f;
    const float dqs = p.dq[(size_t)bh * p.Tm + i];
    const int diag = q + p.M - p.N;  // last key this query sees (causal)
    float rs = 0.0f;                 // rowsum of dS over every key
    bool any = false, ok = true;
    // named barriers OR a failure flag so that the four row warps leave together
    for (int j = 0; j < nj; ++j) {
      const int s = j & 1;
      const float dk0 = p.dk[(size_t)hk * p.Tn + 2 * j];
      const float dk1 = 2 * j + 1 < p.Tn ? p.dk[(size_t)hk * p.Tn + 2 * j + 1] : 0.0f;
      if (kSmoothQ) {
        // dS of key r of the tile, shared with every row through shared memory
        ok = __all_sync(0xffffffffu, mbar_wait(&kv_full[s], (j >> 1) & 1, status, 90, s_abort, p.spin));
        if (ok) s_ds[s * 128 + r] = qbar_dot_row<D>(sK + s * C::T128, s_qb, r) * (r < 64 ? dk0 : dk1) * p.sm_log2;
        if (named_bar_any(kBarRows, 128, !ok)) break;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(s_full, j & 1, status, 91, s_abort, p.spin));
      tc_fence_after();
      float m0 = 0.0f, m1 = 0.0f;
#pragma unroll 1
      for (int ch = 0; ok && ch < 4; ++ch) {
        uint32_t v[32], w[32];
        tmem_ld32(tmem + lane_off + C::C_S + ch * 32, v);
        tmem_ld32(tmem + lane_off + C::C_DP + ch * 32, w);
        tmem_wait_ld();
        const float k1 = dqs * (ch < 2 ? dk0 : dk1) * p.sm_log2;
        float mx = 0.0f;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int key = j * 128 + ch * 32 + e;
          const bool vis = q_ok && key < p.M && (!p.causal || key <= diag);
          const float ds2 = kSmoothQ ? s_ds[s * 128 + ch * 32 + e] : 0.0f;
          const float pr = vis ? ex2_approx(fmaf(__uint_as_float(v[e]), k1, ds2) - lse2) : 0.0f;
          const float dsv = vis ? pr * (__uint_as_float(w[e]) - Dq) : 0.0f;
          rs += dsv;
          mx = fmaxf(mx, fabsf(dsv));
          w[e] = __float_as_uint(dsv);
        }
        if (ch < 2)
          m0 = fmaxf(m0, mx);
        else
          m1 = fmaxf(m1, mx);
        tmem_st32(tmem + lane_off + C::C_DP + ch * 32, w);
      }
      tmem_wait_st();
      m0 = warp_max(m0);
      m1 = warp_max(m1);
      if (lane == 0) {
        s_red[warp * 2] = m0;
        s_red[warp * 2 + 1] = m1;
      }
      if (named_bar_any(kBarRows, 128, !ok)) break;
      const float M0 = fmaxf(fmaxf(s_red[0], s_red[2]), fmaxf(s_red[4], s_red[6]));
      const float M1 = fmaxf(fmaxf(s_red[1], s_red[3]), fmaxf(s_red[5], s_red[7]));
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32];
        uint4 pk[4];
        tmem_ld32(tmem + lane_off + C::C_DP + ch * 32, v);
        tmem_wait_ld();
        const float mm = ch < 2 ? M0 : M1;
        codes32(v, mm > 0.0f ? 127.0f / mm : 0.0f, pk);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4 *>(sDS + (ch >> 1) * C::CHUNK + swz(r, (ch & 1) * 4 + u)) = pk[u];
      }
      // K^ rows past the last key are layout padding the pre-pass need not
      // write (its key blocks end at ceil(M / 64) * 64): zero them before
      // dS^ K^ reads them, since a zero code times a non-finite bit pattern
      // would not be zero (thread r takes row r of the tile)
      if (j * 128 + r >= p.M) {
#pragma unroll
        for (int c16 = 0; c16 < D / 8; ++c16)
          *reinterpret_cast<uint4 *>(sK + s * C::T128 + (c16 / 8) * C::CHUNK + swz(r, c16 % 8)) =
              make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
      // a failed wait sets the abort flag: the next tile's first wait fails
      // too and its barrier takes every warp out
      ok = __all_sync(0xffffffffu, mbar_wait(r_full, j & 1, status, 92, s_abort, p.spin));
      if (!ok) continue;
      tc_fence_after();
      const float sc0 = (M0 / 127.0f) * dk0, sc1 = (M1 / 127.0f) * dk1;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r0[32], r1[32], a[32];
        tmem_ld32(tmem + lane_off + C::C_S + ch * 32, r0);
        tmem_ld32(tmem + lane_off + C::C_DP + ch * 32, r1);
        if (any) tmem_ld32(tmem + lane_off + C::C_ACC + ch * 32, a);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          a[e] = __float_as_uint(fmaf(__uint_as_float(r0[e]), sc0,
                                      fmaf(__uint_as_float(r1[e]), sc1, any ? __uint_as_float(a[e]) : 0.0f)));
        tmem_st32(tmem + lane_off + C::C_ACC + ch * 32, a);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(tm_free);
      any = true;
      // s_red and s_ds[s] are rewritten only after the next tile's barriers
      // (every warp has passed this tile's reads by then)
    }
    // dQ = (accumulator + rowsum(dS) k_bar) * sm_scale
    if (__all_sync(0xffffffffu, !*s_abort)) {
      tc_fence_after();
      const float *kb = p.kbar + (size_t)hk * D;
      float *dst = p.gdq + ((size_t)bh * p.N + q) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t a[32];
        if (any) {
          tmem_ld32(tmem + lane_off + C::C_ACC + ch * 32, a);
          tmem_wait_ld();
        }
        if (q_ok) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 kv = __ldg(reinterpret_cast<const float4 *>(kb + ch * 32 + e));
            float4 x;
            x.x = ((any ? __uint_as_float(a[e]) : 0.0f) + rs * kv.x) * p.sm_scale;
            x.y = ((any ? __uint_as_float(a[e + 1]) : 0.0f) + rs * kv.y) * p.sm_scale;
            x.z = ((any ? __uint_as_float(a[e + 2]) : 0.0f) + rs * kv.z) * p.sm_scale;
            x.w = ((any ? __uint_as_float(a[e + 3]) : 0.0f) + rs * kv.w) * p.sm_scale;
            *reinterpret_cast<float4 *>(dst + ch * 32 + e) = x;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kBwdMma) tmem_dealloc(tmem, 512);
}

template <int D>
sage_status launch_bwd_t(const sage_shape &s, int causal, float sm_scale, int flags, const void *ws,
                         const sage_ws_layout &L, const void *v, const void *dout, float *dq, float *dk, float *dv,
                         cudaStream_t stream) {
  using C = BwdCfg<D>;
  const char *w = (const char *)ws;
  CUtensorMap tk, tv, tq, tdoc, tdo;
  sage_status st;
  const uint64_t rowb = (uint64_t)D * 2;
  if ((st = make_tmap_2d(&tk, w + L.khat, rowb, (uint64_t)s.B * s.Hkv * L.M_pad, rowb, 128, 128, 128)) != SAGE_OK)
    return st;
  if ((st = make_tmap_2d(&tv, v, rowb, (uint64_t)s.B * s.Hkv * s.M, rowb, 128, 128, 128)) != SAGE_OK) return st;
  if ((st = make_tmap_2d(&tq, w + L.qhat, rowb, (uint64_t)s.B * s.Hq * L.N_pad, rowb, 128, 128, 128)) != SAGE_OK)
    return st;
  if ((st = make_tmap_2d(&tdoc, w + L.doc, rowb, (uint64_t)s.B * s.Hq * L.N_pad, rowb, 128, 128, 128)) != SAGE_OK)
    return st;
  if ((st = make_tmap_2d(&tdo, dout, rowb, (uint64_t)s.B * s.Hq * s.N, rowb, 128, 128, 128)) != SAGE_OK) return st;
  BwdParams p;
  p.N = s.N;
  p.M = s.M;
  p.N_pad = L.N_pad;
  p.M_pad = L.M_pad;
  p.Tm = L.Tm;
  p.Tn = L.Tn;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.causal = causal ? 1 : 0;
  p.smooth_q = (flags & SAGE_SMOOTH_Q) ? 1 : 0;
  p.sm_scale = sm_scale;
  p.sm_log2 = sm_scale * 1.4426950408889634f;
  p.dq = (const float *)(w + L.dq);
  p.qbar = (const float *)(w + L.qbar);
  p.dk = (const float *)(w + L.dk);
  p.kbar = (const float *)(w + L.kbar);
  p.lse = (const float *)(w + L.lse);
  p.dos = (const float *)(w + L.dos);
  p.drow = (const float *)(w + L.drow);
  p.gdq = dq;
  p.gdk = dk;
  p.gdv = dv;
  p.status = (int *)(w + L.status);
  p.spin = spin_limit_cycles();
  const int smem_a = 1024 + 5 * C::T128 + 2 * C::PT + (256 + D + 8) * 4 + 128;
  const int smem_b = 1024 + 6 * C::T128 + C::PT + (256 + D + 8) * 4 + 128;
  auto ka = p.smooth_q ? bwd_dkdv_kernel<D, true> : bwd_dkdv_kernel<D, false>;
  auto kb = p.smooth_q ? bwd_dq_kernel<D, true> : bwd_dq_kernel<D, false>;
  if (cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_a) != cudaSuccess ||
      cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_b) != cudaSuccess)
    return SAGE_ERR_CUDA;
  const unsigned ga = (unsigned)(s.B * s.Hkv * (L.M_pad / 128)), gb = (unsigned)(s.B * s.Hq * L.Tm);
  ka<<<ga, kBwdThreads, smem_a, stream>>>(tk, tv, tq, tdoc, tdo, p);
  if (cudaGetLastError() != cudaSuccess) return SAGE_ERR_CUDA;
  kb<<<gb, kBwdThreads, smem_b, stream>>>(tk, tv, tq, tdo, p);
  return cudaGetLastError() == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}

}  // namespace

sage_status launch_attn_bwd(const sage_shape &s, int causal, float sm_scale, int flags, const void *ws,
                            const sage_ws_layout &L, const void *v, const void *dout, float *dq, float *dk, float *dv,
                            cudaStream_t stream) {
  return s.d == 64 ? launch_bwd_t<64>(s, causal, sm_scale, flags, ws, L, v, dout, dq, dk, dv, stream)
                   : launch_bwd_t<128>(s, causal, sm_scale, flags, ws, L, v, dout, dq, dk, dv, stream);
}

}  // namespace sage
