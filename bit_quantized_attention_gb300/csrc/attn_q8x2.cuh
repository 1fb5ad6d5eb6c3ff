#pragma once
// Fused quantized attention for the INT8 / FP8 modes on sm_103a at head dim
// 64 with two query blocks per work item (the kernel template and its
// launcher; attn_q8x2_64.cu instantiates it).
//
// What it computes is what attn_q8.cuh computes, row by row and tile by tile
// (SageAttention2 Technical Report summary §3.4 "The Complete Algorithm";
// "Quantization for Attention, in depth", "The datapath and its quantize
// points"):
//   S_ij  = delta_Q delta_K,j (Q^_i K^_j^T) + dS_ij,  dS_ij = q_bar_i deq(K^_j)^T
//   m_ij  = max(m_i,j-1, rowmax S_ij sm_scale)
//   P~_ij = exp(S_ij sm_scale - m_ij),  l_ij = e^(m_i,j-1 - m_ij) l + rowsum P~
//   P^_ij = e4m3(448 P~_ij)                          (static scale 1/448)
//   R_ij  = P^_ij V^_j        (tile partial, a fresh accumulator per key tile)
//   O_ij  = e^(m_i,j-1 - m_ij) O_i,j-1 + R_ij        (FP32 running output)
//   O_i   = O / l * delta_V / 448 (+ V_m)
// in base 2 with the 448 folded into the exponent, so l carries 448 sum P~.
//
// GB300 mapping.  A persistent CTA per SM walks work items of two 128-row
// query blocks of one head (longest causal rows first, round robin); both
// blocks share every K^ / V^ tile of 64 keys the producer loads.  Each of the
// two softmax warpgroups owns one query block: one row per thread (its TMEM
// lane), all 64 keys of a tile, the row maximum, the exponentials and P^ into
// the swizzled K-major A operand of P^V^ in shared memory; then it folds the
// previous tile's partial into its row of O, held in registers (O = alpha O +
// R), and at the item's end writes the output.  Nothing passes between the
// two softmax warpgroups, so the tensor core works on one block's products
// while the other block's softmax runs, and each thread waits on TMEM twice
// per tile (S, then R).
//   warps 0-3 / 4-7  softmax, P^, accumulation, epilogue of query block 0 / 1
//   warps 8-11       Q smoothing only: dS of each key tile on CUDA cores
//                    (thread c takes key c of one block), published through
//                    shared memory ahead of the softmax
//   warp 12          TMA producer: Q^ pairs, K^ tiles, V^T tiles
//   warp 13          MMA issuer: S = Q^ K^T (kind::f16 on INT8 codes held as
//                    exact fp16 integers -- sm_103a has no INT8 tensor path --
//                    or kind::f8f6f4 on E4M3 codes) one tile ahead, then
//                    R = P^ V^ (kind::f8f6f4)
// TMEM: three 64-column S/R regions per query block (R of a tile overwrites
// its S once the softmax has read S), so S runs up to two tiles ahead of the
// accumulation.  Every barrier's producer can run at most one phase ahead of
// its waiters (per-region and per-buffer barriers).  Waits are bounded: on
// timeout the kernel records SAGE_ERR_TIMEOUT and the site, drains its own TMA
// loads and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.h"
#include "launch.h"
#include "sm103.cuh"

namespace sage {
namespace {

constexpr int kX2Threads = 512;
constexpr int kX2DsWarp0 = 8, kX2Producer = 12, kX2Mma = 13;
constexpr int kX2LaunchRegs = 128, kX2SoftRegs = 168, kX2DsRegs = 96, kX2CtlRegs = 56;
static_assert(128 * (2 * kX2SoftRegs + kX2DsRegs + kX2CtlRegs) <= kX2Threads * kX2LaunchRegs, "register split");
static_assert(kX2SoftRegs >= kX2LaunchRegs && kX2DsRegs <= kX2LaunchRegs && kX2CtlRegs <= kX2LaunchRegs,
              "register split directions");
constexpr float kX2Log2_448 = 8.807354922057604f;
constexpr int kX2NB = 3;  // S/R regions per query block

template <bool kQK16, bool kSmoothQ>
struct X2Cfg {
  static constexpr int D = 64;
  static constexpr int BK = 64;                        // keys per tile (= K scale block)
  static constexpr int QK_EB = kQK16 ? 2 : 1;
  static constexpr int ROWB = D * QK_EB;               // bytes per Q / K row: 128 or 64
  static constexpr int QK_SW = ROWB;                   // one swizzle span per row
  static constexpr int QK_LAYOUT = QK_SW == 128 ? kSwizzle128 : kSwizzle64;
  static constexpr int Q_TILE = 128 * ROWB;
  static constexpr int QB = 2;                         // Q pair buffers
  static constexpr int K_BYTES = BK * ROWB;
  static constexpr int V_BYTES = D * BK;               // V^T tile: D rows of 64 tokens, E4M3
  static constexpr int P_TILE = 128 * BK;              // P^ tile: 128 rows of 64 keys, E4M3
  static constexpr int PB = 2;                         // P^ buffers per query block
  static constexpr int FIXED = QB * 2 * Q_TILE + 2 * PB * P_TILE;
  static constexpr int NFLOAT = kSmoothQ ? (2 * 2 * BK + 2 * 2 * D) : 0;  // s_ds[2][2][BK], s_qb[2][2][D]
  static constexpr int MISC = NFLOAT * 4 + 768;
  static constexpr int BUDGET = 225 * 1024 - 1024 - FIXED - MISC;
  static constexpr int ST_FIT = BUDGET / (K_BYTES + V_BYTES);
  static constexpr int ST = ST_FIT > 6 ? 6 : ST_FIT;  // K and V ring stages
  static_assert(ST >= 3, "shared memory budget");
  static constexpr int SMEM_TOTAL = 1024 + FIXED + ST * (K_BYTES + V_BYTES) + MISC;
  static constexpr int TMEM_COLS = 512;
  static_assert(2 * kX2NB * 64 <= TMEM_COLS, "TMEM columns");
  static constexpr uint32_t IDESC_QK =
      instr_desc(kFmtF32, kQK16 ? kFmtF16 : kFmtE4M3, kQK16 ? kFmtF16 : kFmtE4M3, BK, 128);
  static constexpr uint32_t IDESC_PV = instr_desc(kFmtF32, kFmtE4M3, kFmtE4M3, D, 128);
  static constexpr int QK_KSTEPS = ROWB / 32;
  static constexpr int PV_KSTEPS = BK / 32;
};

struct X2Params {
  int N, M, N_pad, M_pad, Tm, Tn, Tp, Hq, Hkv, causal, flags;
  int items;      // B * Hq * Tp
  float sm_log2;  // sm_scale * log2(e)
  const float *dq, *dqt, *qbar, *dk, *dv, *vm;
  __nv_bfloat16 *o;
  int *status;
  long long spin;
  int stall;  // test hook: the MMA issuer first waits on a barrier nothing arrives on
};

// byte offset of 16-byte chunk c of row r in a K-major tile of SW-byte rows
template <int SW>
__device__ __forceinline__ uint32_t x2_swz(int r, int c) {
  const int x = (SW == 128) ? (r & 7) : ((r & 7) >> 1);
  return (uint32_t)((r >> 3) * (8 * SW) + (r & 7) * SW + ((c ^ x) << 4));
}

// Work item idx: query blocks 2p and 2p + 1 of head bh (longest causal rows
// first, heads interleaved; non-causal: head-major); T key tiles of 64,
// enough for the item's last valid row.
struct X2Item {
  int bh, p, hkv, T;
};
__device__ __forceinline__ X2Item x2_item(const X2Params &q, int idx) {
  X2Item it;
  const int BH = q.items / q.Tp;
  if (q.causal) {  // longest rows first, heads interleaved
    it.p = q.Tp - 1 - idx / BH;
    it.bh = idx % BH;
  } else {  // head-major: the CTAs in flight share a head's K / V tiles in L2
    it.p = idx % q.Tp;
    it.bh = idx / q.Tp;
  }
  const int b = it.bh / q.Hq, h = it.bh % q.Hq;
  it.hkv = b * q.Hkv + h / (q.Hq / q.Hkv);
  const int last_row = min(q.N, it.p * 256 + 256) - 1;
  it.T = q.causal ? min(q.Tn, (last_row + q.M - q.N) / 64 + 1) : q.Tn;
  return it;
}

// sum_d q_bar[d] K^[r, d] for key r of a K^ tile in shared memory (the codes
// are exact in fp16 / E4M3; q_bar in shared memory, every lane the same word)
template <bool kQK16>
__device__ __forceinline__ float x2_qbar_dot(const uint8_t *kt, const float *qbar, int r) {
  using C = X2Cfg<kQK16, true>;
  float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                   make_float2(0.0f, 0.0f)};
#pragma unroll 2
  for (int k = 0; k < C::ROWB / 16; ++k) {
    const uint4 w = *reinterpret_cast<const uint4 *>(kt + x2_swz<C::QK_SW>(r, k));
    const int d0 = k * 16 / C::QK_EB;
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    if (kQK16) {
      const float4 qa = *reinterpret_cast<const float4 *>(qbar + d0);
      const float4 qb = *reinterpret_cast<const float4 *>(qbar + d0 + 4);
      const float2 q2[4] = {make_float2(qa.x, qa.y), make_float2(qa.z, qa.w), make_float2(qb.x, qb.y),
                            make_float2(qb.z, qb.w)};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        acc[e] = __ffma2_rn(__half22float2(*reinterpret_cast<const __half2 *>(&ww[e])), q2[e], acc[e]);
    } else {
#pragma unroll
      for (int e4 = 0; e4 < 4; ++e4) {
        const float4 q = *reinterpret_cast<const float4 *>(qbar + d0 + 4 * e4);
        const uint32_t lo = cvt_e4m3x2_to_f16x2((uint16_t)(ww[e4] & 0xffffu));
        const uint32_t hi = cvt_e4m3x2_to_f16x2((uint16_t)(ww[e4] >> 16));
        acc[e4] = __ffma2_rn(__half22float2(*reinterpret_cast<const __half2 *>(&lo)), make_float2(q.x, q.y), acc[e4]);
        acc[e4] = __ffma2_rn(__half22float2(*reinterpret_cast<const __half2 *>(&hi)), make_float2(q.z, q.w), acc[e4]);
      }
    }
  }
  return ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
}

template <bool kQK16, bool kSmoothQ>
__global__ void __launch_bounds__(kX2Threads, 1)
    attn_q8x2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const X2Params p) {
  using C = X2Cfg<kQK16, kSmoothQ>;
  constexpr int ST = C::ST, QB = C::QB, PB = C::PB, BK = C::BK, D = C::D, NB = kX2NB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = base;                        // [QB][2 blocks]
  uint8_t *sP = sQ + QB * 2 * C::Q_TILE;      // [2 blocks][PB]
  uint8_t *sK = sP + 2 * PB * C::P_TILE;      // [ST]
  uint8_t *sV = sK + ST * C::K_BYTES;         // [ST]
  float *s_ds = (float *)(sV + ST * C::V_BYTES);  // [2 tile parities][2 blocks][BK] dS in t units
  float *s_qb = s_ds + (kSmoothQ ? 4 * BK : 0);   // [2 item parities][2 blocks][D]
  uint64_t *bars = (uint64_t *)(((uintptr_t)(s_qb + (kSmoothQ ? 4 * D : 0)) + 7) & ~(uintptr_t)7);
  uint64_t *q_full = bars;               // [QB]
  uint64_t *q_empty = q_full + QB;       // [QB]
  uint64_t *k_full = q_empty + QB;       // [ST]
  uint64_t *k_empty = k_full + ST;       // [ST]
  uint64_t *v_full = k_empty + ST;       // [ST]
  uint64_t *v_empty = v_full + ST;       // [ST]
  uint64_t *s_full = v_empty + ST;       // [2 blocks][NB] S of the region's tile in TMEM
  uint64_t *r_full = s_full + 2 * NB;    // [2][NB] R of the region's tile in TMEM
  uint64_t *sr_free = r_full + 2 * NB;   // [2][NB] R folded: the region is free
  uint64_t *p_full = sr_free + 2 * NB;   // [2][PB] P^ written
  uint64_t *p_empty = p_full + 2 * PB;   // [2][PB] P^ read by its MMA
  uint64_t *ds_full = p_empty + 2 * PB;  // [2 tile parities] dS in shared memory
  uint64_t *ds_free = ds_full + 2;       // [2] read by both softmax warpgroups
  uint64_t *mma_done = ds_free + 2;
  uint32_t *s_tmem = (uint32_t *)(mma_done + 1);
  volatile int *s_abort = (volatile int *)(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  int *status = p.status;

  if (threadIdx.x == 0) {
    for (int x = 0; x < QB; ++x) {
      mbar_init(&q_full[x], 1);
      mbar_init(&q_empty[x], 1);
    }
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], kSmoothQ ? 1 + 128 : 1);  // both QKs' commit (+ the dS readers)
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int x = 0; x < 2 * NB; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&r_full[x], 1);
      mbar_init(&sr_free[x], 128);
    }
    for (int x = 0; x < 2 * PB; ++x) {
      mbar_init(&p_full[x], 128);
      mbar_init(&p_empty[x], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&ds_full[x], 128);
      mbar_init(&ds_free[x], 256);
    }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kX2Mma) {
    tmem_alloc(s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp >= kX2Producer) {
    reg_dealloc<kX2CtlRegs>();
    if (warp == kX2Producer && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      // Three streams over the CTA's items: Q^ pairs (up to QB items ahead of
      // the K stream), K^ tiles (up to ST ahead of V), V^T tiles.  Never
      // blocks on one stream while another could move; a stretch of the spin
      // limit without progress is a timeout.
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int qn = 0, kn = 0, vn = 0, kj = 0, vj = 0, gk = 0, gv = 0;
      X2Item qit, kit, vit;
      bool q_more = blockIdx.x < p.items, k_more = q_more, v_more = q_more;
      if (q_more) qit = kit = vit = x2_item(p, blockIdx.x);
      long long idle_since = clock64();
      while (q_more || k_more || v_more) {
        bool moved = false;
        if (q_more && qn < kn + QB &&
            (qn < QB || mbar_try_wait(&q_empty[qn % QB], ((qn / QB) - 1) & 1))) {
          const int qb = qn % QB;
          mbar_expect_tx(&q_full[qb], 2 * C::Q_TILE);
#pragma unroll
          for (int t = 0; t < 2; ++t)
            tma_load_2d(sQ + (qb * 2 + t) * C::Q_TILE, &tm_q, &q_full[qb], 0, qit.bh * p.N_pad + qit.p * 256 + t * 128);
          ++qn;
          const int nx = blockIdx.x + qn * G;
          q_more = nx < p.items;
          if (q_more) qit = x2_item(p, nx);
          moved = true;
        }
        if (k_more && gk < gv + ST && (gk < ST || mbar_try_wait(&k_empty[gk % ST], ((gk / ST) - 1) & 1))) {
          const int s = gk % ST;
          mbar_expect_tx(&k_full[s], C::K_BYTES);
          tma_load_2d(sK + s * C::K_BYTES, &tm_k, &k_full[s], 0, kit.hkv * p.M_pad + kj * BK);
          ++gk;
          if (++kj == kit.T) {
            kj = 0;
            const int nx = blockIdx.x + (++kn) * G;
            k_more = nx < p.items;
            if (k_more) kit = x2_item(p, nx);
          }
          moved = true;
        }
        if (v_more && gv < gk && (gv < ST || mbar_try_wait(&v_empty[gv % ST], ((gv / ST) - 1) & 1))) {
          const int s = gv % ST;
          mbar_expect_tx(&v_full[s], C::V_BYTES);
          tma_load_2d(sV + s * C::V_BYTES, &tm_v, &v_full[s], vj * BK, vit.hkv * D);
          ++gv;
          if (++vj == vit.T) {
            vj = 0;
            const int nx = blockIdx.x + (++vn) * G;
            v_more = nx < p.items;
            if (v_more) vit = x2_item(p, nx);
          }
          moved = true;
        }
        if (moved) {
          idle_since = clock64();
        } else {
          if (*s_abort) break;
          if (clock64() - idle_since > p.spin) {
            if (atomicCAS(status, 0, SAGE_ERR_TIMEOUT) == 0) status[1] = 110;
            *s_abort = 1;
            break;
          }
          __nanosleep(32);
        }
      }
      // drain: every load this thread issued lands before the CTA exits
      volatile int no_abort = 0;
      for (int n = max(0, qn - QB); n < qn; ++n)
        mbar_wait(&q_full[n % QB], (n / QB) & 1, status, 111, &no_abort, kDrainSpin);
      for (int j = max(0, gk - ST); j < gk; ++j) mbar_wait(&k_full[j % ST], (j / ST) & 1, status, 111, &no_abort, kDrainSpin);
      for (int j = max(0, gv - ST); j < gv; ++j) mbar_wait(&v_full[j % ST], (j / ST) & 1, status, 111, &no_abort, kDrainSpin);
    } else if (warp == kX2Mma) {
      // ---------------------------------------------------------- MMA issuer
      // Tile g of the CTA's walk: S(0, g) and S(1, g) into region g % NB of
      // each block, then R(0, g - 1) and R(1, g - 1) -- S runs one tile ahead
      // of R, into a region whose previous tile the softmax has folded.
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV), p_base = smem_u32(sP);
      // test hook (SAGE_TEST_STALL): mma_done completes its first phase only
      // after this warp's final commit, so the wait runs out (at half the
      // limit, before any other wait of the CTA could) and the CTA unwinds
      bool ok = !p.stall || __all_sync(0xffffffffu, mbar_wait(mma_done, 0, status, 29, s_abort, p.spin >> 1));
      auto issue_pv = [&](int g) -> bool {
        const int sv = g % ST, rb = g % NB;
        bool w = mbar_wait(&v_full[sv], (g / ST) & 1, status, 120, s_abort, p.spin);
        for (int t = 0; t < 2; ++t) {
          w = w && mbar_wait(&p_full[t * PB + g % PB], (g / PB) & 1, status, 121, s_abort, p.spin);
          if (!__all_sync(0xffffffffu, w)) return false;
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < C::PV_KSTEPS; ++kk) {
              const uint64_t ad = smem_desc(p_base + (t * PB + g % PB) * C::P_TILE + kk * 32, 512, kSwizzle64);
              const uint64_t bd = smem_desc(v_base + sv * C::V_BYTES + kk * 32, 512, kSwizzle64);
              mma_f8(tmem + (t * NB + rb) * 64, ad, bd, C::IDESC_PV, kk > 0);
            }
            mma_commit(&r_full[t * NB + rb]);
            mma_commit(&p_empty[t * PB + g % PB]);
          }
          __syncwarp();
        }
        if (elect_one()) mma_commit(&v_empty[sv]);
        __syncwarp();
        return true;
      };
      int g = 0;
      for (int n = 0; ok && blockIdx.x + n * G < p.items; ++n) {
        const X2Item it = x2_item(p, blockIdx.x + n * G);
        const int qb = n % QB;
        for (int j = 0; ok && j < it.T; ++j, ++g) {
          const int sk = g % ST, rb = g % NB;
          bool w = mbar_wait(&k_full[sk], (g / ST) & 1, status, 123, s_abort, p.spin);
          if (j == 0) w = w && mbar_wait(&q_full[qb], (n / QB) & 1, status, 124, s_abort, p.spin);
          for (int t = 0; t < 2; ++t) {
            if (g >= NB) w = w && mbar_wait(&sr_free[t * NB + rb], ((g / NB) - 1) & 1, status, 125, s_abort, p.spin);
            if (!__all_sync(0xffffffffu, w)) break;
            tc_fence_after();
            if (elect_one()) {
              const uint32_t qa = q_base + (qb * 2 + t) * C::Q_TILE;
#pragma unroll
              for (int kk = 0; kk < C::QK_KSTEPS; ++kk) {
                const uint64_t ad = smem_desc(qa + kk * 32, 8 * C::QK_SW, C::QK_LAYOUT);
                const uint64_t bd = smem_desc(k_base + sk * C::K_BYTES + kk * 32, 8 * C::QK_SW, C::QK_LAYOUT);
                if (kQK16)
                  mma_f16(tmem + (t * NB + rb) * 64, ad, bd, C::IDESC_QK, kk > 0);
                else
                  mma_f8(tmem + (t * NB + rb) * 64, ad, bd, C::IDESC_QK, kk > 0);
              }
              mma_commit(&s_full[t * NB + rb]);
            }
            __syncwarp();
          }
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mma_commit(&k_empty[sk]);
            if (j == it.T - 1) mma_commit(&q_empty[qb]);
          }
          __syncwarp();
          if (g > 0 && !issue_pv(g - 1)) ok = false;
        }
      }
      if (ok && g > 0) issue_pv(g - 1);
      if (elect_one()) mma_commit(mma_done);
      __syncwarp();
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, status, 127, &no_abort, kDrainSpin);
    }
  } else if (warp >= kX2DsWarp0) {
    // -------------------------------------------------------------- dS (Q smoothing)
    reg_dealloc<kX2DsRegs>();
    if constexpr (kSmoothQ) {
      // dS of key tile g for both query blocks of its item, in t units:
      // dS[t][c] = delta_K,j sum_d q_bar_t[d] K^_j[c, d] sm_scale log2(e),
      // thread c < 64 taking key c of block 0, thread 64 + c key c of block 1;
      // buffer g & 1, free again once both softmax warpgroups have read it
      const int c = threadIdx.x & 63, tb = (threadIdx.x >> 6) & 1;
      const float c2 = p.sm_log2;
      int g = 0;
      bool ok = true;
      // the group meets at a named barrier before and after each item's tiles;
      // each barrier ORs a failure flag, so after a wait that gave up every
      // thread leaves together (one leaving alone would strand the others)
      for (int n = 0; blockIdx.x + n * G < p.items; ++n) {
        const X2Item it = x2_item(p, blockIdx.x + n * G);
        float *qb = s_qb + (n & 1) * 2 * D;
        {
          const int qi = it.p * 2 + tb;  // thread tb * 64 + c writes q_bar[tb][c]
          qb[tb * D + c] = qi < p.Tm ? p.qbar[((size_t)it.bh * p.Tm + qi) * D + c] : 0.0f;
        }
        // the item's q_bar rows are read by every thread of the group; the
        // other parity's buffer still holds item n - 1's for slower threads
        if (named_bar_any(2, 128, *s_abort != 0)) break;
        const float *dkr = p.dk + (size_t)it.hkv * p.Tn;
        for (int j = 0; j < it.T; ++j, ++g) {
          const int b = g & 1, sk = g % ST;
          bool w = g < 2 || mbar_wait(&ds_free[b], ((g >> 1) - 1) & 1, status, 130, s_abort, p.spin);
          w = w && mbar_wait(&k_full[sk], (g / ST) & 1, status, 131, s_abort, p.spin);
          if (!w) {
            ok = false;
            break;
          }
          s_ds[(b * 2 + tb) * BK + c] = x2_qbar_dot<kQK16>(sK + sk * C::K_BYTES, qb + tb * D, c) * (dkr[j] * c2);
          mbar_arrive(&ds_full[b]);
          mbar_arrive(&k_empty[sk]);
        }
        if (named_bar_any(2, 128, !ok)) break;
      }
    }
  } else {
    // -------------------------------------------------------------- softmax + accumulation of block t
    reg_alloc<kX2SoftRegs>();
    const int t = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t tB = tmem + ((uint32_t)((warp & 3) * 32) << 16) + t * NB * 64;  // this block's regions
    const float c2 = p.sm_log2;
    bool stop = false;
    int g = 0;
    for (int n = 0; !stop && blockIdx.x + n * G < p.items; ++n) {
      const X2Item it = x2_item(p, blockIdx.x + n * G);
      const int qi = it.p * 2 + t;
      const bool tile_ok = qi < p.Tm;  // the second block of an odd count lies past the end
      const int row0 = qi * 128;
      const int diag = row0 + r + p.M - p.N;  // last key visible to this row (causal)
      const float dq = !tile_ok ? 0.0f
                       : (p.flags & SAGE_Q_PER_TOKEN) ? p.dqt[(size_t)it.bh * p.N_pad + row0 + r]
                                                      : p.dq[(size_t)it.bh * p.Tm + qi];
      const float *dkr = p.dk + (size_t)it.hkv * p.Tn;
      float o[D];  // this thread's row of the FP32 running output
      float m = -INFINITY, l = 0.0f, a_prev = 1.0f;
      float dk_next = dkr[0];
      // j = 0 .. T - 1: softmax of tile j, then the fold of tile j - 1;
      // j = T: the fold of the item's last tile only
      for (int j = 0; j <= it.T; ++j) {
        float alpha = 1.0f;
        if (j < it.T) {
          const int rb = g % NB;
          const float dkj = dk_next;
          const bool okw =
              __all_sync(0xffffffffu, mbar_wait(&s_full[t * NB + rb], (g / NB) & 1, status, 141, s_abort, p.spin) &&
                                          (!kSmoothQ || mbar_wait(&ds_full[g & 1], (g >> 1) & 1, status, 142, s_abort,
                                                                  p.spin)));
          if (!okw) {
            stop = true;
            break;
          }
          tc_fence_after();
          float x[BK];
          {
            uint32_t v[BK];
            tmem_ld32(tB + rb * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(tB + rb * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < BK; ++e) x[e] = __uint_as_float(v[e]);
          }
          if (j + 1 < it.T) dk_next = dkr[j + 1];
          const float k1 = dq * dkj * c2;  // S code -> t
          // x orders like t: the raw MMA output (scale folded into the
          // exponent) when k1 > 0 and there is no dS, else t itself (a masked
          // -inf never meets a zero scale)
          const bool raw = !kSmoothQ && k1 > 0.0f;
          const float xs = raw ? k1 : 1.0f;
          if constexpr (kSmoothQ) {
            const float4 *dsc = reinterpret_cast<const float4 *>(s_ds + ((g & 1) * 2 + t) * BK);
            const float2 k12 = make_float2(k1, k1);
#pragma unroll
            for (int e = 0; e < BK; e += 4) {
              const float4 d4 = dsc[e / 4];
              const float2 t01 = __ffma2_rn(make_float2(x[e], x[e + 1]), k12, make_float2(d4.x, d4.y));
              const float2 t23 = __ffma2_rn(make_float2(x[e + 2], x[e + 3]), k12, make_float2(d4.z, d4.w));
              x[e] = t01.x;
              x[e + 1] = t01.y;
              x[e + 2] = t23.x;
              x[e + 3] = t23.y;
            }
            mbar_arrive(&ds_free[g & 1]);
          } else if (!raw) {
#pragma unroll
            for (int e = 0; e < BK; ++e) x[e] *= k1;
          }
          if ((j * BK + BK > p.M) || (p.causal && j * BK + BK - 1 > row0 + p.M - p.N)) {
            const int lim = (p.causal ? min(p.M, diag + 1) : p.M) - j * BK;  // keys at or past lim are masked
#pragma unroll
            for (int e = 0; e < BK; ++e) x[e] = (e < lim) ? x[e] : -INFINITY;
          }
          float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int e = 0; e < BK; e += 8) {
            mq[0] = fmax3(mq[0], x[e], x[e + 1]);
            mq[1] = fmax3(mq[1], x[e + 2], x[e + 3]);
            mq[2] = fmax3(mq[2], x[e + 4], x[e + 5]);
            mq[3] = fmax3(mq[3], x[e + 6], x[e + 7]);
          }
          const float mx = fmax3(fmaxf(mq[0], mq[1]), mq[2], mq[3]);
          const float mt = (mx == -INFINITY) ? -INFINITY : mx * xs;  // row max of t over the tile
          const float m_new = fmaxf(m, mt);
          alpha = (m_new == -INFINITY) ? 1.0f : ex2_approx(m - m_new);
          // P^ = e4m3(448 exp2(t - m_new)) with the 448 in the exponent's
          // bias; a row with nothing visible yet has only masked keys (-> 0)
          const float mb = (m_new == -INFINITY) ? INFINITY : m_new - kX2Log2_448;
          const float2 xs2 = make_float2(xs, xs), nb2 = make_float2(-mb, -mb);
          float2 rs[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
          for (int e = 0; e < BK; e += 2) {
            const float2 arg = __ffma2_rn(make_float2(x[e], x[e + 1]), xs2, nb2);
            x[e] = ex2_approx(arg.x);
            x[e + 1] = ex2_approx(arg.y);
            rs[(e >> 1) & 1] = __fadd2_rn(rs[(e >> 1) & 1], make_float2(x[e], x[e + 1]));
          }
          l = fmaf(alpha, l, (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y));  // 448 times sum P~ against m_new
          m = m_new;
          // P^ into buffer g % PB of this block once its previous MMA has read it
          if (g >= PB && !__all_sync(0xffffffffu, mbar_wait(&p_empty[t * PB + g % PB], ((g / PB) - 1) & 1, status,
                                                            143, s_abort, p.spin))) {
            stop = true;
            break;
          }
          uint8_t *prow = sP + (t * PB + g % PB) * C::P_TILE;
#pragma unroll
          for (int c16 = 0; c16 < BK / 16; ++c16) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
              const int i0 = c16 * 16 + e;
              pk[e / 4] = (uint32_t)cvt_e4m3x2(x[i0], x[i0 + 1]) | ((uint32_t)cvt_e4m3x2(x[i0 + 2], x[i0 + 3]) << 16);
            }
            *reinterpret_cast<uint4 *>(prow + x2_swz<64>(r, c16)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&p_full[t * PB + g % PB]);
        }
        // ---- fold R of the previous tile (g - 1) into O, then free its region
        if (j > 0) {
          const int gp = g - 1, rp = gp % NB;
          if (!__all_sync(0xffffffffu, mbar_wait(&r_full[t * NB + rp], (gp / NB) & 1, status, 140, s_abort, p.spin))) {
            stop = true;
            break;
          }
          tc_fence_after();
          uint32_t rv[D];
          tmem_ld32(tB + rp * 64, *reinterpret_cast<uint32_t(*)[32]>(&rv[0]));
          tmem_ld32(tB + rp * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&rv[32]));
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&sr_free[t * NB + rp]);
          if (j == 1) {
#pragma unroll
            for (int c = 0; c < D; ++c) o[c] = __uint_as_float(rv[c]);
          } else {
            const float2 a2 = make_float2(a_prev, a_prev);
#pragma unroll
            for (int c = 0; c < D; c += 2) {
              const float2 o2 = __ffma2_rn(make_float2(o[c], o[c + 1]), a2,
                                           make_float2(__uint_as_float(rv[c]), __uint_as_float(rv[c + 1])));
              o[c] = o2.x;
              o[c + 1] = o2.y;
            }
          }
        }
        a_prev = alpha;
        if (j < it.T) ++g;
      }
      if (stop) break;
      // epilogue: O / l * delta_V (+ V_m) in bf16
      const int row = row0 + r;
      if (tile_ok && row < p.N) {
        const float inv_l = 1.0f / l;
        const float *dv = p.dv + (size_t)it.hkv * D, *vm = p.vm + (size_t)it.hkv * D;
        __nv_bfloat16 *dst = p.o + ((size_t)it.bh * p.N + row) * D;
#pragma unroll
        for (int c = 0; c < D; c += 8) {
          const float4 dv0 = __ldg(reinterpret_cast<const float4 *>(dv + c));
          const float4 dv1 = __ldg(reinterpret_cast<const float4 *>(dv + c + 4));
          const float4 vm0 = __ldg(reinterpret_cast<const float4 *>(vm + c));
          const float4 vm1 = __ldg(reinterpret_cast<const float4 *>(vm + c + 4));
          const float dvs[8] = {dv0.x, dv0.y, dv0.z, dv0.w, dv1.x, dv1.y, dv1.z, dv1.w};
          const float vms[8] = {vm0.x, vm0.y, vm0.z, vm0.w, vm1.x, vm1.y, vm1.z, vm1.w};
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(fmaf(o[c + 2 * e], dvs[2 * e] * inv_l, vms[2 * e]),
                                                            fmaf(o[c + 2 * e + 1], dvs[2 * e + 1] * inv_l, vms[2 * e + 1]));
            w[e] = *reinterpret_cast<const uint32_t *>(&v2);
          }
          *reinterpret_cast<uint4 *>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kX2Mma) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <bool kQK16, bool kSmoothQ>
sage_status launch_x2_t(const sage_shape &s, int causal, float sm_scale, int flags, const void *ws,
                        const sage_ws_layout &L, void *o, cudaStream_t stream) {
  using C = X2Cfg<kQK16, kSmoothQ>;
  const char *w = (const char *)ws;
  CUtensorMap tq, tk, tv;
  sage_status st;
  // Q rows of the last pair's second block may lie past the head (zero fill or
  // the next head's rows): their results are never stored
  st = make_tmap_2d(&tq, w + L.qhat, C::ROWB, (uint64_t)s.B * s.Hq * L.N_pad, C::ROWB, C::QK_SW, 128, C::QK_SW);
  if (st != SAGE_OK) return st;
  st = make_tmap_2d(&tk, w + L.khat, C::ROWB, (uint64_t)s.B * s.Hkv * L.M_pad, C::ROWB, C::QK_SW, C::BK, C::QK_SW);
  if (st != SAGE_OK) return st;
  st = make_tmap_2d(&tv, w + L.vhat, (uint64_t)L.M_pad, (uint64_t)s.B * s.Hkv * C::D, (uint64_t)L.M_pad, C::BK, C::D,
                    64);
  if (st != SAGE_OK) return st;
  X2Params p;
  p.N = s.N;
  p.M = s.M;
  p.N_pad = L.N_pad;
  p.M_pad = L.M_pad;
  p.Tm = L.Tm;
  p.Tn = L.Tn;
  p.Tp = (L.Tm + 1) / 2;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.causal = causal ? 1 : 0;
  p.flags = flags;
  p.items = s.B * s.Hq * p.Tp;
  p.sm_log2 = sm_scale * 1.4426950408889634f;
  p.dq = (const float *)(w + L.dq);
  p.dqt = (const float *)(w + L.dqt);
  p.qbar = (const float *)(w + L.qbar);
  p.dk = (const float *)(w + L.dk);
  p.dv = (const float *)(w + L.dv);
  p.vm = (const float *)(w + L.vm);
  p.o = (__nv_bfloat16 *)o;
  p.status = (int *)(w + L.status);
  p.spin = spin_limit_cycles();
  p.stall = test_stall();
  auto kern = attn_q8x2_kernel<kQK16, kSmoothQ>;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return SAGE_ERR_CUDA;
  if (fa.numRegs != kX2LaunchRegs) return SAGE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_TOTAL) != cudaSuccess)
    return SAGE_ERR_CUDA;
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      return SAGE_ERR_CUDA;
  }
  const int grid = p.items < sms ? p.items : sms;
  if (grid <= 0) return SAGE_OK;
  kern<<<(unsigned)grid, kX2Threads, C::SMEM_TOTAL, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}

}  // namespace

sage_status launch_attn_q8x2_64(const sage_shape &s, int causal, float sm_scale, int mode, int flags, const void *ws,
                                const sage_ws_layout &L, void *o, cudaStream_t stream) {
  const bool i8 = mode == SAGE_Q8_PV8, sq = (flags & SAGE_SMOOTH_Q) != 0;
  if (i8)
    return sq ? launch_x2_t<true, true>(s, causal, sm_scale, flags, ws, L, o, stream)
              : launch_x2_t<true, false>(s, causal, sm_scale, flags, ws, L, o, stream);
  return sq ? launch_x2_t<false, true>(s, causal, sm_scale, flags, ws, L, o, stream)
            : launch_x2_t<false, false>(s, causal, sm_scale, flags, ws, L, o, stream);
}

}  // namespace sage
