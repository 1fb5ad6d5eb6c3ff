// Fused NVFP4 attention on sm_103a (SageAttention3 summary §3.4, "FP4
// Attention Kernel Algorithm" and "Two-Level Quantization for P").
//
// Per CTA: one query block i of 128 rows of one (b, q-head); key tiles j of
// 128 keys:
//   S_ij  = FP4MMA(Q^_i, s_Q, K^_j, s_K)          block-scaled, E2M1 x UE4M3
//   m_ij  = max(m_i,j-1, rowmax S_ij sm_scale),   P~ = exp(S sm_scale - m_ij)
//   l_ij  = e^(m_i,j-1 - m_ij) l + rowsum P~        (unquantized P~)
//   s_P1  = rowmax P~_ij / (448 * 6) = exp(rowmax S_ij sm_scale - m_ij) / 2688
//   P2    = P~ / s_P1;  (s_P2, P2^) = phi(P2) over 1x16 blocks of keys
//   R_ij  = FP4MMA(P2^, s_P2, V^_j, s_V)            tile partial, this tile only
//   O_ij  = e^(m_i,j-1 - m_ij) O_i,j-1 + s_P1 R_ij  FP32 running output
//   O_i   = O / l + V_m
// In base 2, P2 = 2688 exp2(t - rowmax t) with t = S sm_scale log2(e), so the
// level-1 scale reuses the row maximum.  The maximum of P2 over a 1x16 block
// is exp2 of the block's largest t, which fixes s_P2 before the block's
// exponentials are taken; those are then computed already divided by s_P2,
// exp2(t + log2 2688 - rowmax t - log2 s_P2), and rounded to E2M1.
//
// Warps: WG0 and WG1 run the softmax and the two-level P quantization of the
// same 128 query rows, WG0 on keys 0-63 of each tile and WG1 on keys 64-127
// (one row per thread, its TMEM lane; the two halves trade row maxima through
// shared memory).  WG2 does the two-level accumulation O = alpha O + s_P1 R
// with O held in TMEM, then the epilogue.  Warp 12 issues the TMA and bulk
// copies, warp 13 (one thread) the tcgen05.cp of scale factors into TMEM and
// the block-scaled tcgen05.mma.  The S/R region and the P^ buffer are
// double-buffered so QK of tile j+1 runs under the softmax of tile j.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.h"
#include "launch.h"
#include "sm103.cuh"

namespace sage {
namespace {

constexpr int kWG = 128;
constexpr int kThreads = 512;
constexpr int kCorrWarp0 = 8, kProducerWarp = 12, kMmaWarp = 13;
constexpr int kLaunchRegs = 128, kSoftmaxRegs = 184, kCorrRegs = 88, kControlRegs = 56;
static_assert(kWG * (2 * kSoftmaxRegs + kCorrRegs + kControlRegs) <= kThreads * kLaunchRegs, "register split");
static_assert(kSoftmaxRegs >= kLaunchRegs && kCorrRegs <= kLaunchRegs && kControlRegs <= kLaunchRegs,
              "register split directions");
constexpr int BK = 128;       // keys per tile
constexpr int HALF = BK / 2;  // keys per softmax warpgroup
constexpr float kLog2_2688 = 11.392317422778762f;
// named barriers (0 is __syncthreads)
constexpr int kBarDs0 = 1;  // + half: dS of one warpgroup's keys
constexpr int kBarMax = 3;  // both softmax warpgroups: row-max exchange

template <int D>
struct Fp4Cfg {
  static constexpr int QROW = D / 2;  // bytes per Q / K row (packed E2M1)
  static constexpr int QK_SW = QROW;  // 64-byte (d=128) or 32-byte (d=64) swizzle
  static constexpr int QK_LAYOUT = QK_SW == 64 ? kSwizzle64 : kSwizzle32;
  static constexpr int Q_BYTES = 128 * QROW;
  static constexpr int QSF_BYTES = (D / 64) * 512;  // scale atoms of 128 rows
  static constexpr int K_BYTES = BK * QROW;
  static constexpr int V_BYTES = D * (BK / 2);       // V^T tile: D rows x BK/2 bytes
  static constexpr int VSF_BYTES = (BK / 64) * 512;  // one 128-channel atom per 64 keys
  static constexpr int P_BYTES = 128 * (BK / 2);
  static constexpr int PSF_BYTES = (BK / 64) * 512;
  static constexpr int STAGE = K_BYTES + QSF_BYTES + V_BYTES + VSF_BYTES;
  static constexpr int FIXED = Q_BYTES + QSF_BYTES + 2 * (P_BYTES + PSF_BYTES);
  static constexpr int STAGES = 4;
  static constexpr int NFLOAT = 2 * 128 /*alpha*/ + 2 * 128 /*s_P1*/ + 2 * 128 /*l*/ + 4 * 128 /*max*/ + 2 * D +
                                2 * BK /*dS*/;
  static constexpr int SMEM_TOTAL = 1024 + FIXED + STAGES * STAGE + NFLOAT * 4 + 256;
  static_assert(SMEM_TOTAL <= 227 * 1024, "shared memory");
  // TMEM columns: two S/R regions, O, scale factors (4 columns per 64-wide K step)
  static constexpr int SRW = 128;
  static constexpr int T_O = 2 * SRW;
  static constexpr int T_SFQ = 384;        // [D/64 steps]
  static constexpr int T_SFK = T_SFQ + 8;  // [2 buffers][D/64 steps]
  static constexpr int T_SFP = T_SFK + 16; // [2][BK/64]
  static constexpr int T_SFV = T_SFP + 16; // [2][BK/64]
  static constexpr int TMEM_COLS = 512;
  static_assert(T_SFV + 16 <= TMEM_COLS, "TMEM columns");
};

// byte offset of 16-byte chunk c of row r in a swizzled tile with SW-byte rows
template <int SW>
__device__ __forceinline__ uint32_t swz_off(int r, int c) {
  const int x = (SW == 128) ? (r & 7) : (SW == 64 ? ((r & 7) >> 1) : ((r & 7) >> 2));
  return (uint32_t)(r * SW + ((c ^ x) << 4));
}

__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
  return __half2float(__ushort_as_half((unsigned short)(cvt_e4m3x2_to_f16x2((uint16_t)(code & 0xFF)) & 0xFFFF)));
}

struct Fp4Params {
  int N, M, N_pad, M_pad, Tm, Tn, Hq, Hkv, causal, flags;
  float sm_log2;
  const uint8_t *qsf, *ksf, *vsf;
  const float *qbar, *vm;
  __nv_bfloat16 *o;
  int *status;
  long long spin;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fp4_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Fp4Params p) {
  using C = Fp4Cfg<D>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = base;
  uint8_t *sP = sQ + C::Q_BYTES;              // [2]
  uint8_t *sK = sP + 2 * C::P_BYTES;          // [ST]
  uint8_t *sV = sK + ST * C::K_BYTES;         // [ST]
  uint8_t *sQsf = sV + ST * C::V_BYTES;
  uint8_t *sPsf = sQsf + C::QSF_BYTES;        // [2]
  uint8_t *sKsf = sPsf + 2 * C::PSF_BYTES;    // [ST]
  uint8_t *sVsf = sKsf + ST * C::QSF_BYTES;   // [ST]
  float *s_alpha = (float *)(sVsf + ST * C::VSF_BYTES);  // [2][128]
  float *s_sp1 = s_alpha + 2 * 128;                      // [2][128]
  float *s_l = s_sp1 + 2 * 128;                          // [2 halves][128]
  float *s_mx = s_l + 2 * 128;                           // [2 buffers][2 halves][128]
  float *s_vm = s_mx + 4 * 128;                          // [D]
  float *s_qbar = s_vm + D;                              // [D]
  float *s_dsc = s_qbar + D;                             // [2 buffers][BK]
  uint64_t *bars = (uint64_t *)(((uintptr_t)(s_dsc + 2 * BK) + 7) & ~(uintptr_t)7);
  uint64_t *q_full = bars;
  uint64_t *k_full = q_full + 1;     // [ST]
  uint64_t *v_full = k_full + ST;    // [ST]
  uint64_t *kv_empty = v_full + ST;  // [ST]
  uint64_t *s_full = kv_empty + ST;  // [2]
  uint64_t *p_full = s_full + 2;     // [2]
  uint64_t *r_full = p_full + 2;     // [2]
  uint64_t *sr_free = r_full + 2;    // [2]
  uint64_t *mma_done = sr_free + 2;
  uint32_t *s_tmem = (uint32_t *)(mma_done + 1);
  volatile int *s_abort = (volatile int *)(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x / p.Tm;
  const int qi = p.Tm - 1 - blockIdx.x % p.Tm;  // longest causal rows first
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int hkv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int row0 = qi * 128;
  const int last_row = min(p.N, row0 + 128) - 1;
  const int T = p.causal ? min(p.Tn, (last_row + p.M - p.N) / BK + 1) : p.Tn;
  const bool smooth_q = (p.flags & SAGE_SMOOTH_Q) != 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 2 * kWG);
      mbar_init(&r_full[x], 1);
      mbar_init(&sr_free[x], kWG);
    }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  for (int c = threadIdx.x; c < D; c += kThreads) {
    s_vm[c] = p.vm[(size_t)hkv * D + c];
    s_qbar[c] = smooth_q ? p.qbar[((size_t)bh * p.Tm + qi) * D + c] : 0.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  int *status = p.status;

  if (warp >= kProducerWarp) {
    reg_dealloc<kControlRegs>();
    if (warp == kProducerWarp && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_expect_tx(q_full, C::Q_BYTES + C::QSF_BYTES);
      tma_load_2d(sQ, &tm_q, q_full, 0, bh * p.N_pad + row0);
      bulk_load(sQsf, p.qsf + ((size_t)bh * p.Tm + qi) * C::QSF_BYTES, C::QSF_BYTES, q_full);
      int issued = 0;
      for (int j = 0; j < T; ++j) {
        const int s = j % ST, n = j / ST;
        if (j >= ST && !mbar_wait(&kv_empty[s], (n - 1) & 1, status, 10, s_abort, p.spin)) break;
        mbar_expect_tx(&k_full[s], C::K_BYTES + C::QSF_BYTES);
        tma_load_2d(sK + s * C::K_BYTES, &tm_k, &k_full[s], 0, hkv * p.M_pad + j * BK);
        bulk_load(sKsf + s * C::QSF_BYTES, p.ksf + ((size_t)hkv * (p.M_pad / 128) + j) * C::QSF_BYTES,
                  C::QSF_BYTES, &k_full[s]);
        mbar_expect_tx(&v_full[s], C::V_BYTES + C::VSF_BYTES);
        tma_load_2d(sV + s * C::V_BYTES, &tm_v, &v_full[s], j * (BK / 2), hkv * D);
        bulk_load(sVsf + s * C::VSF_BYTES, p.vsf + ((size_t)hkv * (p.M_pad / 64) + j * (BK / 64)) * 512,
                  C::VSF_BYTES, &v_full[s]);
        issued = j + 1;
      }
      // before leaving, let the copies in flight land (bounded)
      volatile int no_abort = 0;
      mbar_wait(q_full, 0, status, 11, &no_abort, p.spin);
      for (int j = max(0, issued - ST); j < issued; ++j) {
        const int s = j % ST, n = j / ST;
        mbar_wait(&k_full[s], n & 1, status, 11, &no_abort, p.spin);
        mbar_wait(&v_full[s], n & 1, status, 11, &no_abort, p.spin);
      }
    } else if (warp == kMmaWarp && lane == 0) {
      // ---------------------------------------------------------- tcgen05 issuer
      // Scale-factor columns are double-buffered by tile parity: the copy for
      // tile j overwrites what tile j-2 used, and every MMA of tile j-2 has
      // completed by then (the sr_free wait of tile j-2 implies it).
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV), p_base = smem_u32(sP);
      bool ok = mbar_wait(q_full, 0, status, 23, s_abort, p.spin);
      tc_fence_after();
      if (ok)
        for (int a = 0; a < D / 64; ++a) tmem_cp_32x128b_x4(tmem + C::T_SFQ + 4 * a, smem_u32(sQsf + a * 512));
      auto issue_pv = [&](int jj) -> bool {
        const int bb = jj & 1, s = jj % ST;
        if (!mbar_wait(&p_full[bb], (jj >> 1) & 1, status, 20, s_abort, p.spin)) return false;
        if (!mbar_wait(&v_full[s], (jj / ST) & 1, status, 21, s_abort, p.spin)) return false;
        tc_fence_after();
        const uint32_t sfp = tmem + C::T_SFP + bb * 8, sfv = tmem + C::T_SFV + bb * 8;
#pragma unroll
        for (int a = 0; a < BK / 64; ++a) {
          tmem_cp_32x128b_x4(sfp + 4 * a, smem_u32(sPsf + bb * C::PSF_BYTES + a * 512));
          tmem_cp_32x128b_x4(sfv + 4 * a, smem_u32(sVsf + s * C::VSF_BYTES + a * 512));
        }
#pragma unroll
        for (int kk = 0; kk < BK / 64; ++kk) {
          const uint64_t ad = smem_desc(p_base + bb * C::P_BYTES + kk * 32, 8 * 64, kSwizzle64);
          const uint64_t bd = smem_desc(v_base + s * C::V_BYTES + kk * 32, 8 * 64, kSwizzle64);
          mma_fp4_bs(tmem + bb * C::SRW, ad, bd, instr_desc_fp4(D, 128), sfp + 4 * kk, sfv + 4 * kk, kk > 0);
        }
        mma_commit(&r_full[bb]);
        mma_commit(&kv_empty[s]);
        return true;
      };
      for (int j = 0; ok && j < T; ++j) {
        const int bs = j & 1, s = j % ST;
        if (j >= 2 && !mbar_wait(&sr_free[bs], ((j - 2) >> 1) & 1, status, 24, s_abort, p.spin)) ok = false;
        if (ok && !mbar_wait(&k_full[s], (j / ST) & 1, status, 26, s_abort, p.spin)) ok = false;
        if (!ok) break;
        tc_fence_after();
        const uint32_t sfk = tmem + C::T_SFK + bs * 8;
        for (int a = 0; a < D / 64; ++a) tmem_cp_32x128b_x4(sfk + 4 * a, smem_u32(sKsf + s * C::QSF_BYTES + a * 512));
#pragma unroll
        for (int kk = 0; kk < D / 64; ++kk) {
          const uint64_t ad = smem_desc(q_base + kk * 32, 8 * C::QK_SW, C::QK_LAYOUT);
          const uint64_t bd = smem_desc(k_base + s * C::K_BYTES + kk * 32, 8 * C::QK_SW, C::QK_LAYOUT);
          mma_fp4_bs(tmem + bs * C::SRW, ad, bd, instr_desc_fp4(BK, 128), tmem + C::T_SFQ + 4 * kk, sfk + 4 * kk,
                     kk > 0);
        }
        mma_commit(&s_full[bs]);
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok && T >= 1) issue_pv(T - 1);
      mma_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, status, 25, &no_abort, p.spin);
    }
  } else if (warp >= kCorrWarp0) {
    reg_dealloc<kCorrRegs>();
    // ------------------------------------------------------------ two-level accumulation + epilogue
    const int r = threadIdx.x & (kWG - 1);
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + lane_off + C::T_O;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int bb = j & 1;
      const bool waited = mbar_wait(&p_full[bb], (j >> 1) & 1, status, 40, s_abort, p.spin) &&
                          mbar_wait(&r_full[bb], (j >> 1) & 1, status, 41, s_abort, p.spin);
      // the TMEM accesses below are warp-collective: the warp decides together
      if (!__all_sync(0xffffffffu, waited)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float a = s_alpha[bb * 128 + r], sp1 = s_sp1[bb * 128 + r];
      const float2 a2 = make_float2(a, a), sp2 = make_float2(sp1, sp1);
      const uint32_t tR = tmem + lane_off + bb * C::SRW;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t rv[32], ov[32];
        tmem_ld32(tR + ch * 32, rv);
        if (j > 0) tmem_ld32(tO + ch * 32, ov);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 rr = make_float2(__uint_as_float(rv[e]), __uint_as_float(rv[e + 1]));
          float2 o2 = make_float2(0.0f, 0.0f);
          if (j > 0) o2 = __fmul2_rn(make_float2(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1])), a2);
          o2 = __ffma2_rn(rr, sp2, o2);
          ov[e] = __float_as_uint(o2.x);
          ov[e + 1] = __float_as_uint(o2.y);
        }
        tmem_st32(tO + ch * 32, ov);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sr_free[bb]);
    }
    // epilogue: O / l + V_m in bf16; every lane takes part in the TMEM loads,
    // only the stores are predicated
    if (ok && T >= 1) {
      const int row = row0 + r;
      const bool live = row < p.N;
      const float inv_l = live ? 1.0f / (s_l[r] + s_l[128 + r]) : 0.0f;
      __nv_bfloat16 *dst = p.o + ((size_t)bh * p.N + (live ? row : 0)) * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        __syncwarp();
        tmem_ld32(tO + ch * 32, ov);
        tmem_wait_ld();
        if (live) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int cc = ch * 32 + c + 2 * e;
              const __nv_bfloat162 v2 =
                  __floats2bfloat162_rn(fmaf(__uint_as_float(ov[c + 2 * e]), inv_l, s_vm[cc]),
                                        fmaf(__uint_as_float(ov[c + 2 * e + 1]), inv_l, s_vm[cc + 1]));
              w[e] = *reinterpret_cast<const uint32_t *>(&v2);
            }
            *reinterpret_cast<uint4 *>(dst + ch * 32 + c) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  } else {
    reg_alloc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax + two-level P quantization
    const int r = threadIdx.x & (kWG - 1);
    const int hf = warp >> 2;  // which half of the key tile
    const uint32_t tS = tmem + ((uint32_t)((warp & 3) * 32) << 16) + hf * HALF;
    const int diag = row0 + r + p.M - p.N;  // last key visible to this row (causal)
    const float c2 = p.sm_log2;
    float m = -INFINITY, l = 0.0f;
    for (int j = 0; j < T; ++j) {
      const int bb = j & 1;
      float *dsc = s_dsc + bb * BK;
      bool fail = false;
      if (smooth_q) {
        // dS_j[c] = sum_d q_bar[d] deq(K^_j)[c, d]: thread r < 64 of half hf
        // takes key 64 hf + r from the K tile in shared memory
        const int s = j % ST;
        fail = !mbar_wait(&k_full[s], (j / ST) & 1, status, 31, s_abort, p.spin);
        if (!fail && r < HALF) {
          const int key = hf * HALF + r;
          const uint8_t *kt = sK + s * C::K_BYTES;
          const uint8_t *ksf = sKsf + s * C::QSF_BYTES;
          float acc = 0.0f;
#pragma unroll
          for (int c16 = 0; c16 < C::QROW / 16; ++c16) {
            const uint4 w = *reinterpret_cast<const uint4 *>(kt + swz_off<C::QK_SW>(key, c16));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const int blk = c16 * 2 + hb;  // 16-channel block
              const float sc = e4m3_to_float(ksf[(blk >> 2) * 512 + (key & 31) * 16 + (key >> 5) * 4 + (blk & 3)]);
              float part = 0.0f;
#pragma unroll
              for (int q4 = 0; q4 < 2; ++q4) {
                uint32_t hv[4];
                cvt_e2m1x8_to_f16(ww[hb * 2 + q4], hv);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hv[e]));
                  const int d0 = blk * 16 + q4 * 8 + 2 * e;
                  part = fmaf(s_qbar[d0], f.x, part);
                  part = fmaf(s_qbar[d0 + 1], f.y, part);
                }
              }
              acc = fmaf(part, sc, acc);
            }
          }
          dsc[key] = acc * c2;
        }
        // every thread of the warpgroup reaches this barrier; a failure is
        // carried to the row-max barrier below, where both halves leave together
        named_bar_sync(kBarDs0 + hf, kWG);
      }
      // the TMEM loads are warp-collective: the warp decides together
      const bool ok =
          __all_sync(0xffffffffu, !fail && mbar_wait(&s_full[bb], (j >> 1) & 1, status, 32, s_abort, p.spin));
      float t[HALF];
      float bm[HALF / 16];
      float mx = -INFINITY;
#pragma unroll
      for (int g = 0; g < HALF / 16; ++g) bm[g] = -INFINITY;
      if (ok) {
        tc_fence_after();
        uint32_t v[HALF];
#pragma unroll
        for (int ch = 0; ch < HALF / 32; ++ch)
          tmem_ld32(tS + bb * C::SRW + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[ch * 32]));
        tmem_wait_ld();
        const int k0 = j * BK + hf * HALF;
        const bool need_mask = (k0 + HALF > p.M) || (p.causal && k0 + HALF - 1 > row0 + p.M - p.N);
#pragma unroll
        for (int e = 0; e < HALF; ++e) {
          float x = smooth_q ? fmaf(__uint_as_float(v[e]), c2, dsc[hf * HALF + e]) : __uint_as_float(v[e]) * c2;
          if (need_mask) {
            const int key = k0 + e;
            if (key >= p.M || (p.causal && key > diag)) x = -INFINITY;
          }
          t[e] = x;
        }
#pragma unroll
        for (int g = 0; g < HALF / 16; ++g) {
          float a = fmax3(t[16 * g], t[16 * g + 1], t[16 * g + 2]);
#pragma unroll
          for (int u = 3; u < 15; u += 2) a = fmax3(a, t[16 * g + u], t[16 * g + u + 1]);
          bm[g] = fmaxf(a, t[16 * g + 15]);
        }
        mx = fmax3(fmaxf(bm[0], bm[1]), bm[2], bm[3]);
      }
      s_mx[(bb * 2 + hf) * 128 + r] = mx;
      if (named_bar_any(kBarMax, 2 * kWG, !ok || *s_abort)) break;
      mx = fmaxf(mx, s_mx[(bb * 2 + (hf ^ 1)) * 128 + r]);

      const float m_new = fmaxf(m, mx);
      const float alpha = (m_new == -INFINITY) ? 1.0f : ex2_approx(m - m_new);
      const bool any = mx != -INFINITY;
      const float sp1 = any ? ex2_approx(mx - m_new) * (1.0f / 2688.0f) : 0.0f;
      const float shift = any ? kLog2_2688 - mx : 0.0f;
      uint8_t *prow = sP + bb * C::P_BYTES;
      uint32_t scw = 0;
      uint32_t pk[8];
      float rs = 0.0f;
#pragma unroll
      for (int g = 0; g < HALF / 16; ++g) {
        // s_P2 = E4M3(max P2 / 6) with max P2 = exp2(block max t + shift)
        const float amax = ex2_approx(bm[g] + shift);
        const uint32_t sc = cvt_e4m3x2(amax * (1.0f / 6.0f), 0.0f) & 0xFF;
        const float s2 = e4m3_to_float(sc);
        const float sb = s2 > 0.0f ? shift - lg2_approx(s2) : -INFINITY;
        float qv[16], bs = 0.0f;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          qv[u] = ex2_approx(t[16 * g + u] + sb);
          bs += qv[u];
        }
        rs = fmaf(s2, bs, rs);
        scw |= sc << (8 * g);
        pk[2 * g] = cvt_e2m1x8(qv[0], qv[1], qv[2], qv[3], qv[4], qv[5], qv[6], qv[7]);
        pk[2 * g + 1] = cvt_e2m1x8(qv[8], qv[9], qv[10], qv[11], qv[12], qv[13], qv[14], qv[15]);
      }
      // keys 64 hf .. 64 hf + 63 are bytes 32 hf .. 32 hf + 31 of row r
      *reinterpret_cast<uint4 *>(prow + swz_off<64>(r, 2 * hf)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4 *>(prow + swz_off<64>(r, 2 * hf + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      *reinterpret_cast<uint32_t *>(sPsf + bb * C::PSF_BYTES + hf * 512 + (r & 31) * 16 + (r >> 5) * 4) = scw;
      l = fmaf(alpha, l, sp1 * rs);
      m = m_new;
      if (hf == 0) {
        s_alpha[bb * 128 + r] = alpha;
        s_sp1[bb * 128 + r] = sp1;
      }
      if (j == T - 1) s_l[hf * 128 + r] = l;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[bb]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D>
sage_status launch_t(const sage_shape &s, int causal, float sm_scale, int flags, const void *ws,
                     const sage_ws_layout &L, void *o, cudaStream_t stream) {
  using C = Fp4Cfg<D>;
  const char *w = (const char *)ws;
  CUtensorMap tq, tk, tv;
  sage_status st;
  st = make_tmap_2d(&tq, w + L.qhat, C::QROW, (uint64_t)s.B * s.Hq * L.N_pad, C::QROW, C::QROW, 128, C::QK_SW);
  if (st != SAGE_OK) return st;
  st = make_tmap_2d(&tk, w + L.khat, C::QROW, (uint64_t)s.B * s.Hkv * L.M_pad, C::QROW, C::QROW, BK, C::QK_SW);
  if (st != SAGE_OK) return st;
  st = make_tmap_2d(&tv, w + L.vhat, L.M_pad / 2, (uint64_t)s.B * s.Hkv * D, L.M_pad / 2, BK / 2, D, 64);
  if (st != SAGE_OK) return st;
  Fp4Params p;
  p.N = s.N;
  p.M = s.M;
  p.N_pad = L.N_pad;
  p.M_pad = L.M_pad;
  p.Tm = L.Tm;
  p.Tn = (s.M + BK - 1) / BK;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.causal = causal ? 1 : 0;
  p.flags = flags;
  p.sm_log2 = sm_scale * 1.4426950408889634f;
  p.qsf = (const uint8_t *)(w + L.qsf);
  p.ksf = (const uint8_t *)(w + L.ksf);
  p.vsf = (const uint8_t *)(w + L.vsf);
  p.qbar = (const float *)(w + L.qbar);
  p.vm = (const float *)(w + L.vm);
  p.o = (__nv_bfloat16 *)o;
  p.status = (int *)(w + L.status);
  p.spin = spin_limit_cycles();
  auto kern = attn_fp4_kernel<D>;
  // the register split assumes the block launches with kLaunchRegs per thread
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return SAGE_ERR_CUDA;
  if (fa.numRegs != kLaunchRegs) return SAGE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_TOTAL) != cudaSuccess)
    return SAGE_ERR_CUDA;
  kern<<<(unsigned)(s.B * s.Hq * L.Tm), kThreads, C::SMEM_TOTAL, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}

}  // namespace

sage_status launch_attn_fp4(const sage_shape &s, int causal, float sm_scale, int flags, int bk, const void *ws,
                            const sage_ws_layout &L, void *o, cudaStream_t stream) {
  if (bk != BK) return SAGE_ERR_UNSUPPORTED;
  return s.d == 64 ? launch_t<64>(s, causal, sm_scale, flags, ws, L, o, stream)
                   : launch_t<128>(s, causal, sm_scale, flags, ws, L, o, stream);
}

}  // namespace sage
