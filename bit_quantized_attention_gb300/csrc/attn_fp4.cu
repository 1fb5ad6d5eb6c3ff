// Fused NVFP4 attention on sm_103a (SageAttention3 summary §3.4, "FP4
// Attention Kernel Algorithm" and "Two-Level Quantization for P").
//
// Per CTA: one query block i of 128 rows of one (b, q-head); key tiles j of
// 128 keys:
//   S_ij  = FP4MMA(Q^_i, s_Q, K^_j, s_K)          block-scaled, E2M1 x UE4M3
//   m_ij  = max(m_i,j-1, rowmax S_ij sm_scale),   P~ = exp(S sm_scale - m_ij)
//   l_ij  = e^(m_i,j-1 - m_ij) l + rowsum P~        (unquantized P~)
//   s_P1  = rowmax P~_ij / (448 * 6) = exp(rowmax S_ij sm_scale - m_ij) / 2688
//           (1 under the direct-P~ ablation, which quantizes P~ itself)
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
// (one row per thread, its TMEM lane; the halves trade their maxima through
// shared memory, late enough that neither waits).  WG2 does the two-level accumulation O = alpha O + s_P1 R
// with its row of O held in registers, then the epilogue.  Warp 12 issues the
// TMA and bulk copies; warp 13 issues QK (the scale-factor copies into TMEM
// and the block-scaled tcgen05.mma) and warp 14 issues PV, one elected lane
// each.  Three S/R regions in TMEM (R of tile j overwrites S of tile j) let
// QK run up to three tiles ahead of the accumulation, so neither the MMAs nor
// the accumulation sit on the softmax's critical path.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "layout.h"
#include "launch.h"
#include "sm103.cuh"

namespace sage {
namespace {

constexpr int kWG = 128;
constexpr int kThreads = 512;
constexpr int kCorrWarp0 = 8, kProducerWarp = 12, kQkWarp = 13, kPvWarp = 14;
constexpr int kLaunchRegs = 128, kSoftmaxRegs = 136, kCorrRegs = 184, kControlRegs = 56;
static_assert(kWG * (2 * kSoftmaxRegs + kCorrRegs + kControlRegs) <= kThreads * kLaunchRegs, "register split");
static_assert(kSoftmaxRegs >= kLaunchRegs && kCorrRegs >= kLaunchRegs && kControlRegs <= kLaunchRegs,
              "register split directions");
constexpr int NB = 3;         // S/R regions, P^ buffers
constexpr int BK = 128;       // keys per tile
constexpr int HALF = BK / 2;  // keys per softmax warpgroup
constexpr float kLog2_2688 = 11.392317422778762f;
// named barriers (0 is __syncthreads): 1 + half, one softmax warpgroup (dS)
constexpr int kBarDs0 = 1;

// kPing: the softmax warpgroups take whole key tiles in turn (one more
// [NB][128] float array: each tile's row sum, from which the accumulation
// warpgroup keeps l)
template <int D, bool kPing = false>
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
  static constexpr int FIXED = Q_BYTES + QSF_BYTES + NB * (P_BYTES + PSF_BYTES);
  static constexpr int STAGES = 4;
  static constexpr int NFLOAT = NB * 128 /*alpha*/ + NB * 128 /*s_P1*/ + 2 * 128 /*l*/ + 4 * 128 /*max*/ +
                                2 * D + 4 * BK /*dS*/ + (kPing ? NB * 128 : 0) /*row sums*/;
  static constexpr int SMEM_TOTAL = 1024 + FIXED + STAGES * STAGE + NFLOAT * 4 + 512;
  static_assert(SMEM_TOTAL <= 227 * 1024, "shared memory");
  // TMEM columns: NB S/R regions, then scale factors, 4 columns per 64-wide K
  // step; K, P and V scale slots follow the S/R region of their tile
  static constexpr int SRW = 128;
  static constexpr int T_SFQ = NB * SRW;           // [D/64 steps]
  static constexpr int T_SFK = T_SFQ + 8;          // [NB][D/64 steps]
  static constexpr int T_SFP = T_SFK + 8 * NB;     // [NB][BK/64]
  static constexpr int T_SFV = T_SFP + 8 * NB;     // [NB][BK/64]
  static constexpr int TMEM_COLS = 512;
  static_assert(T_SFV + 8 * NB <= TMEM_COLS, "TMEM columns");
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
  int stall;  // test hook: the QK issuer first waits on a barrier nothing arrives on
  // packed sequences (kVar): block b of the grid takes work item item_tab[b]
  // (code bh * Tm + qi); seq holds each sequence's lengths and first rows
  const int *item_tab;
  const VarSeq *seq;
};

// kSmoothQ: Q smoothing on (dS on CUDA cores, added to the scores); an
// instance of its own, so the others carry none of its code in their loops
template <int D, bool kPing, bool kVar, bool kSmoothQ>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fp4_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Fp4Params p) {
  using C = Fp4Cfg<D, kPing>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = base;
  uint8_t *sP = sQ + C::Q_BYTES;              // [NB]
  uint8_t *sK = sP + NB * C::P_BYTES;         // [ST]
  uint8_t *sV = sK + ST * C::K_BYTES;         // [ST]
  uint8_t *sQsf = sV + ST * C::V_BYTES;
  uint8_t *sPsf = sQsf + C::QSF_BYTES;        // [NB]
  uint8_t *sKsf = sPsf + NB * C::PSF_BYTES;   // [ST]
  uint8_t *sVsf = sKsf + ST * C::QSF_BYTES;   // [ST]
  float *s_alpha = (float *)(sVsf + ST * C::VSF_BYTES);  // [NB][128]
  float *s_sp1 = s_alpha + NB * 128;                     // [NB][128]
  float *s_l = s_sp1 + NB * 128;                         // [2 halves][128]
  float *s_mx = s_l + 2 * 128;                           // [2 parities][2 halves][128]
  float *s_vm = s_mx + 4 * 128;                          // [D]
  float *s_qbar = s_vm + D;                              // [D]
  float *s_dsc = s_qbar + D;                             // [2 buffers][2 halves][BK]
  float *s_rs = s_dsc + 4 * BK;                          // [NB][128] row sums (tiles in turn)
  uint64_t *bars = (uint64_t *)(((uintptr_t)(s_rs + (kPing ? NB * 128 : 0)) + 7) & ~(uintptr_t)7);
  uint64_t *q_full = bars;
  uint64_t *k_full = q_full + 1;     // [ST]
  uint64_t *v_full = k_full + ST;    // [ST]
  uint64_t *kv_empty = v_full + ST;  // [ST]
  uint64_t *s_full = kv_empty + ST;  // [NB]
  uint64_t *p_full = s_full + NB;    // [NB]
  uint64_t *r_full = p_full + NB;    // [NB]
  uint64_t *sr_free = r_full + NB;   // [NB]
  uint64_t *mx_full = sr_free + NB;  // [2 parities][2 halves]
  uint64_t *qk_done = mx_full + 4;
  uint64_t *pv_done = qk_done + 1;
  uint32_t *s_tmem = (uint32_t *)(pv_done + 1);
  volatile int *s_abort = (volatile int *)(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this block's query block: longest causal rows first (batched: by block
  // index; packed sequences: the table's order); Nq, Mk its sequence's counts
  int bh, qi, Nq = p.N, Mk = p.M, q0 = 0;
  if constexpr (kVar) {
    const int code = p.item_tab[blockIdx.x];
    bh = code / p.Tm;
    qi = code % p.Tm;
    const VarSeq sq = p.seq[bh / p.Hq];
    Nq = sq.N;
    Mk = sq.M;
    q0 = sq.q0;
  } else {
    bh = blockIdx.x / p.Tm;
    qi = p.Tm - 1 - blockIdx.x % p.Tm;
  }
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int hkv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int row0 = qi * 128;
  const int last_row = min(Nq, row0 + 128) - 1;
  const int Tn = kVar ? (Mk + BK - 1) / BK : p.Tn;
  const int T = p.causal ? min(Tn, (last_row + Mk - Nq) / BK + 1) : Tn;
  constexpr bool smooth_q = kSmoothQ;
  const bool direct = (p.flags & SAGE_P_DIRECT) != 0;  // phi on P~ itself (ablation)

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int x = 0; x < NB; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], kPing ? kWG : 2 * kWG);  // one or both softmax warpgroups
      mbar_init(&r_full[x], 1);
      mbar_init(&sr_free[x], kWG);
    }
    for (int x = 0; x < 4; ++x) mbar_init(&mx_full[x], kWG);
    mbar_init(qk_done, 1);
    mbar_init(pv_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kQkWarp) {
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
      mbar_wait(q_full, 0, status, 11, &no_abort, kDrainSpin);
      for (int j = max(0, issued - ST); j < issued; ++j) {
        const int s = j % ST, n = j / ST;
        mbar_wait(&k_full[s], n & 1, status, 11, &no_abort, kDrainSpin);
        mbar_wait(&v_full[s], n & 1, status, 11, &no_abort, kDrainSpin);
      }
    } else if (warp == kQkWarp) {
      // ---------------------------------------------------------- QK issuer (whole warp, one lane issues)
      // QK of tile j reuses S/R region j % NB and K scale slot j % NB once the
      // accumulation has consumed R of tile j - NB, which also means every
      // MMA that read them has completed.
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK);
      // test hook (SAGE_TEST_STALL): qk_done completes its first phase only
      // after this warp's final commit, so the wait runs out (at half the
      // limit, before any other wait of the CTA could) and the CTA unwinds
      bool ok = !p.stall || __all_sync(0xffffffffu, mbar_wait(qk_done, 0, status, 29, s_abort, p.spin >> 1));
      ok = ok && __all_sync(0xffffffffu, mbar_wait(q_full, 0, status, 23, s_abort, p.spin));
      tc_fence_after();
      if (ok && elect_one())
        for (int a = 0; a < D / 64; ++a) tmem_cp_32x128b_x4(tmem + C::T_SFQ + 4 * a, smem_u32(sQsf + a * 512));
      __syncwarp();
      for (int j = 0; ok && j < T; ++j) {
        const int b = j % NB, s = j % ST;
        bool w = true;
        if (j >= NB) w = mbar_wait(&sr_free[b], ((j - NB) / NB) & 1, status, 24, s_abort, p.spin);
        w = w && mbar_wait(&k_full[s], (j / ST) & 1, status, 26, s_abort, p.spin);
        if (!__all_sync(0xffffffffu, w)) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t sfk = tmem + C::T_SFK + b * 8;
          for (int a = 0; a < D / 64; ++a)
            tmem_cp_32x128b_x4(sfk + 4 * a, smem_u32(sKsf + s * C::QSF_BYTES + a * 512));
#pragma unroll
          for (int kk = 0; kk < D / 64; ++kk) {
            const uint64_t ad = smem_desc(q_base + kk * 32, 8 * C::QK_SW, C::QK_LAYOUT);
            const uint64_t bd = smem_desc(k_base + s * C::K_BYTES + kk * 32, 8 * C::QK_SW, C::QK_LAYOUT);
            mma_fp4_bs(tmem + b * C::SRW, ad, bd, instr_desc_fp4(BK, 128), tmem + C::T_SFQ + 4 * kk, sfk + 4 * kk,
                       kk > 0);
          }
          mma_commit(&s_full[b]);
        }
        __syncwarp();
      }
      // every MMA of this thread has finished before the CTA may leave
      if (elect_one()) mma_commit(qk_done);
      __syncwarp();
      volatile int no_abort = 0;
      mbar_wait(qk_done, 0, status, 25, &no_abort, kDrainSpin);
    } else if (warp == kPvWarp) {
      // ---------------------------------------------------------- PV issuer (whole warp, one lane issues)
      // PV of tile j writes R into S/R region j % NB once the softmax has read
      // S of tile j; P and V scale slot j % NB were last read by PV of tile
      // j - NB, complete since QK of tile j was issued after its R was consumed.
      const uint32_t v_base = smem_u32(sV), p_base = smem_u32(sP);
      for (int j = 0; j < T; ++j) {
        const int b = j % NB, s = j % ST;
        const bool w = mbar_wait(&p_full[b], (j / NB) & 1, status, 20, s_abort, p.spin) &&
                       mbar_wait(&v_full[s], (j / ST) & 1, status, 21, s_abort, p.spin);
        if (!__all_sync(0xffffffffu, w)) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t sfp = tmem + C::T_SFP + b * 8, sfv = tmem + C::T_SFV + b * 8;
#pragma unroll
          for (int a = 0; a < BK / 64; ++a) {
            tmem_cp_32x128b_x4(sfp + 4 * a, smem_u32(sPsf + b * C::PSF_BYTES + a * 512));
            tmem_cp_32x128b_x4(sfv + 4 * a, smem_u32(sVsf + s * C::VSF_BYTES + a * 512));
          }
#pragma unroll
          for (int kk = 0; kk < BK / 64; ++kk) {
            const uint64_t ad = smem_desc(p_base + b * C::P_BYTES + kk * 32, 8 * 64, kSwizzle64);
            const uint64_t bd = smem_desc(v_base + s * C::V_BYTES + kk * 32, 8 * 64, kSwizzle64);
            mma_fp4_bs(tmem + b * C::SRW, ad, bd, instr_desc_fp4(D, 128), sfp + 4 * kk, sfv + 4 * kk, kk > 0);
          }
          mma_commit(&r_full[b]);
          mma_commit(&kv_empty[s]);
        }
        __syncwarp();
      }
      if (elect_one()) mma_commit(pv_done);
      __syncwarp();
      volatile int no_abort = 0;
      mbar_wait(pv_done, 0, status, 27, &no_abort, kDrainSpin);
    }
  } else if (warp >= kCorrWarp0) {
    reg_alloc<kCorrRegs>();
    // ------------------------------------------------------------ two-level accumulation + epilogue
    const int r = threadIdx.x & (kWG - 1);
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float o[D];  // this thread's row of the FP32 running output
#pragma unroll
    for (int c = 0; c < D; ++c) o[c] = 0.0f;
    float lsum = 0.0f;  // l, kept here when the softmax warpgroups take tiles in turn
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int b = j % NB;
      const bool waited = mbar_wait(&p_full[b], (j / NB) & 1, status, 40, s_abort, p.spin) &&
                          mbar_wait(&r_full[b], (j / NB) & 1, status, 41, s_abort, p.spin);
      // the TMEM loads below are warp-collective: the warp decides together
      if (!__all_sync(0xffffffffu, waited)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float a = s_alpha[b * 128 + r], sp1 = s_sp1[b * 128 + r];
      if constexpr (kPing) lsum = fmaf(a, lsum, s_rs[b * 128 + r]);
      const float2 a2 = make_float2(a, a), sp2 = make_float2(sp1, sp1);
      const uint32_t tR = tmem + lane_off + b * C::SRW;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t rv[32];
        tmem_ld32(tR + ch * 32, rv);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 rr = make_float2(__uint_as_float(rv[e]), __uint_as_float(rv[e + 1]));
          const float2 o2 = __ffma2_rn(rr, sp2, __fmul2_rn(make_float2(o[ch * 32 + e], o[ch * 32 + e + 1]), a2));
          o[ch * 32 + e] = o2.x;
          o[ch * 32 + e + 1] = o2.y;
        }
      }
      tc_fence_before();
      mbar_arrive(&sr_free[b]);
    }
    // epilogue: O / l + V_m in bf16
    if (ok && T >= 1) {
      const int row = row0 + r;
      if (row < Nq) {
        const float inv_l = 1.0f / (kPing ? lsum : s_l[r] + s_l[128 + r]);
        // the output row: batched [B, Hq, N, d], or packed [total_q, Hq, d]
        __nv_bfloat16 *dst = kVar ? p.o + ((size_t)(q0 + row) * p.Hq + h) * D : p.o + ((size_t)bh * p.N + row) * D;
#pragma unroll
        for (int c = 0; c < D; c += 8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(fmaf(o[c + 2 * e], inv_l, s_vm[c + 2 * e]),
                                                            fmaf(o[c + 2 * e + 1], inv_l, s_vm[c + 2 * e + 1]));
            w[e] = *reinterpret_cast<const uint32_t *>(&v2);
          }
          *reinterpret_cast<uint4 *>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  } else if constexpr (kPing) {
    reg_alloc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax + two-level P, whole tiles in turn
    // Warpgroup w takes tiles j with j % 2 == w, all BK keys of its rows,
    // streamed from TMEM in 32-column chunks twice: the 16-key block maxima
    // first, then P2 and its E2M1 codes.  Only the running maximum passes
    // between the warpgroups (s_mx[j % NB] and mx_full[j % NB], published
    // before the exponentials); the tile's row sum goes to the accumulation
    // warpgroup (s_rs), which keeps l.  With Q smoothing the warpgroup computes
    // the tile's dS for all its keys first (thread r takes key r), into a
    // buffer of its own that alternates between its tiles.
    static_assert(NB % 2 == 1, "the reader of a running maximum is its next writer");
    const int r = threadIdx.x & (kWG - 1);
    const int wg = warp >> 2;
    const uint32_t tS0 = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int diag = row0 + r + Mk - Nq;  // last key visible to this row (causal)
    const float c2 = p.sm_log2;
    const float xs = smooth_q ? 1.0f : c2;  // x -> t
    bool stop = false;  // a wait failed late in this warp's previous tile
    for (int j = wg; j < T; j += 2) {
      const int bb = j % NB;
      float *dsc = s_dsc + (((j >> 1) & 1) * 2 + wg) * BK;
      const bool okw = __all_sync(0xffffffffu, mbar_wait(&s_full[bb], (j / NB) & 1, status, 32, s_abort, p.spin));
      if (smooth_q) {
        const int s = j % ST;
        const bool fail = stop || !mbar_wait(&k_full[s], (j / ST) & 1, status, 31, s_abort, p.spin);
        if (!fail) {
          const int key = r;
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
        // the warpgroup leaves together: a warp that stopped alone would strand
        // the others at this barrier in its next tile
        if (named_bar_any(kBarDs0 + wg, kWG, stop || fail || !okw || *s_abort)) break;
      } else if (stop || !okw) {
        break;
      }
      tc_fence_after();
      const int lim = (p.causal ? min(Mk, diag + 1) : Mk) - j * BK;  // tile keys >= lim are invisible
      const bool edge = (j * BK + BK > Mk) || (p.causal && j * BK + BK - 1 > row0 + Mk - Nq);
      const uint32_t tSb = tS0 + bb * C::SRW;
      // pass 1: 16-key block maxima in x (raw S, or t with dS)
      float bm[BK / 16];
#pragma unroll
      for (int ch = 0; ch < BK / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(tSb + ch * 32, v);
        tmem_wait_ld();
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          x[e] = __uint_as_float(v[e]);
          if (smooth_q) x[e] = fmaf(x[e], c2, dsc[ch * 32 + e]);
          if (edge && ch * 32 + e >= lim) x[e] = -INFINITY;
        }
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          float a = fmax3(x[16 * g], x[16 * g + 1], x[16 * g + 2]);
#pragma unroll
          for (int u = 3; u < 15; u += 2) a = fmax3(a, x[16 * g + u], x[16 * g + u + 1]);
          bm[2 * ch + g] = fmaxf(a, x[16 * g + 15]);
        }
      }
      float mx = bm[0];
#pragma unroll
      for (int g = 1; g < BK / 16; ++g) mx = fmaxf(mx, bm[g]);
      const float mt = (mx == -INFINITY) ? -INFINITY : mx * xs;  // row max of t over the tile
      float m_prev = -INFINITY;
      if (j > 0) {
        const int pb = (j - 1) % NB;
        if (!__all_sync(0xffffffffu, mbar_wait(&mx_full[pb], ((j - 1) / NB) & 1, status, 33, s_abort, p.spin))) {
          stop = true;
          if (!smooth_q) break;
          continue;  // leave with the warpgroup at the next dS barrier
        }
        m_prev = s_mx[pb * 128 + r];
      }
      const float m_new = fmaxf(m_prev, mt);
      s_mx[bb * 128 + r] = m_new;
      mbar_arrive(&mx_full[bb]);
      const float alpha = (m_new == -INFINITY) ? 1.0f : ex2_approx(m_prev - m_new);
      const bool any = mt != -INFINITY;
      const float sp1 = !any ? 0.0f : direct ? 1.0f : ex2_approx(mt - m_new) * (1.0f / 2688.0f);
      // P2 = P~ / s_P1 = exp2(t - bias): 2688 exp2(t - m_tile), or P~ itself
      // (direct); nothing visible -> every P2 is 0
      const float bias = !any ? INFINITY : direct ? m_new : mt - kLog2_2688;
      float mult[BK / 16];
      uint32_t scw[BK / 64];
#pragma unroll
      for (int q = 0; q < BK / 64; ++q) scw[q] = 0;
#pragma unroll
      for (int g = 0; g < BK / 16; ++g) {
        // s_P2 = E4M3(max P2 / 6) from the block's largest score
        const float amax = (bm[g] == -INFINITY) ? 0.0f : ex2_approx(fmaf(bm[g], xs, -bias));
        const uint32_t sc = cvt_e4m3x2(amax * (1.0f / 6.0f), 0.0f) & 0xFF;
        const float s2 = e4m3_to_float(sc);
        mult[g] = s2 > 0.0f ? __fdividef(1.0f, s2) : 0.0f;
        scw[g >> 2] |= sc << (8 * (g & 3));
      }
      // pass 2: P2, its E2M1 codes (32 keys = one 16-byte chunk of the 64-byte row)
      uint8_t *prow = sP + bb * C::P_BYTES;
      float2 rs2 = make_float2(0.0f, 0.0f);
      const float2 xs2 = make_float2(xs, xs), nb2 = make_float2(-bias, -bias);
#pragma unroll
      for (int ch = 0; ch < BK / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(tSb + ch * 32, v);
        tmem_wait_ld();
        float qv[32];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float x0 = __uint_as_float(v[e]), x1 = __uint_as_float(v[e + 1]);
          if (smooth_q) {
            x0 = fmaf(x0, c2, dsc[ch * 32 + e]);
            x1 = fmaf(x1, c2, dsc[ch * 32 + e + 1]);
          }
          if (edge) {
            x0 = (ch * 32 + e < lim) ? x0 : -INFINITY;
            x1 = (ch * 32 + e + 1 < lim) ? x1 : -INFINITY;
          }
          const float2 arg = __ffma2_rn(make_float2(x0, x1), xs2, nb2);
          const float p0 = ex2_approx(arg.x), p1 = ex2_approx(arg.y);
          rs2 = __fadd2_rn(rs2, make_float2(p0, p1));
          const float mu = mult[2 * ch + (e >> 4)];
          qv[e] = p0 * mu;
          qv[e + 1] = p1 * mu;
        }
        const uint32_t w0 = cvt_e2m1x8(qv[0], qv[1], qv[2], qv[3], qv[4], qv[5], qv[6], qv[7]);
        const uint32_t w1 = cvt_e2m1x8(qv[8], qv[9], qv[10], qv[11], qv[12], qv[13], qv[14], qv[15]);
        const uint32_t w2 = cvt_e2m1x8(qv[16], qv[17], qv[18], qv[19], qv[20], qv[21], qv[22], qv[23]);
        const uint32_t w3 = cvt_e2m1x8(qv[24], qv[25], qv[26], qv[27], qv[28], qv[29], qv[30], qv[31]);
        *reinterpret_cast<uint4 *>(prow + swz_off<64>(r, ch)) = make_uint4(w0, w1, w2, w3);
      }
#pragma unroll
      for (int q = 0; q < BK / 64; ++q)
        *reinterpret_cast<uint32_t *>(sPsf + bb * C::PSF_BYTES + q * 512 + (r & 31) * 16 + (r >> 5) * 4) = scw[q];
      s_alpha[bb * 128 + r] = alpha;
      s_sp1[bb * 128 + r] = sp1;
      s_rs[bb * 128 + r] = sp1 * (rs2.x + rs2.y);  // this tile's sum of P~ against m_new
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[bb]);
    }
  } else {
    reg_alloc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax + two-level P quantization
    const int r = threadIdx.x & (kWG - 1);
    const int hf = warp >> 2;  // which half of the key tile
    const uint32_t tS0 = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int diag = row0 + r + Mk - Nq;  // last key visible to this row (causal)
    const float c2 = p.sm_log2;
    float m = -INFINITY, l = 0.0f;
    bool stop = false;  // a wait failed late in the previous tile
    for (int j = 0, bb = 0, pj = 0; j < T; ++j, bb = (bb + 1 == NB) ? 0 : bb + 1, pj ^= (bb == 0) ? 1 : 0) {
      // this warpgroup's copy of dS for all BK keys of the tile
      float *dsc = s_dsc + ((j & 1) * 2 + hf) * BK;
      // the TMEM loads are warp-collective: the warp decides together
      const bool okw = __all_sync(0xffffffffu, mbar_wait(&s_full[bb], pj, status, 32, s_abort, p.spin));
      if (smooth_q) {
        // dS_j[c] = sum_d q_bar[d] deq(K^_j)[c, d]: thread r takes key r from
        // the K tile in shared memory (each warpgroup keeps its own copy)
        const int s = j % ST;
        const bool fail = !mbar_wait(&k_full[s], (j / ST) & 1, status, 31, s_abort, p.spin);
        if (!fail) {
          const int key = r;
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
        // the warpgroup leaves together: a warp that stops alone would strand
        // the others at this barrier in the next tile
        if (named_bar_any(kBarDs0 + hf, kWG, stop || fail || !okw || *s_abort)) break;
      } else if (stop || !okw) {
        break;
      }
      tc_fence_after();
      // x: this half's raw scores S (t = x c2), or t itself when dS is added
      // (then c2 is already applied); maxima are taken in x, which orders
      // like t.  Each half publishes its maximum at once and takes its
      // exponentials against it, e = exp2(t - m_half); the tile maximum
      // m_tile then enters as one factor, P2 = 2688 exp2(t - m_tile) =
      // e * 2688 exp2(m_half - m_tile), so neither half waits on the other
      // before its exponentials.
      const int lim = (p.causal ? min(Mk, diag + 1) : Mk) - j * BK;  // tile keys >= lim are invisible
      const bool edge = (j * BK + BK > Mk) || (p.causal && j * BK + BK - 1 > row0 + Mk - Nq);
      const int oh = hf ^ 1;
      float x[HALF];
      float bm[HALF / 16];
      {
        uint32_t v[HALF];
#pragma unroll
        for (int ch = 0; ch < HALF / 32; ++ch)
          tmem_ld32(tS0 + bb * C::SRW + hf * HALF + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[ch * 32]));
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < HALF; ++e) x[e] = __uint_as_float(v[e]);
      }
      if (smooth_q) {
#pragma unroll
        for (int e = 0; e < HALF; ++e) x[e] = fmaf(x[e], c2, dsc[hf * HALF + e]);
      }
      if (edge) {
#pragma unroll
        for (int e = 0; e < HALF; ++e) x[e] = (hf * HALF + e < lim) ? x[e] : -INFINITY;
      }
#pragma unroll
      for (int g = 0; g < HALF / 16; ++g) {
        float a = fmax3(x[16 * g], x[16 * g + 1], x[16 * g + 2]);
#pragma unroll
        for (int u = 3; u < 15; u += 2) a = fmax3(a, x[16 * g + u], x[16 * g + u + 1]);
        bm[g] = fmaxf(a, x[16 * g + 15]);
      }
      const float mh = fmax3(fmaxf(bm[0], bm[1]), bm[2], bm[3]);
      s_mx[((j & 1) * 2 + hf) * 128 + r] = mh;
      mbar_arrive(&mx_full[(j & 1) * 2 + hf]);
      const float xs = smooth_q ? 1.0f : c2;  // x -> t
      const float mht = (mh == -INFINITY) ? 0.0f : mh * xs;
      const float2 xs2 = make_float2(xs, xs), nm2 = make_float2(-mht, -mht);
      float2 se2 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int u = 0; u < HALF; u += 2) {
        const float2 arg = __ffma2_rn(make_float2(x[u], x[u + 1]), xs2, nm2);
        x[u] = ex2_approx(arg.x);
        x[u + 1] = ex2_approx(arg.y);
        se2 = __fadd2_rn(se2, make_float2(x[u], x[u + 1]));
      }
      // the other half's maximum
      if (!__all_sync(0xffffffffu, mbar_wait(&mx_full[(j & 1) * 2 + oh], (j >> 1) & 1, status, 33, s_abort, p.spin))) {
        stop = true;
        if (!smooth_q) break;
        continue;  // leave with the warpgroup at the next dS barrier
      }
      const float mt = fmaxf(mh, s_mx[((j & 1) * 2 + oh) * 128 + r]) * xs;  // row max of t over the tile
      const float m_new = fmaxf(m, mt);
      const float alpha = (m_new == -INFINITY) ? 1.0f : ex2_approx(m - m_new);
      const bool any = mt != -INFINITY;
      // direct P~ (ablation): s_P1 = 1 and P2 = P~ = e exp2(m_half - m_new)
      const float sp1 = !any ? 0.0f : direct ? 1.0f : ex2_approx(mt - m_new) * (1.0f / 2688.0f);
      const float f = (!any || mh == -INFINITY) ? 0.0f
                      : direct                 ? ex2_approx(mht - m_new)
                                               : ex2_approx(mht - mt) * 2688.0f;  // P2 = e f
      uint8_t *prow = sP + bb * C::P_BYTES;
      uint32_t scw = 0;
      uint32_t pk[8];
      float mult[HALF / 16];
#pragma unroll
      for (int g = 0; g < HALF / 16; ++g) {
        // s_P2 = E4M3(max P2 / 6); the block's largest e is exp2 of its largest t
        const float amax = ex2_approx(fmaf(bm[g], xs, -mht)) * f;
        const uint32_t sc = cvt_e4m3x2(amax * (1.0f / 6.0f), 0.0f) & 0xFF;
        const float s2 = e4m3_to_float(sc);
        mult[g] = s2 > 0.0f ? __fdividef(f, s2) : 0.0f;  // P2 / s_P2 = e f / s_P2
        scw |= sc << (8 * g);
      }
#pragma unroll
      for (int g = 0; g < HALF / 16; ++g) {
        const float2 mu2 = make_float2(mult[g], mult[g]);
        float qv[16];
#pragma unroll
        for (int u = 0; u < 16; u += 2) {
          const float2 q2 = __fmul2_rn(make_float2(x[16 * g + u], x[16 * g + u + 1]), mu2);
          qv[u] = q2.x;
          qv[u + 1] = q2.y;
        }
        pk[2 * g] = cvt_e2m1x8(qv[0], qv[1], qv[2], qv[3], qv[4], qv[5], qv[6], qv[7]);
        pk[2 * g + 1] = cvt_e2m1x8(qv[8], qv[9], qv[10], qv[11], qv[12], qv[13], qv[14], qv[15]);
      }
      const float rs = f * (se2.x + se2.y);  // this half's sum of P2
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
  if (warp == kQkWarp) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, bool kPing, bool kVar>
sage_status launch_t(const sage_shape &s, int causal, float sm_scale, int flags, const void *ws,
                     const sage_ws_layout &L, void *o, cudaStream_t stream, const VarDev &var) {
  using C = Fp4Cfg<D, kPing>;
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
  p.stall = test_stall();
  p.item_tab = var.item_tab;
  p.seq = var.seq;
  auto kern = (flags & SAGE_SMOOTH_Q) ? attn_fp4_kernel<D, kPing, kVar, true> : attn_fp4_kernel<D, kPing, kVar, false>;
  // the register split assumes the block launches with kLaunchRegs per thread
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return SAGE_ERR_CUDA;
  if (fa.numRegs != kLaunchRegs) return SAGE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_TOTAL) != cudaSuccess)
    return SAGE_ERR_CUDA;
  const int blocks = kVar ? var.items : s.B * s.Hq * L.Tm;
  if (blocks <= 0) return SAGE_OK;
  kern<<<(unsigned)blocks, kThreads, C::SMEM_TOTAL, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}

}  // namespace

sage_status launch_attn_fp4(const sage_shape &s, int causal, float sm_scale, int flags, int bk, const void *ws,
                            const sage_ws_layout &L, void *o, cudaStream_t stream, const VarDev &var) {
  if (bk != BK) return SAGE_ERR_UNSUPPORTED;
  if (var.item_tab)  // packed sequences: the split schedule
    return s.d == 64 ? launch_t<64, false, true>(s, causal, sm_scale, flags, ws, L, o, stream, var)
                     : launch_t<128, false, true>(s, causal, sm_scale, flags, ws, L, o, stream, var);
  // whole key tiles in turn between the softmax warpgroups (SAGE_PINGPONG=1)
  const char *pp = getenv("SAGE_PINGPONG");
  if (pp && pp[0] == '1')
    return s.d == 64 ? launch_t<64, true, false>(s, causal, sm_scale, flags, ws, L, o, stream, var)
                     : launch_t<128, true, false>(s, causal, sm_scale, flags, ws, L, o, stream, var);
  return s.d == 64 ? launch_t<64, false, false>(s, causal, sm_scale, flags, ws, L, o, stream, var)
                   : launch_t<128, false, false>(s, causal, sm_scale, flags, ws, L, o, stream, var);
}

}  // namespace sage
