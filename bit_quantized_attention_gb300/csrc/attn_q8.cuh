#pragma once
// Fused quantized attention for the INT8 / FP8 modes on sm_103a (the kernel
// template and its launcher; attn_q8.cu, attn_q8_ping.cu and attn_q8_var.cu
// instantiate the schedules and request kinds, so they compile in parallel).
//
// What it computes, per query block i of 128 rows of one (b, q-head), over the
// key tiles j = 0..T-1 of its kv-head (SageAttention2 Technical Report summary
// §3.4 "The Complete Algorithm"; "Quantization for Attention, in depth",
// "The datapath and its quantize points"):
//   S_ij  = delta_Q delta_K,j (Q^_i K^_j^T) + dS_ij,  dS_ij = q_bar_i deq(K^_j)^T
//           (delta_Q one per query block, or one per row with per-token Q scales)
//   m_ij  = max(m_i,j-1, rowmax S_ij * sm_scale)
//   P~_ij = exp(S_ij sm_scale - m_ij),  l_ij = e^(m_i,j-1 - m_ij) l + rowsum P~
//   P^_ij = e4m3(448 P~_ij)                          (static scale 1/448)
//   R_ij  = P^_ij V^_j        (tile partial, accumulated over this tile only)
//   O_ij  = e^(m_i,j-1 - m_ij) O_i,j-1 + R_ij        (FP32 running output)
//   O_i   = O / l * delta_V / 448 (+ V_m)
// Scores are handled in the base-2 domain, t = S sm_scale log2 e, and the 448
// of P^ is folded into the exponent, so l carries 448 * sum P~ and the final
// scale is delta_V / l.
//
// GB300 mapping (the pages' Ada/Hopper register-level design is prior art):
// a persistent CTA per SM walks its share of the work items (one query block
// of one head each: head-major, or for causal masks pairs of complementary
// blocks of one head; round robin over the CTAs) with 16 warps; every ring and barrier phase runs on tile counters that continue
// across items, so the next item's loads and first MMAs overlap the previous
// item's last tiles and epilogue.
//   warps 0-7   two warpgroups on the same 128 query rows (one row per thread,
//               its TMEM lane); warpgroup h takes keys [h BK/2, (h+1) BK/2) of
//               every tile: dequantize (adding dS where it is not folded into
//               S), mask, exponentials, P^ into the
//               swizzled K-major A operand of the PV MMA in shared memory.
//               Each half publishes its own maximum at once and takes its
//               exponentials against it, e = exp2(t - m_half); the new running
//               maximum enters afterwards as one factor, P^ = e4m3(e * 448
//               exp2(m_half - m_new)), so neither half waits on the other
//               before its exponentials.
//   warps 8-11  two-level accumulation O = alpha O + R with the thread's row
//               of O in registers, then the epilogue; with Q smoothing also
//               dS ahead of the softmax: read from TMEM (one key per thread)
//               where the tensor core computed it and written as the tile's
//               key augmentation (the correction then comes folded into S),
//               else computed from the K^ tile in shared memory for the
//               softmax to add
//   warp 12     TMA producer: Q^ once, K^_j and V^T_j into a ring of stages
//   warp 13     QK issuer: S(j) = Q^ K^_j^T (kind::f16 on INT8 codes held as
//               exact fp16 integers -- sm_103a has no INT8 tensor path -- or
//               kind::f8f6f4 on E4M3 codes); with Q smoothing on INT8 codes
//               and 128-key tiles also dS^T(j) = K^_j U^T, U the item's q_bar
//               as fp16 hi / lo rows (kind::f16, M = 128 keys, N = 16), run
//               ahead, and S(j) starts from one kind::tf32 step
//               [1/delta_Q rows] x [dS keys]^T of the augmentation operands
//   warp 14     PV issuer: R(j) = P^(j) V^_j (kind::f8f6f4)
// TMEM: three S/R regions (R of tile j overwrites S of tile j once the softmax
// has read it), so QK runs up to three tiles ahead of the accumulation; with
// the tensor-core dS, three 16-column dS regions after them.
// Waits are bounded: on timeout the kernel records SAGE_ERR_TIMEOUT and the
// site, drains its own TMA loads and MMAs, frees TMEM and returns.
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

constexpr int kWG = 128;       // threads per warpgroup
constexpr int kThreads = 512;  // softmax x2, accumulation, control
constexpr int kCorrWarp0 = 8, kProducerWarp = 12, kQkWarp = 13, kPvWarp = 14;
// Register split (setmaxnreg) from the 128 per thread the block launches with.
constexpr int kLaunchRegs = 128, kSoftmaxRegs = 136, kCorrRegs = 184, kControlRegs = 56;
static_assert(kWG * (2 * kSoftmaxRegs + kCorrRegs + kControlRegs) <= kThreads * kLaunchRegs, "register split");
static_assert(kSoftmaxRegs >= kLaunchRegs && kCorrRegs >= kLaunchRegs && kControlRegs <= kLaunchRegs,
              "register split directions");
constexpr int NB = 3;  // S/R regions and P^ buffers
constexpr float kLog2_448 = 8.807354922057604f;

// kDsT: dS on the tensor core (Q smoothing with INT8 codes and 128-key tiles):
// a 16-row tile of q_bar (fp16 hi / lo rows) per item parity in shared memory
// and NB 16-column dS regions in TMEM.  kPV16: the SageBwd forward, P^ and V^
// as INT8 codes held in fp16 (kind::f16 PV), with a per-row factor
// s_P s_V,j per tile for the accumulation and the row statistics kept
template <int D, int BK, bool kQK16, bool kDsT = false, bool kPV16 = false>
struct Cfg {
  static constexpr int HALF = BK / 2;                    // keys per softmax warpgroup
  static constexpr int QK_EB = kQK16 ? 2 : 1;           // bytes per stored Q/K code
  static constexpr int ROWB = D * QK_EB;                 // bytes per Q/K row
  static constexpr int QK_SW = ROWB >= 128 ? 128 : 64;   // swizzle span of Q/K tiles
  static constexpr int QK_CHUNKS = ROWB / QK_SW;         // swizzle spans per row
  static constexpr int PV_EB = kPV16 ? 2 : 1;           // bytes per stored P^ / V^ code
  static constexpr int PV_SW = BK * PV_EB >= 128 ? 128 : 64;  // swizzle span of P^ and V^T tiles
  static constexpr int Q_BYTES = 128 * ROWB;
  static constexpr int K_BYTES = BK * ROWB;
  static constexpr int V_BYTES = D * BK * PV_EB;
  static constexpr int P_BYTES = 128 * BK * PV_EB;
  static constexpr int QK_KSTEPS = ROWB / 32;            // one MMA consumes 32 bytes of K
  static constexpr int PV_KSTEPS = BK * PV_EB / 32;
  static constexpr int NFLOAT = NB * 128 /*alpha*/ + NB * 256 /*l*/ + 4 * 128 /*max*/ + NB * BK /*dS*/ + 2 * D /*q_bar*/ +
                                (kPV16 ? 2 * NB * 128 : 0) /*s_P s_V, final max*/;
  static constexpr int UB_BYTES = kDsT ? 16 * ROWB : 0;  // one q_bar tile (16 rows, K-major, swizzled)
  // one augmentation operand of the QK product: 128 rows of 8 TF32 words
  // (32-byte rows, 32-byte swizzle); per item the rows' 1/delta_Q, per tile the keys' dS
  static constexpr int AUG_BYTES = kDsT ? 128 * 32 : 0;
  static constexpr int FIXED = Q_BYTES + NB * P_BYTES + 2 * UB_BYTES + (2 + NB) * AUG_BYTES;
  static constexpr int MISC = NFLOAT * 4 + 512;  // floats, then barriers
  // K and V have rings of their own: a K tile is free once its QK has run
  // (and, with dS, once the accumulation warpgroup has read it); a V tile once its PV has
  static constexpr int BUDGET = 225 * 1024 - 1024 - FIXED - MISC;
  static constexpr int VST = 2 * (K_BYTES + V_BYTES) <= BUDGET - K_BYTES ? 3 : 2;
  static constexpr int KST_FIT = (BUDGET - VST * V_BYTES) / K_BYTES;
  static constexpr int KST = KST_FIT > 4 ? 4 : KST_FIT;
  static_assert(KST >= 2 && VST >= 2, "shared memory budget");
  static constexpr int SRW = BK > D ? BK : D;            // columns of one S / R region
  static constexpr int DS_COL = NB * SRW;                // first column of the dS regions
  static constexpr int TMEM_COLS = NB * SRW + (kDsT ? NB * 16 : 0) <= 256 ? 256 : 512;
  static_assert(NB * SRW + (kDsT ? NB * 16 : 0) <= 512, "TMEM columns");
  static_assert(!kDsT || (kQK16 && BK == 128 && QK_SW == 128), "dS on the tensor core: INT8 codes, 128-key tiles");
  static constexpr int SMEM_TOTAL = 1024 + FIXED + KST * K_BYTES + VST * V_BYTES + MISC;
  static constexpr uint32_t IDESC_QK =
      instr_desc(kFmtF32, kQK16 ? kFmtF16 : kFmtE4M3, kQK16 ? kFmtF16 : kFmtE4M3, BK, 128);
  static constexpr uint32_t IDESC_PV =
      instr_desc(kFmtF32, kPV16 ? kFmtF16 : kFmtE4M3, kPV16 ? kFmtF16 : kFmtE4M3, D, 128);
  static_assert(!kPV16 || (kQK16 && BK == 64), "SageBwd forward: INT8 codes, 64-key tiles");
  // dS^T = K^ (128 keys x d, A) x q_bar tile (16 x d, B): column 0 the hi row, 1 the lo row
  static constexpr uint32_t IDESC_DS = instr_desc(kFmtF32, kFmtF16, kFmtF16, 16, 128);
  // S = [1/delta_Q row augmentation] x [dS key augmentation]^T, then += Q^ K^T
  static constexpr uint32_t IDESC_AUG = instr_desc(kFmtF32, kFmtTF32, kFmtTF32, BK, 128);
};

// The causal work order's per-launch constants (see causal_item): the grid G,
// pairs per head PH = Tm / 2, the items in full rounds of pairs, the pairs left
// after them, the middle blocks (one per head when Tm is odd), and 1/G, 1/PH.
struct CausalOrder {
  int G, PH, full, rest, mid;
  float invG, invPH;
};

struct AttnParams {
  int N, M, N_pad, M_pad, Tm, Tn, Hq, Hkv, causal, flags;
  int items;      // work items (one query block of one head each): B * Hq * Tm, or the table's
  float sm_log2;  // sm_scale * log2(e)
  const float *dq, *qbar, *dk, *dv, *vm;
  const float *dqt;  // per-row Q scales [B*Hq*N_pad] (SAGE_Q_PER_TOKEN)
  const float *dvb;  // per-block V scales [B*Hkv*Tn] (SageBwd forward)
  float *lse;        // per-row log-sum-exp [B*Hq*N_pad] (SageBwd forward)
  // packed sequences: the work item codes (bh * Tm + qi, longest first) and
  // each sequence's lengths and first packed rows; null for a batched request
  const int *item_tab;
  const VarSeq *seq;
  __nv_bfloat16 *o;
  int *status;
  long long spin;
  int stall;  // test hook: the QK issuer first waits on a barrier nothing arrives on
  CausalOrder cz;
};

// byte offset of 16-byte chunk `c` of row `r` in a K-major swizzled tile whose
// rows are `SW` bytes wide (8-row atoms of 8*SW bytes, 1024-aligned base)
template <int SW>
__device__ __forceinline__ uint32_t swz_off(int r, int c) {
  const int x = (SW == 128) ? (r & 7) : ((r & 7) >> 1);
  return (uint32_t)((r >> 3) * (8 * SW) + (r & 7) * SW + ((c ^ x) << 4));
}

// Work item idx of the grid-wide list: longest causal rows first (batched
// causal: by block index, heads interleaved; batched non-causal: head-major;
// kVar, packed sequences: the table's order).  N, M: the
// item's query and key counts (the request's, or its sequence's); q0: the
// sequence's first row in the packed output (kVar).
struct Item {
  int bh, qi, hkv, row0, T, N, M, q0;
};
// a / d for 0 <= a < 2^24 and d >= 1, given inv = fl(1/d): the float quotient
// is within one of the truth, and one step each way corrects it
__device__ __forceinline__ int div_small(int a, int d, float inv) {
  int q = __float2int_rz(__int2float_rn(a) * inv);
  q -= (q * d > a) ? 1 : 0;
  q += ((q + 1) * d <= a) ? 1 : 0;
  return q;
}

// Causal items differ in length, but a head's query blocks qi and Tm - 1 - qi
// together always take the same number of key tiles.  Items are handed out in
// such pairs: in round k of the grid (items k G .. k G + G - 1) CTA c takes the
// long block of pair (k / 2) G + c when k is even, its short block when k is
// odd.  Every CTA then gets the same work per two rounds, runs both blocks of
// a pair back to back on one head's K / V, and the CTAs in flight share
// G / (Tm / 2) heads' K / V tiles in L2.  The pairs left after the full rounds,
// and the middle block of each head when Tm is odd, come last, longest first.
// The launcher supplies G and the pair counts (AttnParams::cz); every division
// here is by one of them.  Returns (head, query block).
__device__ __forceinline__ int2 causal_item(const AttnParams &p, int idx) {
  const CausalOrder &z = p.cz;
  int P;
  bool lng;
  if (idx < z.full) {  // full rounds of pairs
    const int k = div_small(idx, z.G, z.invG);
    P = (k >> 1) * z.G + (idx - k * z.G);
    lng = (k & 1) == 0;
  } else {
    const int rem = idx - z.full;
    if (rem >= z.rest && rem < z.rest + z.mid) return make_int2(rem - z.rest, z.PH);  // middle blocks
    lng = rem < z.rest;  // long blocks of the last pairs, then their short blocks
    P = z.full / 2 + (lng ? rem : rem - z.rest - z.mid);
  }
  const int h = div_small(P, z.PH, z.invPH), j = P - h * z.PH;
  return make_int2(h, lng ? p.Tm - 1 - j : j);
}

template <bool kVar>
__device__ __forceinline__ Item item_of(const AttnParams &p, int idx, int BK) {
  Item it;
  if constexpr (kVar) {
    const int code = p.item_tab[idx];
    it.qi = code % p.Tm;
    it.bh = code / p.Tm;
    const VarSeq sq = p.seq[it.bh / p.Hq];
    it.N = sq.N;
    it.M = sq.M;
    it.q0 = sq.q0;
  } else if (p.causal) {
    const int2 bq = causal_item(p, idx);
    it.bh = bq.x;
    it.qi = bq.y;
    it.N = p.N;
    it.M = p.M;
    it.q0 = 0;
  } else {
    // head-major: items of equal length, and the CTAs in flight share one or
    // two heads' K / V tiles, which stay in L2 while every block streams them
    it.qi = idx % p.Tm;
    it.bh = idx / p.Tm;
    it.N = p.N;
    it.M = p.M;
    it.q0 = 0;
  }
  const int b = it.bh / p.Hq, h = it.bh % p.Hq;
  it.hkv = b * p.Hkv + h / (p.Hq / p.Hkv);
  it.row0 = it.qi * 128;
  const int Tn = kVar ? (it.M + BK - 1) / BK : p.Tn;
  const int last_row = min(it.N, it.row0 + 128) - 1;
  it.T = p.causal ? min(Tn, (last_row + it.M - it.N) / BK + 1) : Tn;
  return it;
}

// sum_d q_bar[d] K^[r, d] for key r of a K^ tile in shared memory (the codes
// are exact in fp16 / E4M3; q_bar in shared memory too, every lane the same word)
template <int D, int BK, bool kQK16>
__device__ __forceinline__ float qbar_dot_key(const uint8_t *kt, const float *qbar, int r) {
  using C = Cfg<D, BK, kQK16>;
  constexpr int kSpan = C::QK_SW / 16;  // 16-byte chunks per swizzle span
  // four independent chains; a short unroll: the caller keeps its row of O live
  // in registers meanwhile
  float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                   make_float2(0.0f, 0.0f)};
#pragma unroll 2
  for (int k = 0; k < C::ROWB / 16; ++k) {
    const int cc = k / kSpan, c16 = k % kSpan;
    const uint4 w = *reinterpret_cast<const uint4 *>(kt + cc * BK * C::QK_SW + swz_off<C::QK_SW>(r, c16));
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

// kSmoothQ: Q smoothing on (dS added to the scores, or folded into S by the
// tensor core); its instances carry the dS stream, the others none of its
// state.  kPV16: the SageBwd forward.  kPing:
// the softmax warpgroups take whole key tiles in turn instead of halves of
// every tile (INT8 / FP8 P~).  kVar: packed sequences (work item table and
// per-sequence lengths).
template <int D, int BK, bool kQK16, bool kSmoothQ, bool kPV16, bool kPing = false, bool kVar = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_q8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  // dS on the tensor core where the codes allow it (INT8 as fp16, 128-key tiles),
  // folded into S; otherwise the accumulation warpgroup takes it on CUDA cores
  // and the softmax adds it
  constexpr bool kDsMma = kSmoothQ && kQK16 && BK == 128;
  // the softmax adds dS itself (the CUDA-core dS); with kDsMma it comes inside S
  constexpr bool kDsAdd = kSmoothQ && !kDsMma;
  static_assert(!kPing || !kPV16, "tiles in turn: FP8 P~");
  using C = Cfg<D, BK, kQK16, kDsMma, kPV16>;
  constexpr int KST = C::KST, VST = C::VST;
  // tensor-core dS: how many tiles ahead of a QK the issuer runs the dS MMA
  // (it waits for that K^ tile first, so the lead stays below the K^ ring)
  constexpr int kDsAhead = KST >= 3 ? 2 : 1;
  constexpr int HALF = C::HALF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = base;
  uint8_t *sP = sQ + C::Q_BYTES;        // [NB]
  uint8_t *sK = sP + NB * C::P_BYTES;   // [KST]
  uint8_t *sV = sK + KST * C::K_BYTES;  // [VST]
  uint8_t *sU = sV + VST * C::V_BYTES;  // [2 item parities] q_bar tiles (dS on the tensor core)
  uint8_t *sAq = sU + 2 * C::UB_BYTES;   // [2 item parities] row augmentation: 1/delta_Q
  uint8_t *sAk = sAq + 2 * C::AUG_BYTES; // [NB] key augmentation: dS of a tile
  float *s_alpha = (float *)(sAk + NB * C::AUG_BYTES);  // [NB][128]
  float *s_l = s_alpha + NB * 128;                   // [NB][2 halves][128], at an item's last tile
  float *s_mx = s_l + NB * 256;                      // [2 parities][2 halves][128]
  float *s_ds = s_mx + 4 * 128;                      // [NB][BK] dS of a tile, in t units
  float *s_qb = s_ds + NB * BK;                      // [2 item parities][D] q_bar of the dS stream
  float *s_w = s_qb + 2 * D;                         // [NB][128] s_P s_V,j of a tile (SageBwd)
  float *s_mrow = s_w + (kPV16 ? NB * 128 : 0);      // [NB][128] running max at an item's last tile (SageBwd)
  uint64_t *bars = (uint64_t *)(((uintptr_t)(s_mrow + (kPV16 ? NB * 128 : 0)) + 7) & ~(uintptr_t)7);
  uint64_t *q_full = bars;
  uint64_t *q_empty = q_full + 1;
  uint64_t *k_full = q_empty + 1;    // [KST]
  uint64_t *k_empty = k_full + KST;  // [KST]
  uint64_t *v_full = k_empty + KST;  // [VST]
  uint64_t *v_empty = v_full + VST;  // [VST]
  uint64_t *s_full = v_empty + VST;  // [NB] S in TMEM
  uint64_t *p_full = s_full + NB;    // [NB] P^, alpha written; S read
  uint64_t *r_full = p_full + NB;    // [NB] R in TMEM
  uint64_t *sr_free = r_full + NB;   // [NB] R folded into O; region free
  uint64_t *mx_full = sr_free + NB;  // [2 parities][2 halves] half maxima
  uint64_t *ds_full = mx_full + 4;   // [NB] dS of the tile in s_ds
  uint64_t *qb_full = ds_full + NB;  // [2] q_bar of the dS stream's item in s_qb
  uint64_t *dsr_full = qb_full + 2;  // [NB] dS^T of a tile in TMEM (tensor-core dS)
  uint64_t *dsr_free = dsr_full + NB;  // [NB] that TMEM region read
  uint64_t *ub_full = dsr_free + NB;   // [2] q_bar tile of an item written
  uint64_t *ub_empty = ub_full + 2;    // [2] its last dS MMA and QK done
  uint64_t *aug_full = ub_empty + 2;   // [NB] key augmentation of a tile written
  uint64_t *aug_empty = aug_full + NB; // [NB] its QK done
  uint64_t *qk_done = aug_empty + NB;
  uint64_t *pv_done = qk_done + 1;
  uint32_t *s_tmem = (uint32_t *)(pv_done + 1);
  volatile int *s_abort = (volatile int *)(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  constexpr bool smooth_q = kSmoothQ;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], (smooth_q && !kDsMma) ? 1 + kWG : 1);  // QK commit (+ the dS readers)
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int x = 0; x < NB; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], kPing ? kWG : 2 * kWG);  // one or both softmax warpgroups
      mbar_init(&r_full[x], 1);
      mbar_init(&sr_free[x], kWG);
      mbar_init(&ds_full[x], kWG);
      mbar_init(&dsr_full[x], 1);
      mbar_init(&dsr_free[x], kWG);
      mbar_init(&aug_full[x], kWG);
      mbar_init(&aug_empty[x], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&ub_full[x], kWG);
      mbar_init(&ub_empty[x], 1);
    }
    for (int x = 0; x < 4; ++x) mbar_init(&mx_full[x], kWG);
    for (int x = 0; x < 2; ++x) mbar_init(&qb_full[x], kWG);
    mbar_init(qk_done, 1);
    mbar_init(pv_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kQkWarp) {
    tmem_alloc(s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  int *status = p.status;

  if (warp >= kProducerWarp) {
    reg_dealloc<kControlRegs>();
    if (warp == kProducerWarp && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      // Three streams walk the CTA's items: Q once per item (after the previous
      // item's last QK has run), K tiles up to KST ahead of V, V tiles.  The
      // thread never blocks on one stream while another could move; a stretch
      // of spin_limit cycles without progress is a timeout.
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int qn = 0, kn = 0, vn = 0;            // local item of the Q, K, V streams
      int kj = 0, vj = 0, gk = 0, gv = 0;    // tile within the item; global tile counters
      Item qit, kit, vit;
      if (blockIdx.x < p.items) qit = kit = vit = item_of<kVar>(p, blockIdx.x, BK);
      bool q_more = blockIdx.x < p.items, k_more = q_more, v_more = q_more;
      long long idle_since = clock64();
      while (k_more || v_more || q_more) {
        bool moved = false;
        if (q_more && qn <= kn && (qn == 0 || mbar_try_wait(q_empty, (qn - 1) & 1))) {
          mbar_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
          for (int c = 0; c < C::QK_CHUNKS; ++c)
            tma_load_2d(sQ + c * 128 * C::QK_SW, &tm_q, q_full, c * C::QK_SW, qit.bh * p.N_pad + qit.row0);
          ++qn;
          const int nx = blockIdx.x + qn * G;
          q_more = nx < p.items;
          if (q_more) qit = item_of<kVar>(p, nx, BK);
          moved = true;
        }
        if (k_more && gk < gv + KST && (gk < KST || mbar_try_wait(&k_empty[gk % KST], ((gk / KST) - 1) & 1))) {
          const int s = gk % KST;
          mbar_expect_tx(&k_full[s], C::K_BYTES);
#pragma unroll
          for (int c = 0; c < C::QK_CHUNKS; ++c)
            tma_load_2d(sK + s * C::K_BYTES + c * BK * C::QK_SW, &tm_k, &k_full[s], c * C::QK_SW,
                        kit.hkv * p.M_pad + kj * BK);
          ++gk;
          if (++kj == kit.T) {
            kj = 0;
            const int nx = blockIdx.x + (++kn) * G;
            k_more = nx < p.items;
            if (k_more) kit = item_of<kVar>(p, nx, BK);
          }
          moved = true;
        }
        if (v_more && gv < gk && (gv < VST || mbar_try_wait(&v_empty[gv % VST], ((gv / VST) - 1) & 1))) {
          const int s = gv % VST;
          mbar_expect_tx(&v_full[s], C::V_BYTES);
          tma_load_2d(sV + s * C::V_BYTES, &tm_v, &v_full[s], vj * BK * C::PV_EB, vit.hkv * D);
          ++gv;
          if (++vj == vit.T) {
            vj = 0;
            const int nx = blockIdx.x + (++vn) * G;
            v_more = nx < p.items;
            if (v_more) vit = item_of<kVar>(p, nx, BK);
          }
          moved = true;
        }
        if (moved) {
          idle_since = clock64();
        } else {
          if (*s_abort) break;
          if (clock64() - idle_since > p.spin) {
            if (atomicCAS(status, 0, SAGE_ERR_TIMEOUT) == 0) status[1] = 10;
            *s_abort = 1;
            break;
          }
          __nanosleep(32);
        }
      }
      // drain: every load this warp issued lands before the CTA exits
      volatile int no_abort = 0;
      if (qn > 0) mbar_wait(q_full, (qn - 1) & 1, status, 11, &no_abort, kDrainSpin);
      for (int j = max(0, gk - KST); j < gk; ++j) mbar_wait(&k_full[j % KST], (j / KST) & 1, status, 11, &no_abort, kDrainSpin);
      for (int j = max(0, gv - VST); j < gv; ++j) mbar_wait(&v_full[j % VST], (j / VST) & 1, status, 11, &no_abort, kDrainSpin);
    } else if (warp == kQkWarp) {
      // ---------------------------------------------------------- QK issuer (whole warp, one lane issues)
      // S goes to S/R region gt % NB once the accumulation has consumed the R of
      // tile gt - NB there; the Q buffer is released after an item's last QK.
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK);
      // test hook (SAGE_TEST_STALL): qk_done completes its first phase only
      // after this warp's final commit, so the wait runs out (at half the
      // limit, before any other wait of the CTA could) and the CTA unwinds
      bool ok = !p.stall || __all_sync(0xffffffffu, mbar_wait(qk_done, 0, status, 29, s_abort, p.spin >> 1));
      int gt = 0;
      // Q smoothing on the tensor core: dS^T(tile) = K^ q_bar^T into dS region
      // dg % NB as soon as the K^ tile has landed, kDsAhead tiles ahead of its QK.
      // The accumulation warpgroup turns it into the key augmentation of the
      // tile, and QK(tile) starts from [1/delta_Q] x [dS]^T (one TF32 step)
      // before adding Q^ K^T, so S arrives with dS / delta_Q folded in.  dS
      // stream: tile dg is tile dj of the CTA's item dn (dT tiles).
      int dg = 0, dn = 0, dj = 0, dT = 0;
      bool d_more = kDsMma && blockIdx.x < p.items;
      if (d_more) dT = item_of<kVar>(p, blockIdx.x, BK).T;
      auto issue_ds = [&]() -> bool {  // false: a wait failed
        const int b2 = dg % NB, s2 = dg % KST;
        // the item's q_bar tile and row augmentation, a free dS region, the K^ tile
        bool w = dj > 0 || mbar_wait(&ub_full[dn & 1], (dn >> 1) & 1, status, 26, s_abort, p.spin);
        if (dg >= NB) w = w && mbar_wait(&dsr_free[b2], ((dg - NB) / NB) & 1, status, 28, s_abort, p.spin);
        w = w && mbar_wait(&k_full[s2], (dg / KST) & 1, status, 21, s_abort, p.spin);
        if (!__all_sync(0xffffffffu, w)) return false;
        tc_fence_after();
        if (elect_one()) {
          // the K^ tile as A (128 keys), the item's q_bar tile as B (16 rows: hi, lo, zeros)
          const uint32_t u_base = smem_u32(sU) + (dn & 1) * C::UB_BYTES;
#pragma unroll
          for (int kk = 0; kk < C::QK_KSTEPS; ++kk) {
            const int byte = kk * 32;
            const uint32_t ak = k_base + s2 * C::K_BYTES + (byte / C::QK_SW) * BK * C::QK_SW + (byte % C::QK_SW);
            const uint32_t bu = u_base + (byte / C::QK_SW) * 16 * C::QK_SW + (byte % C::QK_SW);
            mma_f16(tmem + C::DS_COL + b2 * 16, smem_desc(ak, 8 * C::QK_SW, kSwizzle128),
                    smem_desc(bu, 8 * C::QK_SW, kSwizzle128), C::IDESC_DS, kk > 0);
          }
          mma_commit(&dsr_full[b2]);
        }
        __syncwarp();
        ++dg;
        if (++dj == dT) {
          dj = 0;
          const int nx = blockIdx.x + (++dn) * G;
          d_more = nx < p.items;
          if (d_more) dT = item_of<kVar>(p, nx, BK).T;
        }
        return true;
      };
      for (int n = 0; ok && blockIdx.x + n * G < p.items; ++n) {
        const Item it = item_of<kVar>(p, blockIdx.x + n * G, BK);
        if (!__all_sync(0xffffffffu, mbar_wait(q_full, n & 1, status, 23, s_abort, p.spin))) break;
        for (int j = 0; j < it.T; ++j, ++gt) {
          const int b = gt % NB, s = gt % KST;
          while (kDsMma && ok && d_more && dg <= gt + kDsAhead) ok = issue_ds();
          if (!ok) break;
          bool w = true;
          if (gt >= NB) w = mbar_wait(&sr_free[b], ((gt - NB) / NB) & 1, status, 20, s_abort, p.spin);
          if (kDsMma)  // the key augmentation (its K^ tile landed before its dS MMA)
            w = w && mbar_wait(&aug_full[b], (gt / NB) & 1, status, 30, s_abort, p.spin);
          else
            w = w && mbar_wait(&k_full[s], (gt / KST) & 1, status, 21, s_abort, p.spin);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            if constexpr (kDsMma)
              mma_tf32(tmem + b * C::SRW, smem_desc(smem_u32(sAq) + (n & 1) * C::AUG_BYTES, 256, kSwizzle32),
                       smem_desc(smem_u32(sAk) + b * C::AUG_BYTES, 256, kSwizzle32), C::IDESC_AUG, 0);
#pragma unroll
            for (int kk = 0; kk < C::QK_KSTEPS; ++kk) {
              const int byte = kk * 32;
              const uint32_t aq = q_base + (byte / C::QK_SW) * 128 * C::QK_SW + (byte % C::QK_SW);
              const uint32_t bk = k_base + s * C::K_BYTES + (byte / C::QK_SW) * BK * C::QK_SW + (byte % C::QK_SW);
              const uint64_t ad = smem_desc(aq, 8 * C::QK_SW, C::QK_SW == 128 ? kSwizzle128 : kSwizzle64);
              const uint64_t bd = smem_desc(bk, 8 * C::QK_SW, C::QK_SW == 128 ? kSwizzle128 : kSwizzle64);
              if (kQK16)
                mma_f16(tmem + b * C::SRW, ad, bd, C::IDESC_QK, kDsMma || kk > 0);
              else
                mma_f8(tmem + b * C::SRW, ad, bd, C::IDESC_QK, kk > 0);
            }
            mma_commit(&s_full[b]);
            if (kDsMma) mma_commit(&aug_empty[b]);
            mma_commit(&k_empty[s]);
            if (j == it.T - 1) {
              mma_commit(q_empty);  // Q^ may be replaced once these MMAs are done
              if (kDsMma) mma_commit(&ub_empty[n & 1]);  // and the item's q_bar tile and row augmentation
            }
          }
          __syncwarp();
        }
      }
      // every MMA of this thread has finished before the CTA may leave
      if (elect_one()) mma_commit(qk_done);
      __syncwarp();
      volatile int no_abort = 0;
      mbar_wait(qk_done, 0, status, 25, &no_abort, kDrainSpin);
    } else if (warp == kPvWarp) {
      // ---------------------------------------------------------- PV issuer (whole warp, one lane issues)
      // R = P^ V^, a fresh accumulator over one key tile, into S/R region gt % NB
      // once the softmax has read S there
      const uint32_t v_base = smem_u32(sV), p_base = smem_u32(sP);
      int gt = 0;
      bool ok = true;
      for (int n = 0; ok && blockIdx.x + n * G < p.items; ++n) {
        const Item it = item_of<kVar>(p, blockIdx.x + n * G, BK);
        for (int j = 0; j < it.T; ++j, ++gt) {
          const int b = gt % NB, s = gt % VST;
          const bool w = mbar_wait(&p_full[b], (gt / NB) & 1, status, 22, s_abort, p.spin) &&
                         mbar_wait(&v_full[s], (gt / VST) & 1, status, 24, s_abort, p.spin);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < C::PV_KSTEPS; ++kk) {
              const uint64_t ad = smem_desc(p_base + b * C::P_BYTES + kk * 32, 8 * C::PV_SW,
                                            C::PV_SW == 128 ? kSwizzle128 : kSwizzle64);
              const uint64_t bd = smem_desc(v_base + s * C::V_BYTES + kk * 32, 8 * C::PV_SW,
                                            C::PV_SW == 128 ? kSwizzle128 : kSwizzle64);
              if (kPV16)
                mma_f16(tmem + b * C::SRW, ad, bd, C::IDESC_PV, kk > 0);
              else
                mma_f8(tmem + b * C::SRW, ad, bd, C::IDESC_PV, kk > 0);
            }
            mma_commit(&r_full[b]);
            mma_commit(&v_empty[s]);
          }
          __syncwarp();
        }
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
    bool ok = true;
    int gt = 0;
    // dS stream (Q smoothing): tile dg = item dn, tile dj of it.  Before the
    // accumulation of tile gt the stream has produced dS up to tile gt + 1
    // (waiting for its K^ if need be) and tile gt + 2 as well when that K^ has
    // already landed: the wait on a K^ tile never holds up the accumulation
    // that the QK issuer needs to free an S/R region.  Buffer dg % NB was last
    // read by the softmax of tile dg - NB <= gt - 1, whose p_full this
    // warpgroup has waited for; K^ stage dg % KST goes back to the producer
    // after this read and the QK commit.  q_bar of item dn sits in
    // s_qb[dn & 1], published through qb_full[dn & 1]: every thread arrives
    // there after its last dS of item dn - 1, so no one still reads the
    // buffer's previous item dn - 2.  With the tensor-core dS the stream
    // reaches up to tile gt + 1 + kDsAhead, the tiles past gt + 1 only when
    // their dS and key-augmentation buffer are there already.
    static_assert(NB >= 3, "dS buffers: tiles gt + 1 and gt + 2 beside gt - 1");
    int dn = 0, dj = 0, dg = 0, dT = 0;
    const float *d_dk = nullptr;  // delta_K row of item dn
    bool d_more = smooth_q && blockIdx.x < p.items, qb_wait = d_more;
    auto ds_item = [&](int idx) {  // stage item idx of this CTA's list as item dn
      const Item t1 = item_of<kVar>(p, idx, BK);
      if constexpr (!kDsMma) {
        if (r < D) s_qb[(dn & 1) * D + r] = p.qbar[((size_t)t1.bh * p.Tm + t1.qi) * D + r];
        mbar_arrive(&qb_full[dn & 1]);
      }
      d_dk = p.dk + (size_t)t1.hkv * p.Tn;
      dT = t1.T;
    };
    // Tensor-core dS: the q_bar tile of item u (fp16 rows: hi = q_bar rounded
    // toward zero, lo = the rest rounded to nearest; |q_bar| < 2^16 by the
    // pre-pass range check, so hi + lo carries 22 bits) and the item's row
    // augmentation go into buffer u & 1 once the item u - 2 that used them has
    // had its last QK (ub_empty), and are published to the QK issuer through
    // ub_full (every thread arrives after its writes and a proxy fence).  Rows
    // 2..15 of the q_bar tile stay zero.  Row r of the augmentation holds
    // a = 1/u_r as TF32 hi, hi, lo, lo in its logical first 16 bytes and zeros
    // in the other 16 (u_r = delta_Q of the row, or 1 where that is 0: a block
    // whose smoothed Q codes are all zero); key c of the key augmentation holds
    // dS_c as hi, lo, hi, lo the same way.  The 32-byte swizzle exchanges the
    // two halves of rows 4..7 of every 8-row group (address bit 7 into bit 4),
    // so logical half 0 of row r is physical half (r >> 2) & 1; the other half
    // is zeroed once and never written.  un counts the items written so far.
    int un = 0;
    auto prep_ub = [&](int u, bool block) -> int {  // 1 written, 0 not yet, -1 wait failed
      if (u >= 2) {
        const uint32_t ph = ((u - 2) >> 1) & 1;
        const bool ready = block ? mbar_wait(&ub_empty[u & 1], ph, status, 44, s_abort, p.spin)
                                 : mbar_test_wait(&ub_empty[u & 1], ph);
        if (!__all_sync(0xffffffffu, ready)) return block ? -1 : 0;
      }
      const Item t = item_of<kVar>(p, blockIdx.x + u * G, BK);
      if (r < D) {
        const float qv = p.qbar[((size_t)t.bh * p.Tm + t.qi) * D + r];
        const __half hi = __float2half_rz(qv);
        const __half lo = __float2half_rn(qv - __half2float(hi));
        uint8_t *ub = sU + (u & 1) * C::UB_BYTES;
        const int byte = 2 * r, cc = byte / C::QK_SW, bb = byte % C::QK_SW;
        *reinterpret_cast<__half *>(ub + cc * 16 * C::QK_SW + swz_off<C::QK_SW>(0, bb / 16) + (bb & 15)) = hi;
        *reinterpret_cast<__half *>(ub + cc * 16 * C::QK_SW + swz_off<C::QK_SW>(1, bb / 16) + (bb & 15)) = lo;
      }
      {
        const float dq = (p.flags & SAGE_Q_PER_TOKEN) ? p.dqt[(size_t)t.bh * p.N_pad + t.row0 + r]
                                                      : p.dq[(size_t)t.bh * p.Tm + t.qi];
        const float a = 1.0f / (dq > 0.0f ? dq : 1.0f);
        const uint32_t ah = __float_as_uint(a) & kTf32Mask;
        const uint32_t al = __float_as_uint(a - __uint_as_float(ah)) & kTf32Mask;
        uint4 *row = reinterpret_cast<uint4 *>(sAq + (u & 1) * C::AUG_BYTES + r * 32);
        row[(r >> 2) & 1] = make_uint4(ah, ah, al, al);  // logical chunk 0; chunk 1 stays zero
      }
      fence_proxy_async_smem();
      mbar_arrive(&ub_full[u & 1]);
      return 1;
    };
    if constexpr (kDsMma) {
      // zero both q_bar tiles (rows 0 and 1 are rewritten per item) and the
      // augmentation buffers (only each row's logical chunk 0 is rewritten) once
      for (int i = r; i < (2 * C::UB_BYTES + (2 + NB) * C::AUG_BYTES) / 16; i += kWG)
        reinterpret_cast<uint4 *>(sU)[i] = make_uint4(0, 0, 0, 0);
      named_bar_sync(3, kWG);
    }
    if (d_more) ds_item(blockIdx.x);
    const float c2 = p.sm_log2;
    for (int n = 0; ok && blockIdx.x + n * G < p.items; ++n) {
      const Item it = item_of<kVar>(p, blockIdx.x + n * G, BK);
      float o[D];  // this thread's row of the FP32 running output
#pragma unroll
      for (int c = 0; c < D; ++c) o[c] = 0.0f;
      float lsum = 0.0f, mrow = 0.0f;
      for (int j = 0; j < it.T; ++j, ++gt) {
        const int b = gt % NB;
        while (kDsMma && d_more && dg < gt + 2 + kDsAhead) {
          // the key augmentation of tile dg from its dS^T = K^ q_bar^T in TMEM:
          // thread r takes key r, b = K^_r . q_bar split into TF32 hi + lo.
          // Up to tile gt + 1 the warpgroup waits for what it needs; beyond
          // that it takes a tile only if everything is there already
          const bool lazy = dg >= gt + 2;
          // the q_bar tiles: every item up to dn (waiting for a buffer unless
          // lazy) and item dn + 1 if its buffer is free; one call site keeps
          // this loop's code small
          int pr = 1;
          while (un <= dn + 1) {
            const bool need = un <= dn;
            if (!need && blockIdx.x + un * G >= p.items) break;  // no item dn + 1
            const int rv = prep_ub(un, need && !lazy);
            if (rv > 0) {
              ++un;
              continue;
            }
            if (need) pr = rv;  // 0: not yet (lazy), -1: the wait failed
            break;              // item dn + 1's buffer not free yet: later
          }
          if (pr < 0) {
            ok = false;
            break;
          }
          if (pr == 0) break;  // not yet: later
          const int b2 = dg % NB;
          const uint32_t ph = (dg / NB) & 1;
          // dS of the tile in TMEM; its buffer's previous tile dg - NB has had its QK
          const uint32_t pe = ((dg - NB) / NB) & 1;
          if (lazy) {
            if (!__all_sync(0xffffffffu, mbar_test_wait(&dsr_full[b2], ph) &&
                                             (dg < NB || mbar_test_wait(&aug_empty[b2], pe))))
              break;  // not yet: later
          } else if (!__all_sync(0xffffffffu, mbar_wait(&dsr_full[b2], ph, status, 42, s_abort, p.spin) &&
                                                  (dg < NB || mbar_wait(&aug_empty[b2], pe, status, 45, s_abort, p.spin)))) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t dh, dl;
          tmem_ld2(tmem + lane_off + C::DS_COL + b2 * 16, dh, dl);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&dsr_free[b2]);
          const float bv = __uint_as_float(dh) + __uint_as_float(dl);
          const uint32_t bh = __float_as_uint(bv) & kTf32Mask;
          const uint32_t bl = __float_as_uint(bv - __uint_as_float(bh)) & kTf32Mask;
          uint4 *row = reinterpret_cast<uint4 *>(sAk + b2 * C::AUG_BYTES + r * 32);
          row[(r >> 2) & 1] = make_uint4(bh, bl, bh, bl);  // logical chunk 0; chunk 1 stays zero
          fence_proxy_async_smem();
          mbar_arrive(&aug_full[b2]);
          ++dg;
          if (++dj == dT) {
            dj = 0;
            const int nx = blockIdx.x + (++dn) * G;
            d_more = nx < p.items;
            if (d_more) ds_item(nx);
          }
        }
        while (!kDsMma && d_more && dg < gt + 3) {
          // dS_j[c] = delta_K,j sum_d q_bar[d] K^_j[c, d], in t units: thread r takes key r
          const int s = dg % KST;
          const uint32_t ph = (dg / KST) & 1;
          if (dg == gt + 2) {
            if (!__all_sync(0xffffffffu, mbar_test_wait(&k_full[s], ph))) break;  // not yet: later
          } else if (!__all_sync(0xffffffffu, mbar_wait(&k_full[s], ph, status, 42, s_abort, p.spin))) {
            ok = false;
            break;
          }
          if (qb_wait) {
            if (!__all_sync(0xffffffffu, mbar_wait(&qb_full[dn & 1], (dn >> 1) & 1, status, 43, s_abort, p.spin))) {
              ok = false;
              break;
            }
            qb_wait = false;
          }
          if (r < BK)
            s_ds[(dg % NB) * BK + r] = qbar_dot_key<D, BK, kQK16>(sK + s * C::K_BYTES, s_qb + (dn & 1) * D, r) * d_dk[dj] * c2;
          mbar_arrive(&ds_full[dg % NB]);
          mbar_arrive(&k_empty[s]);
          ++dg;
          if (++dj == dT) {
            dj = 0;
            const int nx = blockIdx.x + (++dn) * G;
            d_more = nx < p.items;
            if (d_more) {
              ds_item(nx);
              qb_wait = true;
            }
          }
        }
        if (!ok) break;
        // alpha in shared memory once p_full says so, R in TMEM once r_full
        // does; the TMEM loads are warp-collective, so the warp decides together
        const bool waited = mbar_wait(&p_full[b], (gt / NB) & 1, status, 40, s_abort, p.spin) &&
                            mbar_wait(&r_full[b], (gt / NB) & 1, status, 41, s_abort, p.spin);
        if (!__all_sync(0xffffffffu, waited)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float a = s_alpha[b * 128 + r];
        if constexpr (kPing) {
          lsum = fmaf(a, lsum, s_l[b * 128 + r]);  // l from each tile's row sum
        } else if (j == it.T - 1) {
          lsum = s_l[(b * 2 + 0) * 128 + r] + s_l[(b * 2 + 1) * 128 + r];
          if constexpr (kPV16) mrow = s_mrow[b * 128 + r];
        }
        const float2 a2 = make_float2(a, a);
        // SageBwd: R holds integer sums of code products; s_P s_V,j scales them
        const float wv = kPV16 ? s_w[b * 128 + r] : 1.0f;
        const float2 w2 = make_float2(wv, wv);
        const uint32_t tR = tmem + lane_off + b * C::SRW;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t rv[32];
          tmem_ld32(tR + ch * 32, rv);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float2 r2 = make_float2(__uint_as_float(rv[e]), __uint_as_float(rv[e + 1]));
            if constexpr (kPV16) r2 = __fmul2_rn(r2, w2);
            const float2 o2 = __ffma2_rn(make_float2(o[ch * 32 + e], o[ch * 32 + e + 1]), a2, r2);
            o[ch * 32 + e] = o2.x;
            o[ch * 32 + e + 1] = o2.y;
          }
        }
        tc_fence_before();
        mbar_arrive(&sr_free[b]);
      }
      if (!ok) break;
      // epilogue of this item: O / l * delta_V (+ V_m) in bf16; SageBwd: O / l
      // (+ V_m), the scales being inside O, and the row's log-sum-exp
      // ln2 (m + log2 l) in the units of S sm_scale
      const int row = it.row0 + r;
      if (kPV16 && row < it.N) p.lse[(size_t)it.bh * p.N_pad + row] = (mrow + log2f(lsum)) * 0.6931471805599453f;
      if (row < it.N) {
        const float inv_l = 1.0f / lsum;
        const float *dv = p.dv + (size_t)it.hkv * D, *vm = p.vm + (size_t)it.hkv * D;
        // the output row: batched [B, Hq, N, d], or packed [total_q, Hq, d]
        __nv_bfloat16 *dst = kVar ? p.o + ((size_t)(it.q0 + row) * p.Hq + it.bh % p.Hq) * D
                                  : p.o + ((size_t)it.bh * p.N + row) * D;
#pragma unroll
        for (int c = 0; c < D; c += 8) {
          const float4 one4 = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
          const float4 dv0 = kPV16 ? one4 : __ldg(reinterpret_cast<const float4 *>(dv + c));
          const float4 dv1 = kPV16 ? one4 : __ldg(reinterpret_cast<const float4 *>(dv + c + 4));
          const float4 vm0 = __ldg(reinterpret_cast<const float4 *>(vm + c));
          const float4 vm1 = __ldg(reinterpret_cast<const float4 *>(vm + c + 4));
          const float dvs[8] = {dv0.x, dv0.y, dv0.z, dv0.w, dv1.x, dv1.y, dv1.z, dv1.w};
          const float vms[8] = {vm0.x, vm0.y, vm0.z, vm0.w, vm1.x, vm1.y, vm1.z, vm1.w};
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 v2 =
                __floats2bfloat162_rn(fmaf(o[c + 2 * e], dvs[2 * e] * inv_l, vms[2 * e]),
                                      fmaf(o[c + 2 * e + 1], dvs[2 * e + 1] * inv_l, vms[2 * e + 1]));
            w[e] = *reinterpret_cast<const uint32_t *>(&v2);
          }
          *reinterpret_cast<uint4 *>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  } else if constexpr (kPing) {
    reg_alloc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax, whole tiles in turn
    // Warpgroup w takes the key tiles gt with gt % 2 == w: all BK keys of its
    // 128 rows (one row per thread, its TMEM lane), streamed from TMEM in
    // 32-column chunks twice, the row maximum first, then the exponentials and
    // P^.  Only the running maximum passes between the warpgroups: tile gt
    // publishes m_gt (s_mx[gt % NB], mx_full[gt % NB]) as soon as it has its own
    // row maximum and m_gt-1, before its exponentials, so the other
    // warpgroup's next tile waits on a few instructions of this one.  Each
    // tile hands the accumulation warpgroup alpha and its row sum (s_l), from
    // which that warpgroup keeps l.  Buffer reuse: s_mx[b] of tile gt is read
    // by tile gt + 1 and next written by tile gt + NB, both of the same
    // warpgroup (NB odd); s_alpha / s_l as in the split form.
    static_assert(NB % 2 == 1, "the reader of a running maximum is its next writer");
    const int r = threadIdx.x & (kWG - 1);
    const int wg = warp >> 2;
    const uint32_t tS = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float c2 = p.sm_log2;
    bool stop = false;
    int gt = 0;
    for (int n = 0; !stop && blockIdx.x + n * G < p.items; ++n) {
      const Item it = item_of<kVar>(p, blockIdx.x + n * G, BK);
      const int diag = it.row0 + r + it.M - it.N;  // last key visible to this row (causal)
      const float dq0 = (p.flags & SAGE_Q_PER_TOKEN) ? p.dqt[(size_t)it.bh * p.N_pad + it.row0 + r]
                                                     : p.dq[(size_t)it.bh * p.Tm + it.qi];
      const float dq = (kDsMma && !(dq0 > 0.0f)) ? 1.0f : dq0;  // the unit S comes in (dS folded)
      const float *dkr = p.dk + (size_t)it.hkv * p.Tn;
      for (int j = 0; j < it.T; ++j, ++gt) {
        if ((gt & 1) != wg) continue;
        const int bb = gt % NB;
        const float dkj = dkr[j];  // in flight during the S wait
        const bool okw = mbar_wait(&s_full[bb], (gt / NB) & 1, status, 32, s_abort, p.spin) &&
                         (!kDsAdd || mbar_wait(&ds_full[bb], (gt / NB) & 1, status, 31, s_abort, p.spin));
        if (!__all_sync(0xffffffffu, okw)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const float k1 = dq * dkj * c2;  // S code -> t
        // x orders like t: the raw MMA output with the scale folded into the
        // exponent when k1 > 0 and there is no dS, else t itself (a masked -inf
        // never meets a 0)
        const bool raw = !kDsAdd && k1 > 0.0f;
        const float *dsc = s_ds + bb * BK;  // dS of the tile in t units (Q smoothing)
        const float xs = raw ? k1 : 1.0f;
        const bool edge = (j * BK + BK > it.M) || (p.causal && j * BK + BK - 1 > it.row0 + it.M - it.N);
        const int lim = (p.causal ? min(it.M, diag + 1) : it.M) - j * BK;  // keys at or past lim are masked
        const uint32_t tSb = tS + bb * C::SRW;
        // pass 1: the row maximum
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int ch = 0; ch < BK / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(tSb + ch * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float x = __uint_as_float(v[e]);
            if constexpr (kDsAdd)
              x = fmaf(x, k1, dsc[ch * 32 + e]);
            else if (!raw)
              x *= k1;
            if (edge && ch * 32 + e >= lim) x = -INFINITY;
            mq[e & 3] = fmaxf(mq[e & 3], x);
          }
        }
        const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        const float mt = (mx == -INFINITY) ? -INFINITY : mx * xs;  // row max of t over the tile
        // the running maximum: the previous tile's, from the other warpgroup
        float m_prev = -INFINITY;
        if (j > 0) {
          const int pb = (gt - 1) % NB;
          if (!__all_sync(0xffffffffu, mbar_wait(&mx_full[pb], ((gt - 1) / NB) & 1, status, 33, s_abort, p.spin))) {
            stop = true;
            break;
          }
          m_prev = s_mx[pb * 128 + r];
        }
        const float m_new = fmaxf(m_prev, mt);
        s_mx[bb * 128 + r] = m_new;
        mbar_arrive(&mx_full[bb]);
        const float alpha = (m_new == -INFINITY) ? 1.0f : ex2_approx(m_prev - m_new);
        // pass 2: P^ = e4m3(448 exp2(t - m_new)) with the 448 in the exponent's
        // bias; a row with nothing visible yet has only masked keys (-> 0)
        const float mb = (m_new == -INFINITY) ? INFINITY : m_new - kLog2_448;
        const float2 xs2 = make_float2(xs, xs), nb2 = make_float2(-mb, -mb);
        uint8_t *prow = sP + bb * C::P_BYTES;
        float2 rs2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int ch = 0; ch < BK / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(tSb + ch * 32, v);
          tmem_wait_ld();
          float pv[32];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x0 = __uint_as_float(v[e]), x1 = __uint_as_float(v[e + 1]);
            if constexpr (kDsAdd) {
              const float2 t2 = __ffma2_rn(make_float2(x0, x1), make_float2(k1, k1),
                                           *reinterpret_cast<const float2 *>(dsc + ch * 32 + e));
              x0 = t2.x;
              x1 = t2.y;
            } else if (!raw) {
              x0 *= k1;
              x1 *= k1;
            }
            if (edge) {
              x0 = (ch * 32 + e < lim) ? x0 : -INFINITY;
              x1 = (ch * 32 + e + 1 < lim) ? x1 : -INFINITY;
            }
            const float2 arg = __ffma2_rn(make_float2(x0, x1), xs2, nb2);
            pv[e] = ex2_approx(arg.x);
            pv[e + 1] = ex2_approx(arg.y);
            rs2 = __fadd2_rn(rs2, make_float2(pv[e], pv[e + 1]));
          }
          // keys 32 ch .. 32 ch + 31 are 16-byte chunks 2 ch and 2 ch + 1 of row r
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
              const int i0 = h * 16 + e;
              pk[e / 4] = (uint32_t)cvt_e4m3x2(pv[i0], pv[i0 + 1]) | ((uint32_t)cvt_e4m3x2(pv[i0 + 2], pv[i0 + 3]) << 16);
            }
            *reinterpret_cast<uint4 *>(prow + swz_off<C::PV_SW>(r, 2 * ch + h)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
        s_alpha[bb * 128 + r] = alpha;
        s_l[bb * 128 + r] = rs2.x + rs2.y;  // 448 times this tile's sum of P~, against m_new
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[bb]);
      }
    }
  } else {
    reg_alloc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax of one half of each key tile
    const int r = threadIdx.x & (kWG - 1);  // query row within the block == TMEM lane
    const int hf = warp >> 2;               // which half of the key tile
    const int oh = hf ^ 1;
    const uint32_t tS = tmem + ((uint32_t)((warp & 3) * 32) << 16) + hf * HALF;
    const float c2 = p.sm_log2;
    bool stop = false;  // a wait failed
    int gt = 0, bb = 0, pj = 0;
    for (int n = 0; !stop && blockIdx.x + n * G < p.items; ++n) {
      const Item it = item_of<kVar>(p, blockIdx.x + n * G, BK);
      const int diag = it.row0 + r + it.M - it.N;  // last key visible to this row (causal)
      // this row's Q scale: its own (per-token Q) or its block's
      const float dq0 = (p.flags & SAGE_Q_PER_TOKEN) ? p.dqt[(size_t)it.bh * p.N_pad + it.row0 + r]
                                                     : p.dq[(size_t)it.bh * p.Tm + it.qi];
      const float dq = (kDsMma && !(dq0 > 0.0f)) ? 1.0f : dq0;  // the unit S comes in (dS folded)
      float m = -INFINITY, l = 0.0f;
      const float *dkr = p.dk + (size_t)it.hkv * p.Tn;
      const float *dvbr = kPV16 ? p.dvb + (size_t)it.hkv * p.Tn : nullptr;  // SageBwd V block scales
      float dk_next = dkr[0];
      for (int j = 0; j < it.T; ++j, ++gt, bb = (bb + 1 == NB) ? 0 : bb + 1, pj ^= (bb == 0) ? 1 : 0) {
        const float dkj = dk_next;
        const float dvbj = kPV16 ? dvbr[j] : 0.0f;  // used at the tile's end, its latency hidden
        const float k1 = dq * dkj * c2;  // S code -> t
        // the TMEM loads are warp-collective: the warp decides together
        const bool okw = __all_sync(0xffffffffu, mbar_wait(&s_full[bb], pj, status, 32, s_abort, p.spin) &&
                                                     (!kDsAdd || mbar_wait(&ds_full[bb], pj, status, 31, s_abort, p.spin)));
        if (!okw) {
          stop = true;
          break;
        }
        tc_fence_after();
        if (j + 1 < it.T) dk_next = dkr[j + 1];  // the next tile's, its latency behind this tile
        // x: this half's scores in a domain that orders like t.  Without dS and
        // with k1 > 0 that is the raw MMA output (t = x k1, the scale folded
        // into the exponent below); otherwise t itself (xs = 1), so a masked
        // -inf never meets a zero scale.
        const bool raw = !kDsAdd && k1 > 0.0f;
        const float xs = raw ? k1 : 1.0f;
        float x[HALF];
        {
          uint32_t v[HALF];
#pragma unroll
          for (int ch = 0; ch < HALF / 32; ++ch)
            tmem_ld32(tS + bb * C::SRW + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[ch * 32]));
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < HALF; ++e) x[e] = __uint_as_float(v[e]);
        }
        if (!raw) {
          if (kDsAdd) {
            const float4 *dsc = reinterpret_cast<const float4 *>(s_ds + bb * BK + hf * HALF);
            const float2 k12 = make_float2(k1, k1);
#pragma unroll
            for (int e = 0; e < HALF; e += 4) {
              const float4 d4 = dsc[e / 4];
              const float2 t01 = __ffma2_rn(make_float2(x[e], x[e + 1]), k12, make_float2(d4.x, d4.y));
              const float2 t23 = __ffma2_rn(make_float2(x[e + 2], x[e + 3]), k12, make_float2(d4.z, d4.w));
              x[e] = t01.x;
              x[e + 1] = t01.y;
              x[e + 2] = t23.x;
              x[e + 3] = t23.y;
            }
          } else {
#pragma unroll
            for (int e = 0; e < HALF; ++e) x[e] *= k1;
          }
        }
        if (__builtin_expect((j * BK + BK > it.M) || (p.causal && j * BK + BK - 1 > it.row0 + it.M - it.N), 0)) {
          // edge tile: keys at or past lim are invisible to this row
          const int lim = (p.causal ? min(it.M, diag + 1) : it.M) - j * BK - hf * HALF;
#pragma unroll
          for (int e = 0; e < HALF; ++e) x[e] = (e < lim) ? x[e] : -INFINITY;
        }
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < HALF; e += 8) {
          mq[0] = fmax3(mq[0], x[e], x[e + 1]);
          mq[1] = fmax3(mq[1], x[e + 2], x[e + 3]);
          mq[2] = fmax3(mq[2], x[e + 4], x[e + 5]);
          mq[3] = fmax3(mq[3], x[e + 6], x[e + 7]);
        }
        const float mh = fmax3(fmaxf(mq[0], mq[1]), mq[2], mq[3]);
        s_mx[((gt & 1) * 2 + hf) * 128 + r] = mh;
        mbar_arrive(&mx_full[(gt & 1) * 2 + hf]);
        // e = exp2(t - m_half) in place
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
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&mx_full[(gt & 1) * 2 + oh], (gt >> 1) & 1, status, 33, s_abort, p.spin))) {
          stop = true;
          break;
        }
        const float mt = fmaxf(mh * xs, s_mx[((gt & 1) * 2 + oh) * 128 + r] * xs);  // row max of t over the tile
        const float m_new = fmaxf(m, mt);
        const float alpha = (m_new == -INFINITY) ? 1.0f : ex2_approx(m - m_new);
        if constexpr (kPV16) {
          uint8_t *prow = sP + bb * C::P_BYTES;
          // SageBwd (SageAttention3 summary, "SageBwd Forward Pass"): one P~
          // scale per row and tile, s_P = exp2(m_tile - m_new) / 127, so
          // P^ = rint(P~ / s_P) = rint(127 exp2(t - m_tile)) = rint(e g3); the
          // codes go out as fp16 integers, 8 keys per 16-byte chunk
          const float g3 = (mh == -INFINITY) ? 0.0f : 127.0f * ex2_approx(mht - mt);
          const float2 g32 = make_float2(g3, g3);
#pragma unroll
          for (int ch = 0; ch < HALF / 8; ++ch) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const float2 p2 = __fmul2_rn(make_float2(x[ch * 8 + e], x[ch * 8 + e + 1]), g32);
              const __half2 h = __floats2half2_rn(fminf(rintf(p2.x), 127.0f), fminf(rintf(p2.y), 127.0f));
              pk[e / 2] = *reinterpret_cast<const uint32_t *>(&h);
            }
            // keys hf HALF + 8 ch .. +7 are 16-byte chunk (hf HALF / 8 + ch) of row r
            *reinterpret_cast<uint4 *>(prow + swz_off<C::PV_SW>(r, hf * (HALF / 8) + ch)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
          // l sums the unquantized P~ = e exp2(m_half - m_new)
          const float u = (mh == -INFINITY) ? 0.0f : ex2_approx(mht - m_new);
          l = fmaf(alpha, l, u * (se2.x + se2.y));
          if (hf == 0) s_w[bb * 128 + r] = (mt == -INFINITY) ? 0.0f : ex2_approx(mt - m_new) * (1.0f / 127.0f) * dvbj;
          if (hf == 0 && j == it.T - 1) s_mrow[bb * 128 + r] = m_new;
        } else {
        // P^ = e4m3(448 exp2(t - m_new)) = e4m3(e g)
        const float g = (mh == -INFINITY) ? 0.0f : ex2_approx(mht - m_new + kLog2_448);
        const float2 g2 = make_float2(g, g);
        uint8_t *prow = sP + bb * C::P_BYTES;
#pragma unroll
        for (int ch = 0; ch < HALF / 16; ++ch) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const int i0 = ch * 16 + e;
            const float2 p01 = __fmul2_rn(make_float2(x[i0], x[i0 + 1]), g2);
            const float2 p23 = __fmul2_rn(make_float2(x[i0 + 2], x[i0 + 3]), g2);
            pk[e / 4] = (uint32_t)cvt_e4m3x2(p01.x, p01.y) | ((uint32_t)cvt_e4m3x2(p23.x, p23.y) << 16);
          }
          // keys hf HALF + 16 ch .. +15 are 16-byte chunk (hf HALF / 16 + ch) of row r
          *reinterpret_cast<uint4 *>(prow + swz_off<C::PV_SW>(r, hf * (HALF / 16) + ch)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        l = fmaf(alpha, l, g * (se2.x + se2.y));  // 448 times this half's sum of P~
        }
        m = m_new;
        if (hf == 0) s_alpha[bb * 128 + r] = alpha;
        if (j == it.T - 1) s_l[(bb * 2 + hf) * 128 + r] = l;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[bb]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kQkWarp) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, int BK, bool kQK16, bool kPV16, bool kPing, bool kVar>
sage_status launch_t(const sage_shape &s, int causal, float sm_scale, int flags, const void *ws,
                     const sage_ws_layout &L, void *o, cudaStream_t stream, const VarDev &var) {
  using C = Cfg<D, BK, kQK16, false, kPV16>;
  const char *w = (const char *)ws;
  CUtensorMap tq, tk, tv;
  sage_status st;
  st = make_tmap_2d(&tq, w + L.qhat, C::ROWB, (uint64_t)s.B * s.Hq * L.N_pad, C::ROWB, C::QK_SW, 128, C::QK_SW);
  if (st != SAGE_OK) return st;
  st = make_tmap_2d(&tk, w + L.khat, C::ROWB, (uint64_t)s.B * s.Hkv * L.M_pad, C::ROWB, C::QK_SW, BK, C::QK_SW);
  if (st != SAGE_OK) return st;
  st = make_tmap_2d(&tv, w + L.vhat, (uint64_t)L.M_pad * C::PV_EB, (uint64_t)s.B * s.Hkv * D,
                    (uint64_t)L.M_pad * C::PV_EB, BK * C::PV_EB, D, C::PV_SW);
  if (st != SAGE_OK) return st;
  AttnParams p;
  p.N = s.N;
  p.M = s.M;
  p.N_pad = L.N_pad;
  p.M_pad = L.M_pad;
  p.Tm = L.Tm;
  p.Tn = L.Tn;
  p.items = var.item_tab ? var.items : s.B * s.Hq * L.Tm;
  p.item_tab = var.item_tab;
  p.seq = var.seq;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.causal = causal ? 1 : 0;
  p.flags = flags;
  p.sm_log2 = sm_scale * 1.4426950408889634f;
  p.dq = (const float *)(w + L.dq);
  p.dqt = (const float *)(w + L.dqt);
  p.dvb = (const float *)(w + L.dvb);
  p.lse = (float *)(w + L.lse);
  p.qbar = (const float *)(w + L.qbar);
  p.dk = (const float *)(w + L.dk);
  p.dv = (const float *)(w + L.dv);
  p.vm = (const float *)(w + L.vm);
  p.o = (__nv_bfloat16 *)o;
  p.status = (int *)(w + L.status);
  p.spin = spin_limit_cycles();
  p.stall = test_stall();
  const bool sq = (flags & SAGE_SMOOTH_Q) != 0;
  auto kern = sq ? attn_q8_kernel<D, BK, kQK16, true, kPV16, kPing, kVar>
                 : attn_q8_kernel<D, BK, kQK16, false, kPV16, kPing, kVar>;
  // the Q-smoothing instance with INT8 codes and 128-key tiles holds the q_bar tiles too
  const int smem = sq ? Cfg<D, BK, kQK16, kQK16 && BK == 128, kPV16>::SMEM_TOTAL : C::SMEM_TOTAL;
  // the register split needs the launch allocation it was computed for
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return SAGE_ERR_CUDA;
  if (fa.numRegs != kLaunchRegs) return SAGE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SAGE_ERR_CUDA;
  // one persistent CTA per SM (fewer when there are fewer items)
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      return SAGE_ERR_CUDA;
  }
  const int grid = p.items < sms ? p.items : sms;
  if (grid <= 0) return SAGE_OK;  // no work item (packed sequences without queries are rejected earlier)
  if (p.causal && !var.item_tab) {
    if (p.items >= (1 << 24)) return SAGE_ERR_UNSUPPORTED;  // causal_item divides in fp32
    CausalOrder &z = p.cz;
    const int BH = p.items / p.Tm, NP = BH * (p.Tm / 2), R = NP / grid;
    z.G = grid;
    z.PH = p.Tm / 2;
    z.full = 2 * R * grid;
    z.rest = NP - R * grid;
    z.mid = (p.Tm & 1) ? BH : 0;
    z.invG = 1.0f / (float)grid;
    z.invPH = z.PH > 0 ? 1.0f / (float)z.PH : 0.0f;
  }
  kern<<<(unsigned)grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}


// The launcher instance of a request: SageBwd (64-key tiles), else by head
// dim, key tile and INT8 / E4M3 Q and K.  kPing: whole key tiles in turn
// (not for the SageBwd forward).  kVar: packed sequences.
template <bool kPing, bool kVar>
sage_status dispatch_q8(const sage_shape &s, int causal, float sm_scale, int mode, int flags, int bk,
                        const void *ws, const sage_ws_layout &L, void *o, cudaStream_t stream, const VarDev &var) {
  if (mode == SAGE_SAGEBWD_I8) {  // INT8 codes throughout, 64-key tiles (checked by the caller)
    if constexpr (kPing) {
      return SAGE_ERR_UNSUPPORTED;
    } else {
      if (bk != 64) return SAGE_ERR_UNSUPPORTED;
      return s.d == 64 ? launch_t<64, 64, true, true, false, kVar>(s, causal, sm_scale, flags, ws, L, o, stream, var)
                       : launch_t<128, 64, true, true, false, kVar>(s, causal, sm_scale, flags, ws, L, o, stream, var);
    }
  }
  const bool i8 = (mode == SAGE_Q8_PV8);
  if (s.d == 64) {
    if (bk == 64)
      return i8 ? launch_t<64, 64, true, false, kPing, kVar>(s, causal, sm_scale, flags, ws, L, o, stream, var)
                : launch_t<64, 64, false, false, kPing, kVar>(s, causal, sm_scale, flags, ws, L, o, stream, var);
    return i8 ? launch_t<64, 128, true, false, kPing, kVar>(s, causal, sm_scale, flags, ws, L, o, stream, var)
              : launch_t<64, 128, false, false, kPing, kVar>(s, causal, sm_scale, flags, ws, L, o, stream, var);
  }
  if (bk == 64)
    return i8 ? launch_t<128, 64, true, false, kPing, kVar>(s, causal, sm_scale, flags, ws, L, o, stream, var)
              : launch_t<128, 64, false, false, kPing, kVar>(s, causal, sm_scale, flags, ws, L, o, stream, var);
  return i8 ? launch_t<128, 128, true, false, kPing, kVar>(s, causal, sm_scale, flags, ws, L, o, stream, var)
            : launch_t<128, 128, false, false, kPing, kVar>(s, causal, sm_scale, flags, ws, L, o, stream, var);
}

}  // namespace
}  // namespace sage
