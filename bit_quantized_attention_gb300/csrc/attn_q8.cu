// Fused quantized attention for the INT8 / FP8 modes on sm_103a.
//
// What it computes, per query block i of 128 rows of one (b, q-head), over the
// key tiles j = 0..T-1 of its kv-head (SageAttention2 Technical Report summary
// §3.4 "The Complete Algorithm"; "Quantization for Attention, in depth",
// "The datapath and its quantize points"):
//   S_ij  = delta_Q delta_K,j (Q^_i K^_j^T) + dS_ij,  dS_ij = q_bar_i deq(K^_j)^T
//   m_ij  = max(m_i,j-1, rowmax S_ij * sm_scale)
//   P~_ij = exp(S_ij sm_scale - m_ij),  l_ij = e^(m_i,j-1 - m_ij) l + rowsum P~
//   P^_ij = e4m3(448 P~_ij)                          (static scale 1/448)
//   R_ij  = P^_ij V^_j        (tile partial, accumulated over this tile only)
//   O_ij  = e^(m_i,j-1 - m_ij) O_i,j-1 + R_ij        (FP32 running output)
//   O_i   = O / l * delta_V / 448 (+ V_m)
// Scores are handled in the base-2 domain (sm_scale * log2 e folded into the
// dequantization multiply) and the 448 of P^ is folded into the exponent, so
// l carries 448 * sum P~ and the final scale is delta_V / l.
//
// GB300 mapping (the pages' Ada/Hopper register-level design is prior art).
// Each CTA owns two query blocks (tiles t = 0, 1) of one head; every K^/V^
// tile is loaded once for both.  Four warpgroups:
//   WG0, WG1   softmax of tile 0 / tile 1, one query row per thread (its TMEM
//              lane): the whole score row in one TMEM read, dequant + dS, mask,
//              online max / sum, P^ to shared memory (the swizzled K-major A
//              operand of the next MMA), alpha and l to shared memory
//   WG2        two-level accumulation for both tiles: R from TMEM, O from TMEM,
//              O = alpha O + R in FP32, O back to TMEM; then the epilogue
//   WG3        warp 12: TMA producer (Q^ tiles once, K^_j / V^T_j into a ring
//              of shared-memory stages); warp 13: the tcgen05 MMA issuer (one
//              thread): S_t = Q^_t K^_j^T (kind::f16 on INT8 codes held as
//              exact fp16 integers — sm_103a has no INT8 tensor path — or
//              kind::f8f6f4 on E4M3 codes) and R_t = P^_t V^_j (kind::f8f6f4)
// TMEM (512 columns): per tile one region that holds S_t(j) and then, once the
// softmax has read it, the tile partial R_t(j) (a fresh accumulator, zeroed by
// its first k-step), and the FP32 running output O_t.  While one tile is in its
// softmax or correction, the tensor core runs the other tile's MMAs.
// Waits suspend the waiting thread instead of polling and are bounded: on
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

constexpr int kWG = 128;       // threads per warpgroup
constexpr int kThreads = 512;  // softmax x2, correction, control
constexpr int kCorrWarp0 = 8, kProducerWarp = 12, kMmaWarp = 13;
// Register split (setmaxnreg) from the 128 per thread the block launches with:
// the softmax warpgroups rise, the correction and control warpgroups drop.
constexpr int kLaunchRegs = 128, kSoftmaxRegs = 184, kCorrRegs = 88, kControlRegs = 56;
static_assert(2 * kWG * kSoftmaxRegs + kWG * kCorrRegs + kWG * kControlRegs <= kThreads * kLaunchRegs,
              "register split");
static_assert(kSoftmaxRegs >= kLaunchRegs && kCorrRegs <= kLaunchRegs && kControlRegs <= kLaunchRegs,
              "register split directions");
constexpr float kLog2_448 = 8.807354922057604f;

template <int D, int BK, bool kQK16>
struct Cfg {
  static constexpr int QK_EB = kQK16 ? 2 : 1;           // bytes per stored Q/K code
  static constexpr int ROWB = D * QK_EB;                 // bytes per Q/K row
  static constexpr int QK_SW = ROWB >= 128 ? 128 : 64;   // swizzle span of Q/K tiles
  static constexpr int QK_CHUNKS = ROWB / QK_SW;         // swizzle spans per row
  static constexpr int PV_SW = BK >= 128 ? 128 : 64;     // swizzle span of P^ and V^T tiles
  static constexpr int Q_BYTES = 128 * ROWB;
  static constexpr int K_BYTES = BK * ROWB;
  static constexpr int V_BYTES = D * BK;
  static constexpr int P_BYTES = 128 * BK;
  static constexpr int QK_KSTEPS = ROWB / 32;            // one MMA consumes 32 bytes of K
  static constexpr int PV_KSTEPS = BK / 32;
  static constexpr int FIXED = 2 * Q_BYTES + 2 * P_BYTES;
  static constexpr int ST_FIT = (216 * 1024 - FIXED) / (K_BYTES + V_BYTES);
  static constexpr int STAGES = ST_FIT > 4 ? 4 : ST_FIT;
  static_assert(STAGES >= 2, "shared memory budget");
  static constexpr int SRW = BK > D ? BK : D;            // columns of the S / R region of a tile
  static constexpr int TMEM_O = 2 * SRW;                 // O_t at TMEM_O + t * D
  static constexpr int TMEM_NEED = 2 * SRW + 2 * D;
  static constexpr int TMEM_COLS = TMEM_NEED <= 256 ? 256 : 512;
  static_assert(TMEM_NEED <= 512, "tensor memory budget");
  static constexpr int SMEM_TILES = FIXED + STAGES * (K_BYTES + V_BYTES);
  static constexpr int SMEM_MISC = (4 * BK + 4 * D + 4 * 128) * 4 + (1 + 3 * STAGES + 8 + 1) * 8 + 16;
  static constexpr int SMEM_TOTAL = 1024 + SMEM_TILES + SMEM_MISC;
  static constexpr uint32_t IDESC_QK =
      instr_desc(kFmtF32, kQK16 ? kFmtF16 : kFmtE4M3, kQK16 ? kFmtF16 : kFmtE4M3, BK, 128);
  static constexpr uint32_t IDESC_PV = instr_desc(kFmtF32, kFmtE4M3, kFmtE4M3, D, 128);
};

struct AttnParams {
  int N, M, N_pad, M_pad, Tm, Tm2, Tn, Hq, Hkv, causal, flags;
  float sm_log2;  // sm_scale * log2(e)
  const float *dq, *qbar, *dk, *dv, *vm;
  __nv_bfloat16 *o;
  int *status;
  long long spin;
};

// byte offset of 16-byte chunk `c` of row `r` in a K-major swizzled tile whose
// rows are `SW` bytes wide (8-row atoms of 8*SW bytes, 1024-aligned base)
template <int SW>
__device__ __forceinline__ uint32_t swz_off(int r, int c) {
  const int x = (SW == 128) ? (r & 7) : ((r & 7) >> 1);
  return (uint32_t)((r >> 3) * (8 * SW) + (r & 7) * SW + ((c ^ x) << 4));
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

template <int D, int BK, bool kQK16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_q8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D, BK, kQK16>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = base;                        // 2 query tiles
  uint8_t *sP = sQ + 2 * C::Q_BYTES;         // P^ of each query tile
  uint8_t *sK = sP + 2 * C::P_BYTES;         // ST stages
  uint8_t *sV = sK + ST * C::K_BYTES;        // ST stages
  float *s_dsc = (float *)(sV + ST * C::V_BYTES);  // [2 tiles][2 buffers][BK]
  float *s_qbar = s_dsc + 4 * BK;                  // [2][D]
  float *s_dv = s_qbar + 2 * D;                    // [D]
  float *s_vm = s_dv + D;                          // [D]
  float *s_alpha = s_vm + D;                       // [2][128] rescale factor of the current tile
  float *s_l = s_alpha + 2 * 128;                  // [2][128] final row sums
  uint64_t *bars = (uint64_t *)(((uintptr_t)(s_l + 2 * 128) + 7) & ~(uintptr_t)7);
  uint64_t *q_full = bars;
  uint64_t *k_full = q_full + 1;
  uint64_t *v_full = k_full + ST;
  uint64_t *kv_empty = v_full + ST;
  uint64_t *s_full = kv_empty + ST;  // [2] S_t ready in TMEM
  uint64_t *p_full = s_full + 2;     // [2] P^_t, alpha_t written; S_t read
  uint64_t *r_full = p_full + 2;     // [2] R_t ready in TMEM
  uint64_t *sr_free = r_full + 2;    // [2] R_t folded into O_t; region free
  uint64_t *mma_done = sr_free + 2;
  uint32_t *s_tmem = (uint32_t *)(mma_done + 1);
  volatile int *s_abort = (volatile int *)(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x / p.Tm2;
  const int pair = p.Tm2 - 1 - blockIdx.x % p.Tm2;  // heaviest causal blocks first
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int hkv = b * p.Hkv + h / (p.Hq / p.Hkv);
  // key tiles each query tile needs (0 when the tile is past the last block)
  int Tt[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qi = 2 * pair + t;
    if (qi >= p.Tm) {
      Tt[t] = 0;
    } else {
      const int last_row = min(p.N, qi * 128 + 128) - 1;
      Tt[t] = p.causal ? min(p.Tn, (last_row + p.M - p.N) / BK + 1) : p.Tn;
    }
  }
  const int T = max(Tt[0], Tt[1]);
  const bool smooth_q = (p.flags & SAGE_SMOOTH_Q) != 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], kWG);
      mbar_init(&r_full[t], 1);
      mbar_init(&sr_free[t], kWG);
    }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x < 2 * kWG) {
    const int t = threadIdx.x / kWG, c0 = threadIdx.x % kWG;
    const int qi = min(2 * pair + t, p.Tm - 1);
    for (int c = c0; c < D; c += kWG) {
      s_qbar[t * D + c] = smooth_q ? p.qbar[((size_t)bh * p.Tm + qi) * D + c] : 0.0f;
      if (t == 0) {
        s_dv[c] = p.dv[(size_t)hkv * D + c];
        s_vm[c] = p.vm[(size_t)hkv * D + c];
      }
    }
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
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int nq = Tt[1] > 0 ? 2 : 1;
      mbar_expect_tx(q_full, nq * C::Q_BYTES);
      for (int t = 0; t < nq; ++t)
#pragma unroll
        for (int c = 0; c < C::QK_CHUNKS; ++c)
          tma_load_2d(sQ + t * C::Q_BYTES + c * 128 * C::QK_SW, &tm_q, q_full, c * C::QK_SW,
                      bh * p.N_pad + (2 * pair + t) * 128);
      int issued = 0;
      for (int j = 0; j < T; ++j) {
        const int s = j % ST, n = j / ST;
        if (j >= ST && !mbar_wait(&kv_empty[s], (n - 1) & 1, status, 10, s_abort, p.spin)) break;
        mbar_expect_tx(&k_full[s], C::K_BYTES);
#pragma unroll
        for (int c = 0; c < C::QK_CHUNKS; ++c)
          tma_load_2d(sK + s * C::K_BYTES + c * BK * C::QK_SW, &tm_k, &k_full[s], c * C::QK_SW,
                      hkv * p.M_pad + j * BK);
        mbar_expect_tx(&v_full[s], C::V_BYTES);
        tma_load_2d(sV + s * C::V_BYTES, &tm_v, &v_full[s], j * BK, hkv * D);
        issued = j + 1;
      }
      // drain: every load this warp issued must land before the CTA exits
      volatile int no_abort = 0;
      mbar_wait(q_full, 0, status, 11, &no_abort, p.spin);
      for (int j = max(0, issued - ST); j < issued; ++j) {
        const int s = j % ST, n = j / ST;
        mbar_wait(&k_full[s], n & 1, status, 11, &no_abort, p.spin);
        mbar_wait(&v_full[s], n & 1, status, 11, &no_abort, p.spin);
      }
    } else if (warp == kMmaWarp && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV), p_base = smem_u32(sP);
      bool ok = mbar_wait(q_full, 0, status, 23, s_abort, p.spin);
      tc_fence_after();
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % ST;
        // S_t(j) = Q^_t K^_j^T into the tile's S/R region, once R_t(j-1) is folded into O_t
        for (int t = 0; ok && t < 2; ++t) {
          if (j >= Tt[t]) continue;
          if (j >= 1 && !mbar_wait(&sr_free[t], (j - 1) & 1, status, 20, s_abort, p.spin)) ok = false;
          if (ok && !mbar_wait(&k_full[s], (j / ST) & 1, status, 21, s_abort, p.spin)) ok = false;
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C::QK_KSTEPS; ++kk) {
            const int byte = kk * 32;
            const uint32_t aq = q_base + t * C::Q_BYTES + (byte / C::QK_SW) * 128 * C::QK_SW + (byte % C::QK_SW);
            const uint32_t bk = k_base + s * C::K_BYTES + (byte / C::QK_SW) * BK * C::QK_SW + (byte % C::QK_SW);
            const uint64_t ad = smem_desc(aq, 8 * C::QK_SW, C::QK_SW == 128 ? kSwizzle128 : kSwizzle64);
            const uint64_t bd = smem_desc(bk, 8 * C::QK_SW, C::QK_SW == 128 ? kSwizzle128 : kSwizzle64);
            if (kQK16)
              mma_f16(tmem + t * C::SRW, ad, bd, C::IDESC_QK, kk > 0);
            else
              mma_f8(tmem + t * C::SRW, ad, bd, C::IDESC_QK, kk > 0);
          }
          mma_commit(&s_full[t]);
        }
        // R_t(j) = P^_t V^_j, a fresh accumulator over this key tile only
        for (int t = 0; ok && t < 2; ++t) {
          if (j >= Tt[t]) continue;
          if (!mbar_wait(&p_full[t], j & 1, status, 22, s_abort, p.spin)) ok = false;
          if (ok && !mbar_wait(&v_full[s], (j / ST) & 1, status, 24, s_abort, p.spin)) ok = false;
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C::PV_KSTEPS; ++kk) {
            const uint64_t ad = smem_desc(p_base + t * C::P_BYTES + kk * 32, 8 * C::PV_SW,
                                          C::PV_SW == 128 ? kSwizzle128 : kSwizzle64);
            const uint64_t bd = smem_desc(v_base + s * C::V_BYTES + kk * 32, 8 * C::PV_SW,
                                          C::PV_SW == 128 ? kSwizzle128 : kSwizzle64);
            mma_f8(tmem + t * C::SRW, ad, bd, C::IDESC_PV, kk > 0);
          }
          mma_commit(&r_full[t]);
        }
        if (ok) mma_commit(&kv_empty[s]);
      }
      // drain: all MMAs this thread issued complete before TMEM is freed
      mma_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, status, 25, &no_abort, p.spin);
    }
  } else if (warp >= kCorrWarp0) {
    reg_dealloc<kCorrRegs>();
    // ------------------------------------------------------------ two-level accumulation + epilogue
    const int r = threadIdx.x & (kWG - 1);
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    for (int j = 0; ok && j < T; ++j) {
      for (int t = 0; ok && t < 2; ++t) {
        if (j >= Tt[t]) continue;
        // alpha_t(j) is in shared memory once p_full says so; R_t(j) once r_full does.
        // The TMEM loads and stores below are warp-collective, so the warp decides
        // together whether to go on.
        const bool waited = mbar_wait(&p_full[t], j & 1, status, 40, s_abort, p.spin) &&
                            mbar_wait(&r_full[t], j & 1, status, 41, s_abort, p.spin);
        if (!__all_sync(0xffffffffu, waited)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float a = s_alpha[t * 128 + r];
        const uint32_t tR = tmem + lane_off + t * C::SRW;
        const uint32_t tO = tmem + lane_off + C::TMEM_O + t * D;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t rv[32], ov[32];
          tmem_ld32(tR + ch * 32, rv);
          if (j > 0) tmem_ld32(tO + ch * 32, ov);
          tmem_wait_ld();
          if (j > 0) {
            const float2 aa = f2(a, a);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 o2 = __ffma2_rn(f2(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1])), aa,
                                           f2(__uint_as_float(rv[e]), __uint_as_float(rv[e + 1])));
              ov[e] = __float_as_uint(o2.x);
              ov[e + 1] = __float_as_uint(o2.y);
            }
            tmem_st32(tO + ch * 32, ov);
          } else {
            tmem_st32(tO + ch * 32, rv);  // O_t(0) = R_t(0)
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sr_free[t]);
      }
    }
    // epilogue: O / l * delta_V (+ V_m) in bf16, one row per thread.  Every lane
    // takes part in the (warp-collective) TMEM loads; only rows < N are stored.
    for (int t = 0; ok && t < 2; ++t) {
      if (Tt[t] == 0) continue;
      const int row = (2 * pair + t) * 128 + r;
      const bool live = row < p.N;
      const float inv_l = live ? 1.0f / s_l[t * 128 + r] : 0.0f;
      const uint32_t tO = tmem + lane_off + C::TMEM_O + t * D;
      __nv_bfloat16 *dst = p.o + ((size_t)bh * p.N + (live ? row : 0)) * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        tmem_ld32(tO + ch * 32, ov);
        tmem_wait_ld();
        if (!live) continue;
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int cc = ch * 32 + c + 2 * e;
            const float o0 = fmaf(__uint_as_float(ov[c + 2 * e]), s_dv[cc] * inv_l, s_vm[cc]);
            const float o1 = fmaf(__uint_as_float(ov[c + 2 * e + 1]), s_dv[cc + 1] * inv_l, s_vm[cc + 1]);
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(o0, o1);
            w[e] = *reinterpret_cast<const uint32_t *>(&v2);
          }
          *reinterpret_cast<uint4 *>(dst + ch * 32 + c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  } else {
    reg_alloc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax of tile t
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int r = threadIdx.x & (kWG - 1);   // query row within the tile == TMEM lane
    const int T_t = Tt[t];
    const uint32_t sS = tmem + ((uint32_t)((warp & 3) * 32) << 16) + t * C::SRW;
    const int qi = 2 * pair + t;
    const int row0 = qi * 128;
    const int diag = row0 + r + p.M - p.N;  // last key visible to this row (causal)
    const float c2 = p.sm_log2;
    const float dq = (T_t > 0) ? p.dq[(size_t)bh * p.Tm + qi] : 0.0f;
    // dS of key tile j lives in buffer j & 1: a thread writing tile j+1 cannot
    // overwrite values a slower thread of the warpgroup still reads for tile j
    float *dsc_t = s_dsc + t * 2 * BK;
    const float *qbar = s_qbar + t * D;
    uint8_t *prow = sP + t * C::P_BYTES;
    float m = -INFINITY, l = 0.0f;
    for (int j = 0; j < T_t; ++j) {
      const int s = j % ST;
      const float dkj = p.dk[(size_t)hkv * p.Tn + j];
      const float k1 = dq * dkj * c2;
      float *dsc = dsc_t + (j & 1) * BK;
      if (smooth_q) {
        // dS_j[c] = delta_K,j * sum_d q_bar[d] K^_j[c, d]: one key column per thread
        bool fail = !mbar_wait(&k_full[s], (j / ST) & 1, status, 31, s_abort, p.spin);
        if (!fail && r < BK) {
          const uint8_t *kt = sK + s * C::K_BYTES;
          float acc = 0.0f;
#pragma unroll
          for (int cc = 0; cc < C::QK_CHUNKS; ++cc) {
#pragma unroll
            for (int c16 = 0; c16 < C::QK_SW / 16; ++c16) {
              const uint4 w = *reinterpret_cast<const uint4 *>(kt + cc * BK * C::QK_SW + swz_off<C::QK_SW>(r, c16));
              const int d0 = (cc * C::QK_SW + c16 * 16) / C::QK_EB;
              const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
              if (kQK16) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ww[e]));
                  acc = fmaf(qbar[d0 + 2 * e], f.x, acc);
                  acc = fmaf(qbar[d0 + 2 * e + 1], f.y, acc);
                }
              } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const uint32_t h2 = cvt_e4m3x2_to_f16x2((uint16_t)(ww[e >> 1] >> ((e & 1) * 16)));
                  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
                  acc = fmaf(qbar[d0 + 2 * e], f.x, acc);
                  acc = fmaf(qbar[d0 + 2 * e + 1], f.y, acc);
                }
              }
            }
          }
          dsc[r] = acc * dkj * c2;
        }
        // leave together: a thread that stops here must not strand the others
        // at this barrier in the next tile
        if (named_bar_any(1 + t, kWG, fail || *s_abort)) break;
      }
      // the TMEM loads below are warp-collective: the warp decides together
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1, status, 32, s_abort, p.spin))) break;
      tc_fence_after();
      // the whole score row in one TMEM read
      uint32_t v[BK];
#pragma unroll
      for (int ch = 0; ch < BK / 32; ++ch) tmem_ld32(sS + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[ch * 32]));
      tmem_wait_ld();
      const bool need_mask = ((j + 1) * BK > p.M) || (p.causal && (j + 1) * BK - 1 > row0 + p.M - p.N);
      if (smooth_q) {
#pragma unroll
        for (int e = 0; e < BK; ++e) v[e] = __float_as_uint(fmaf(__uint_as_float(v[e]), k1, dsc[e]));
      }
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < BK; ++e) {
          const int key = j * BK + e;
          if (key >= p.M || (p.causal && key > diag)) v[e] = __float_as_uint(-INFINITY);
        }
      }
      // row max; without dS, k1 >= 0 makes max(k1 s) = k1 max(s)
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < BK; e += 8) {
        mx[0] = fmax3(mx[0], __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
        mx[1] = fmax3(mx[1], __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
        mx[2] = fmax3(mx[2], __uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
        mx[3] = fmax3(mx[3], __uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
      }
      const float mraw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const float mt = smooth_q ? mraw : (mraw == -INFINITY ? -INFINITY : mraw * k1);
      const float m_new = fmaxf(m, mt);
      const float alpha = ex2_approx(m - m_new);
      const float mb = m_new - kLog2_448;
      // P^ = e4m3(448 exp2(t - m_new)); row sum of the unquantized values
      const float2 kk2 = smooth_q ? f2(1.0f, 1.0f) : f2(k1, k1);
      const float2 nb2 = f2(-mb, -mb);
      float2 rs2 = f2(0.0f, 0.0f);
#pragma unroll
      for (int ch = 0; ch < BK / 32; ++ch) {
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const int i0 = ch * 32 + e;
          const float2 x01 = __ffma2_rn(f2(__uint_as_float(v[i0]), __uint_as_float(v[i0 + 1])), kk2, nb2);
          const float2 x23 = __ffma2_rn(f2(__uint_as_float(v[i0 + 2]), __uint_as_float(v[i0 + 3])), kk2, nb2);
          const float2 p01 = f2(ex2_approx(x01.x), ex2_approx(x01.y));
          const float2 p23 = f2(ex2_approx(x23.x), ex2_approx(x23.y));
          rs2 = __fadd2_rn(rs2, __fadd2_rn(p01, p23));
          pk[e / 4] = (uint32_t)cvt_e4m3x2(p01.x, p01.y) | ((uint32_t)cvt_e4m3x2(p23.x, p23.y) << 16);
        }
        *reinterpret_cast<uint4 *>(prow + swz_off<C::PV_SW>(r, 2 * ch)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4 *>(prow + swz_off<C::PV_SW>(r, 2 * ch + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
      l = fmaf(alpha, l, rs2.x + rs2.y);
      m = m_new;
      s_alpha[t * 128 + r] = alpha;
      if (j == T_t - 1) s_l[t * 128 + r] = l;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[t]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, int BK, bool kQK16>
sage_status launch_t(const sage_shape &s, int causal, float sm_scale, int flags, const void *ws,
                     const sage_ws_layout &L, void *o, cudaStream_t stream) {
  using C = Cfg<D, BK, kQK16>;
  const char *w = (const char *)ws;
  CUtensorMap tq, tk, tv;
  sage_status st;
  st = make_tmap_2d(&tq, w + L.qhat, C::ROWB, (uint64_t)s.B * s.Hq * L.N_pad, C::ROWB, C::QK_SW, 128, C::QK_SW);
  if (st != SAGE_OK) return st;
  st = make_tmap_2d(&tk, w + L.khat, C::ROWB, (uint64_t)s.B * s.Hkv * L.M_pad, C::ROWB, C::QK_SW, BK, C::QK_SW);
  if (st != SAGE_OK) return st;
  st = make_tmap_2d(&tv, w + L.vhat, L.M_pad, (uint64_t)s.B * s.Hkv * D, L.M_pad, BK, D, C::PV_SW);
  if (st != SAGE_OK) return st;
  AttnParams p;
  p.N = s.N;
  p.M = s.M;
  p.N_pad = L.N_pad;
  p.M_pad = L.M_pad;
  p.Tm = L.Tm;
  p.Tm2 = (L.Tm + 1) / 2;
  p.Tn = L.Tn;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.causal = causal ? 1 : 0;
  p.flags = flags;
  p.sm_log2 = sm_scale * 1.4426950408889634f;
  p.dq = (const float *)(w + L.dq);
  p.qbar = (const float *)(w + L.qbar);
  p.dk = (const float *)(w + L.dk);
  p.dv = (const float *)(w + L.dv);
  p.vm = (const float *)(w + L.vm);
  p.o = (__nv_bfloat16 *)o;
  p.status = (int *)(w + L.status);
  p.spin = spin_limit_cycles();
  auto kern = attn_q8_kernel<D, BK, kQK16>;
  // the register split needs the launch allocation it was computed for
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return SAGE_ERR_CUDA;
  if (fa.numRegs < kLaunchRegs) return SAGE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_TOTAL) != cudaSuccess)
    return SAGE_ERR_CUDA;
  const unsigned grid = (unsigned)(s.B * s.Hq * p.Tm2);
  kern<<<grid, kThreads, C::SMEM_TOTAL, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}

}  // namespace

sage_status launch_attn_q8(const sage_shape &s, int causal, float sm_scale, int mode, int flags, int bk,
                           const void *ws, const sage_ws_layout &L, void *o, cudaStream_t stream) {
  const bool i8 = (mode == SAGE_Q8_PV8);
  if (s.d == 64) {
    if (bk == 64)
      return i8 ? launch_t<64, 64, true>(s, causal, sm_scale, flags, ws, L, o, stream)
                : launch_t<64, 64, false>(s, causal, sm_scale, flags, ws, L, o, stream);
    return i8 ? launch_t<64, 128, true>(s, causal, sm_scale, flags, ws, L, o, stream)
              : launch_t<64, 128, false>(s, causal, sm_scale, flags, ws, L, o, stream);
  }
  if (bk == 64)
    return i8 ? launch_t<128, 64, true>(s, causal, sm_scale, flags, ws, L, o, stream)
              : launch_t<128, 64, false>(s, causal, sm_scale, flags, ws, L, o, stream);
  return i8 ? launch_t<128, 128, true>(s, causal, sm_scale, flags, ws, L, o, stream)
            : launch_t<128, 128, false>(s, causal, sm_scale, flags, ws, L, o, stream);
}

}  // namespace sage
