// Fused quantized attention for the INT8 / FP8 modes on sm_103a.
//
// Per CTA: one query block i of 128 rows of one (b, q-head), streaming the key
// tiles j = 0..T-1 of its kv-head (SageAttention2 Technical Report summary,
// §3.4 "The Complete Algorithm"; "Quantization for Attention, in depth",
// "The datapath and its quantize points"):
//   S_ij  = delta_Q delta_K,j (Q^_i K^_j^T) + dS_ij,  dS_ij = q_bar_i deq(K^_j)^T
//   m_ij  = max(m_i,j-1, rowmax S_ij * sm_scale)
//   P~_ij = exp(S_ij sm_scale - m_ij),  l_ij = e^(m_i,j-1 - m_ij) l + rowsum P~
//   P^_ij = e4m3(448 P~_ij)                          (static scale 1/448)
//   R_ij  = P^_ij V^_j        (tile partial, accumulated over this tile only)
//   O_ij  = e^(m_i,j-1 - m_ij) O_i,j-1 + R_ij        (FP32 running output)
//   O_i   = O / l * delta_V / 448 (+ V_m)
// Scores are kept in the base-2 domain (sm_scale * log2 e folded into the
// dequantization multiply) and the 448 of P^ is folded into the exponent, so
// l carries 448 * sum P~ and the final scale is delta_V / l.
//
// GB300 mapping (not the pages' Ada/Hopper register-level design):
//   warp 4     TMA producer: Q^ once, then K^_j / V^T_j into a STAGES-deep ring
//   warp 5     tcgen05 MMA issuer (one thread): S_j = Q^ K^_j^T into TMEM
//              (kind::f16 on INT8 codes held as exact fp16 integers — sm_103a
//              has no INT8 tensor path — or kind::f8f6f4 on E4M3 codes), and
//              R_j = P^_j V^_j (kind::f8f6f4) into a separate TMEM buffer,
//              zero-initialised by the first k-step of each tile
//   warps 0-3  one query row per thread: TMEM -> registers, dequant + dS,
//              mask, online softmax, P^ to shared memory (128B/64B swizzle,
//              the A operand of the next MMA), then the two-level update
//              O = alpha O + R with O in registers
// S and R are double-buffered in TMEM so QK_{j+1} and PV_j overlap the
// softmax of tile j+1.  Every mbarrier wait is bounded: on timeout the kernel
// records SAGE_ERR_TIMEOUT and the site, drains its own TMA loads and MMAs,
// frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.h"
#include "launch.h"
#include "sm103.cuh"

namespace sage {
namespace {

constexpr int kSoftmaxThreads = 128;
constexpr int kThreads = 192;  // 4 softmax warps, 1 TMA warp, 1 MMA warp
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
  static constexpr int STAGES = (Q_BYTES + 2 * P_BYTES + 3 * (K_BYTES + V_BYTES) <= 200 * 1024) ? 3 : 2;
  static constexpr int TMEM_R = 2 * BK;                  // S buffers at columns [0, 2BK)
  static constexpr int TMEM_NEED = 2 * BK + 2 * D;
  static constexpr int TMEM_COLS = TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int SMEM_TILES = Q_BYTES + STAGES * (K_BYTES + V_BYTES) + 2 * P_BYTES;
  static constexpr int SMEM_MISC = (BK + 3 * D) * 4 + (1 + 3 * STAGES + 6 + 1) * 8 + 16;
  static constexpr int SMEM_TOTAL = 1024 + SMEM_TILES + SMEM_MISC;
  static constexpr uint32_t IDESC_QK = instr_desc(kFmtF32, kQK16 ? kFmtF16 : kFmtE4M3, kQK16 ? kFmtF16 : kFmtE4M3, BK, 128);
  static constexpr uint32_t IDESC_PV = instr_desc(kFmtF32, kFmtE4M3, kFmtE4M3, D, 128);
};

struct AttnParams {
  int N, M, N_pad, M_pad, Tm, Tn, Hq, Hkv, causal, flags;
  float sm_log2;  // sm_scale * log2(e)
  const float *dq, *qbar, *dk, *dv, *vm;
  __nv_bfloat16 *o;
  int *status;
  long long spin;
};

// byte address of 16-byte chunk `c` of row `r` in a K-major swizzled tile whose
// rows are `SW` bytes wide (8-row atoms of 8*SW bytes, 1024-aligned base)
template <int SW>
__device__ __forceinline__ uint32_t swz_off(int r, int c) {
  const int x = (SW == 128) ? (r & 7) : ((r & 7) >> 1);
  return (uint32_t)((r >> 3) * (8 * SW) + (r & 7) * SW + ((c ^ x) << 4));
}

template <int D, int BK, bool kQK16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_q8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D, BK, kQK16>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = base;
  uint8_t *sK = sQ + C::Q_BYTES;
  uint8_t *sV = sK + ST * C::K_BYTES;
  uint8_t *sP = sV + ST * C::V_BYTES;
  float *s_dsc = (float *)(sP + 2 * C::P_BYTES);
  float *s_qbar = s_dsc + BK;
  float *s_dv = s_qbar + D;
  float *s_vm = s_dv + D;
  uint64_t *bars = (uint64_t *)(((uintptr_t)(s_vm + D) + 7) & ~(uintptr_t)7);
  uint64_t *q_full = bars;
  uint64_t *k_full = q_full + 1;
  uint64_t *v_full = k_full + ST;
  uint64_t *kv_empty = v_full + ST;
  uint64_t *s_full = kv_empty + ST;
  uint64_t *p_full = s_full + 2;
  uint64_t *r_full = p_full + 2;
  uint64_t *r_empty = r_full + 2;
  uint64_t *mma_done = r_empty + 2;
  uint32_t *s_tmem = (uint32_t *)(mma_done + 1);
  volatile int *s_abort = (volatile int *)(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int bh = tile / p.Tm;
  const int qi = p.Tm - 1 - tile % p.Tm;  // heaviest causal blocks first
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int hkv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int row0 = qi * 128;
  const int last_row = min(p.N, row0 + 128) - 1;
  int T = p.Tn;
  if (p.causal) T = min(p.Tn, (last_row + p.M - p.N) / BK + 1);
  const bool smooth_q = (p.flags & SAGE_SMOOTH_Q) != 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], kSoftmaxThreads);
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], kSoftmaxThreads);
    }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x < kSoftmaxThreads) {
    for (int c = threadIdx.x; c < D; c += kSoftmaxThreads) {
      s_qbar[c] = smooth_q ? p.qbar[((size_t)bh * p.Tm + qi) * D + c] : 0.0f;
      s_dv[c] = p.dv[(size_t)hkv * D + c];
      s_vm[c] = p.vm[(size_t)hkv * D + c];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  int *status = p.status;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
      for (int c = 0; c < C::QK_CHUNKS; ++c)
        tma_load_2d(sQ + c * 128 * C::QK_SW, &tm_q, q_full, c * C::QK_SW, bh * p.N_pad + row0);
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
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV), p_base = smem_u32(sP);
      auto qk_desc = [&](uint32_t tile_base, int rows, int kk) {
        const int byte = kk * 32;
        const uint32_t a = tile_base + (byte / C::QK_SW) * rows * C::QK_SW + (byte % C::QK_SW);
        return smem_desc(a, 8 * C::QK_SW, C::QK_SW == 128 ? kSwizzle128 : kSwizzle64);
      };
      auto pv_desc = [&](uint32_t tile_base, int kk) {
        return smem_desc(tile_base + kk * 32, 8 * C::PV_SW, C::PV_SW == 128 ? kSwizzle128 : kSwizzle64);
      };
      auto issue_pv = [&](int jj) -> bool {
        const int bb = jj & 1, s = jj % ST, n = jj / ST;
        if (!mbar_wait(&p_full[bb], (jj >> 1) & 1, status, 20, s_abort, p.spin)) return false;
        if (!mbar_wait(&v_full[s], n & 1, status, 21, s_abort, p.spin)) return false;
        if (jj >= 2 && !mbar_wait(&r_empty[bb], ((jj - 2) >> 1) & 1, status, 22, s_abort, p.spin)) return false;
        tc_fence_after();
        const uint32_t dR = tmem + C::TMEM_R + bb * D;
#pragma unroll
        for (int kk = 0; kk < C::PV_KSTEPS; ++kk)
          mma_f8(dR, pv_desc(p_base + bb * C::P_BYTES, kk), pv_desc(v_base + s * C::V_BYTES, kk), C::IDESC_PV,
                 kk > 0);
        mma_commit(&r_full[bb]);
        mma_commit(&kv_empty[s]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, status, 23, s_abort, p.spin);
      tc_fence_after();
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % ST, n = j / ST, sb = j & 1;
        if (!mbar_wait(&k_full[s], n & 1, status, 24, s_abort, p.spin)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dS = tmem + sb * BK;
#pragma unroll
        for (int kk = 0; kk < C::QK_KSTEPS; ++kk) {
          const uint64_t ad = qk_desc(q_base, 128, kk), bd = qk_desc(k_base + s * C::K_BYTES, BK, kk);
          if (kQK16)
            mma_f16(dS, ad, bd, C::IDESC_QK, kk > 0);
          else
            mma_f8(dS, ad, bd, C::IDESC_QK, kk > 0);
        }
        mma_commit(&s_full[sb]);
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok && T >= 1) issue_pv(T - 1);
      // drain: all MMAs this thread issued complete before TMEM is freed
      mma_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, status, 25, &no_abort, p.spin);
    }
  } else {
    // ------------------------------------------------------------ softmax / correction
    const int r = threadIdx.x;  // query row within the block == TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float c2 = p.sm_log2;
    const float dq = p.dq[(size_t)bh * p.Tm + qi];
    const int row = row0 + r;
    const int diag = row + p.M - p.N;  // last key visible to this row (causal)
    float O[D];
#pragma unroll
    for (int c = 0; c < D; ++c) O[c] = 0.0f;
    float m = -INFINITY, l = 0.0f, alpha_prev = 0.0f;
    bool ok = true;

    auto correction = [&](int jj, float a) -> bool {
      const int bb = jj & 1;
      if (!mbar_wait(&r_full[bb], (jj >> 1) & 1, status, 30, s_abort, p.spin)) return false;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + C::TMEM_R + bb * D + ch * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) O[ch * 32 + e] = fmaf(O[ch * 32 + e], a, __uint_as_float(v[e]));
      }
      tc_fence_before();
      mbar_arrive(&r_empty[bb]);
      return true;
    };

    for (int j = 0; j < T; ++j) {
      const int bq = j & 1, s = j % ST;
      const float dkj = p.dk[(size_t)hkv * p.Tn + j];
      const float k1 = dq * dkj * c2;
      if (smooth_q) {
        // dS_j[c] = delta_K,j * sum_d q_bar[d] K^_j[c, d], one key column per thread
        if (!mbar_wait(&k_full[s], (j / ST) & 1, status, 31, s_abort, p.spin)) {
          ok = false;
        }
        if (ok && r < BK) {
          const uint8_t *kt = sK + s * C::K_BYTES;
          float acc = 0.0f;
#pragma unroll
          for (int cc = 0; cc < C::QK_CHUNKS; ++cc) {
#pragma unroll
            for (int c16 = 0; c16 < C::QK_SW / 16; ++c16) {
              const uint4 w = *reinterpret_cast<const uint4 *>(kt + cc * BK * C::QK_SW + swz_off<C::QK_SW>(r, c16));
              const int d0 = (cc * C::QK_SW + c16 * 16) / C::QK_EB;
              if (kQK16) {
                const __half2 *hp = reinterpret_cast<const __half2 *>(&w);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 f = __half22float2(hp[e]);
                  acc = fmaf(s_qbar[d0 + 2 * e], f.x, acc);
                  acc = fmaf(s_qbar[d0 + 2 * e + 1], f.y, acc);
                }
              } else {
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const uint32_t h2 = cvt_e4m3x2_to_f16x2((uint16_t)(ww[e >> 1] >> ((e & 1) * 16)));
                  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
                  acc = fmaf(s_qbar[d0 + 2 * e], f.x, acc);
                  acc = fmaf(s_qbar[d0 + 2 * e + 1], f.y, acc);
                }
              }
            }
          }
          s_dsc[r] = acc * dkj * c2;
        }
        // leave together: a thread that stops here must not strand the others
        // at this barrier in the next tile
        if (named_bar_any(1, kSoftmaxThreads, !ok || *s_abort)) {
          ok = false;
          break;
        }
      }
      if (!ok || !mbar_wait(&s_full[bq], (j >> 1) & 1, status, 32, s_abort, p.spin)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool need_mask = ((j + 1) * BK > p.M) || (p.causal && (j + 1) * BK - 1 > row0 + p.M - p.N);
      const uint32_t sS = tmem + lane_off + bq * BK;
      // pass 1: row max of the scaled, dequantized, corrected scores
      float mt = -INFINITY;
#pragma unroll
      for (int ch = 0; ch < BK / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(sS + ch * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float t = fmaf(__uint_as_float(v[e]), k1, smooth_q ? s_dsc[ch * 32 + e] : 0.0f);
          if (need_mask) {
            const int key = j * BK + ch * 32 + e;
            if (key >= p.M || (p.causal && key > diag)) t = -INFINITY;
          }
          mt = fmaxf(mt, t);
        }
      }
      const float m_new = fmaxf(m, mt);
      const float alpha = ex2_approx(m - m_new);
      const float mb = m_new - kLog2_448;
      // pass 2: P^ = e4m3(448 exp2(t - m_new)), row sum of the unquantized values
      float rs = 0.0f;
      uint8_t *prow = sP + bq * C::P_BYTES;
#pragma unroll
      for (int ch = 0; ch < BK / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(sS + ch * 32, v);
        tmem_wait_ld();
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float pp[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float t = fmaf(__uint_as_float(v[e + u]), k1, smooth_q ? s_dsc[ch * 32 + e + u] : 0.0f);
            if (need_mask) {
              const int key = j * BK + ch * 32 + e + u;
              if (key >= p.M || (p.causal && key > diag)) t = -INFINITY;
            }
            pp[u] = ex2_approx(t - mb);
            rs += pp[u];
          }
          pk[e / 4] = (uint32_t)cvt_e4m3x2(pp[0], pp[1]) | ((uint32_t)cvt_e4m3x2(pp[2], pp[3]) << 16);
        }
        *reinterpret_cast<uint4 *>(prow + swz_off<C::PV_SW>(r, 2 * ch)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4 *>(prow + swz_off<C::PV_SW>(r, 2 * ch + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
      l = fmaf(alpha, l, rs);
      m = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[bq]);
      if (j >= 1 && !correction(j - 1, alpha_prev)) {
        ok = false;
        break;
      }
      alpha_prev = alpha;
    }
    if (ok && T >= 1) ok = correction(T - 1, alpha_prev);

    // epilogue: O / l * delta_V (+ V_m), bf16, one row per thread
    if (ok && row < p.N) {
      const float inv_l = 1.0f / l;
      __nv_bfloat16 *dst = p.o + ((size_t)bh * p.N + row) * D;
#pragma unroll
      for (int c = 0; c < D; c += 8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float o0 = fmaf(O[c + 2 * e], s_dv[c + 2 * e] * inv_l, s_vm[c + 2 * e]);
          const float o1 = fmaf(O[c + 2 * e + 1], s_dv[c + 2 * e + 1] * inv_l, s_vm[c + 2 * e + 1]);
          const __nv_bfloat162 v2 = __floats2bfloat162_rn(o0, o1);
          w[e] = *reinterpret_cast<const uint32_t *>(&v2);
        }
        *reinterpret_cast<uint4 *>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, C::TMEM_COLS);
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
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_TOTAL) != cudaSuccess)
    return SAGE_ERR_CUDA;
  const unsigned grid = (unsigned)(s.B * s.Hq * L.Tm);
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
