// Smoothing + quantization pre-pass for the INT8 / FP8 modes.
//
// What it computes (SageAttention2 Technical Report summary, §3.2 item 1 and
// §3.4 "Smoothing Q" / "FP8 Quantization for P~V" / "Optional Smoothing of V";
// SageAttention3 summary §3.4 "SageBwd Forward Pass" for the per-block INT8
// quantizer):
//   k_bar = mean over tokens of K, gamma(K) = K - k_bar     (if SMOOTH_K)
//   per K block j of bk tokens: delta_K = max|gamma(K_j)| / 127, K^ = round(gamma/delta_K)
//   q_bar_i = mean of the block's rows, gamma(Q_i) = Q_i - q_bar_i (if SMOOTH_Q)
//   per Q block i of 128 rows: delta_Q = max|gamma(Q_i)| / 127, Q^ = round(gamma/delta_Q)
//   V_m = mean over tokens of V (if SMOOTH_V), V' = V - V_m
//   per channel c: delta_V[c] = max_t |V'[t,c]| / 448, V^ = e4m3(V' / delta_V)
// (FP8 Q/K mode: / 448 and E4M3 codes instead of / 127 and integers.)
//
// Every arithmetic step is one IEEE binary32 (or binary64 for the mean)
// operation with round-to-nearest-even, issued through the _rn intrinsics, so
// the results are a fixed function of the inputs:
//   - means use an exact integer sum of the values in fixed point (lsb 2^-24,
//     truncated toward zero), converted once to double and divided once;
//     integer addition is associative, so any reduction order gives the same
//     bits;
//   - the V per-channel absmax after subtracting V_m is taken from the channel
//     min and max (rounded subtraction is monotone, so
//     max_t |fl(v_t - m)| = max(|fl(max v - m)|, |fl(min v - m)|)), which lets
//     one statistics pass carry everything the quantize pass needs.
//
// Launches: init (clear stats + status), stats (K/V column sums, V min/max),
// quantize (Q blocks, K blocks, V token chunks in one grid).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "layout.h"
#include "launch.h"
#include "sm103.cuh"

namespace sage {
namespace {

constexpr int kThreads = 256;
constexpr int kQuantCtas = 4;  // resident quantize CTAs per SM (caps registers at 64)
constexpr int kStatTokens = 256;  // tokens per statistics CTA (at most 64 rows per thread)

__device__ __forceinline__ int order_key(float f) {
  int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float order_val(int k) { return __int_as_float(k >= 0 ? k : (k ^ 0x7FFFFFFF)); }

__device__ __forceinline__ bool in_range(float f) { return fabsf(f) < 65536.0f; }  // false for NaN too

// trunc(x * 2^24) toward zero for a bf16 x (its fp32 value f), from the bits:
// x = (-1)^s * (128 + mant) * 2^(e - 134), so x * 2^24 = (128 + mant) * 2^(e - 110);
// a right shift truncates the magnitude toward zero.  Zero and subnormals give 0;
// inf / NaN (rejected by the range check) are clamped to keep the shift defined.
__device__ __forceinline__ long long fixed24(float f) {
  const uint32_t b = __float_as_uint(f) >> 16;
  const int e = (int)((b >> 7) & 0xFF);
  const long long m = (long long)((b & 0x7F) | 0x80);
  const int sh = min(e - 110, 40);
  long long a = (sh >= 0) ? (m << sh) : (sh > -8 ? (m >> -sh) : 0);
  if (e == 0) a = 0;
  return (b & 0x8000) ? -a : a;
}

// The same value accumulated into two 32-bit buckets, in units of 1 (lo) and
// of 2^16 (hi): with e - 110 = sh, m << sh for 0 <= sh < 16 and
// (m << (sh - 16)) * 2^16 for sh >= 16.  For |x| < 2^16 a term is below 2^24 in
// either bucket, so 64 terms fit in an int; the shift is clamped for inf / NaN.
__device__ __forceinline__ void fixed24_acc(uint32_t b, int &lo, int &hi) {
  const int e = (int)((b >> 7) & 0xFF);
  const int m = (int)((b & 0x7F) | 0x80);
  const int sh = e - 110;
  const bool big = sh >= 16;
  const int t = big ? min(sh - 16, 16) : sh;
  int v = t >= 0 ? (m << t) : (t > -9 ? (m >> -t) : 0);
  v = (b & 0x8000) ? -v : v;
  if (big)
    hi += v;
  else
    lo += v;
}

__device__ __forceinline__ float mean_from_sum(long long sum, int n) {
  return __double2float_rn(__ddiv_rn(__dmul_rn(__ll2double_rn(sum), 0x1p-24), (double)n));
}

__device__ __forceinline__ void raise_status(int *status, int code, int site) {
  if (atomicCAS(status, 0, code) == 0) status[1] = site;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 &u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// block-wide max of non-negative floats (all threads get the result)
__device__ float block_max(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
  return m;
}

// ------------------------------------------------------------------ init
__global__ void init_kernel(StatsView st, int n, int *status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    st.ksum[i] = 0;
    st.vsum[i] = 0;
    st.vmin[i] = order_key(__int_as_float(0x7F800000));   // +inf
    st.vmax[i] = order_key(__int_as_float(0xFF800000));   // -inf
  }
  if (i < 4) status[i] = 0;
}

// ------------------------------------------------------------------ stats
// grid (ceil(M / kStatTokens), B*Hkv).  Fixed-point column sums of K (when K
// is smoothed) and V (when V is smoothed), column min / max of V, range check
// of K and V.  Each thread owns 8 channels of every RPP-th row; loads are
// issued in batches of kBatch rows so several are in flight.  Min / max run
// on packed bf16 pairs with NaN propagation (they are exact, and a NaN or an
// out-of-range value shows in the extremes).
// Packed sequences (seq non-null): batch b is sequence b, its M its own key
// count, and its rows sit at (k0 + t) * Hkv + h of the packed [total, Hkv, d]
// inputs; CTAs past the sequence's keys have nothing to do.
template <int D, bool kSumK, bool kSumV, bool kVar>
__global__ void __launch_bounds__(kThreads) stats_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                         int M, StatsView st, int *status, const VarSeq *seq,
                                                         int Hkv) {
  constexpr int VPR = D / 8;               // 16-byte vectors per row (threads per row)
  constexpr int RPP = kThreads / VPR;      // rows per pass
  constexpr int kBatch = 4;
  constexpr int NW = kThreads / 32;
  __shared__ long long sk[kSumK ? NW : 1][D];
  __shared__ long long sv[kSumV ? NW : 1][D];
  __shared__ int smin[NW][D];
  __shared__ int smax[NW][D];
  const int hb = blockIdx.y;
  const int vc = threadIdx.x % VPR, rr = threadIdx.x / VPR;
  const int t0 = blockIdx.x * kStatTokens;
  // row of token t: hb * M + t (batched) or (k0 + t) * Hkv + h (packed)
  long long row_base = (long long)hb * M, row_step = 1;
  if constexpr (kVar) {
    const VarSeq sq = seq[hb / Hkv];
    M = sq.M;
    row_base = (long long)sq.k0 * Hkv + hb % Hkv;
    row_step = Hkv;
    if (t0 >= M) return;  // the whole CTA: nothing of this sequence here
  }
  const int t1 = min(M, t0 + kStatTokens);
  int klo[8], khi[8], vlo[8], vhi[8];
  __nv_bfloat162 kmn[4], kmx[4], vmn[4], vmx[4];
  const __nv_bfloat162 pinf = __halves2bfloat162(__ushort_as_bfloat16(0x7F80), __ushort_as_bfloat16(0x7F80));
  const __nv_bfloat162 ninf = __halves2bfloat162(__ushort_as_bfloat16(0xFF80), __ushort_as_bfloat16(0xFF80));
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    klo[e] = khi[e] = vlo[e] = vhi[e] = 0;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    kmn[i] = pinf;
    vmn[i] = pinf;
    kmx[i] = ninf;
    vmx[i] = ninf;
  }
  for (int tb = t0 + rr; tb < t1; tb += kBatch * RPP) {
    uint4 kb[kBatch], vb[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int t = tb + i * RPP;
      const size_t off = kVar ? (size_t)(row_base + (long long)min(t, t1 - 1) * row_step) * VPR + vc
                              : ((size_t)hb * M + min(t, t1 - 1)) * VPR + vc;
      kb[i] = k[off];
      vb[i] = v[off];
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (tb + i * RPP >= t1) break;
      const uint32_t kw[4] = {kb[i].x, kb[i].y, kb[i].z, kb[i].w};
      const uint32_t vw[4] = {vb[i].x, vb[i].y, vb[i].z, vb[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162 kx = *reinterpret_cast<const __nv_bfloat162 *>(&kw[q]);
        const __nv_bfloat162 vx = *reinterpret_cast<const __nv_bfloat162 *>(&vw[q]);
        kmn[q] = __hmin2_nan(kmn[q], kx);
        kmx[q] = __hmax2_nan(kmx[q], kx);
        vmn[q] = __hmin2_nan(vmn[q], vx);
        vmx[q] = __hmax2_nan(vmx[q], vx);
        if (kSumK) {
          fixed24_acc(kw[q] & 0xFFFF, klo[2 * q], khi[2 * q]);
          fixed24_acc(kw[q] >> 16, klo[2 * q + 1], khi[2 * q + 1]);
        }
        if (kSumV) {
          fixed24_acc(vw[q] & 0xFFFF, vlo[2 * q], vhi[2 * q]);
          fixed24_acc(vw[q] >> 16, vlo[2 * q + 1], vhi[2 * q + 1]);
        }
      }
    }
  }
  // range: every |x| < 2^16 and no NaN (a NaN fails both comparisons)
  float vmnf[8], vmxf[8];
  bool bad_k = false, bad_v = false;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 a = __bfloat1622float2(kmn[q]), b = __bfloat1622float2(kmx[q]);
    const float2 c = __bfloat1622float2(vmn[q]), d = __bfloat1622float2(vmx[q]);
    if (t0 + rr < t1) {
      bad_k |= !(a.x > -65536.0f && a.y > -65536.0f && b.x < 65536.0f && b.y < 65536.0f);
      bad_v |= !(c.x > -65536.0f && c.y > -65536.0f && d.x < 65536.0f && d.y < 65536.0f);
    }
    vmnf[2 * q] = c.x;
    vmnf[2 * q + 1] = c.y;
    vmxf[2 * q] = d.x;
    vmxf[2 * q + 1] = d.y;
  }
  if (bad_k) raise_status(status, SAGE_ERR_RANGE, 1);
  if (bad_v) raise_status(status, SAGE_ERR_RANGE, 2);
  long long ks[8], vs[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ks[e] = (long long)khi[e] * 65536 + klo[e];
    vs[e] = (long long)vhi[e] * 65536 + vlo[e];
  }
  // lanes vc, vc + VPR, ... of a warp hold the same channels
#pragma unroll
  for (int o = VPR; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (kSumK) ks[e] += __shfl_xor_sync(0xffffffffu, ks[e], o);
      if (kSumV) vs[e] += __shfl_xor_sync(0xffffffffu, vs[e], o);
      vmnf[e] = fminf(vmnf[e], __shfl_xor_sync(0xffffffffu, vmnf[e], o));
      vmxf[e] = fmaxf(vmxf[e], __shfl_xor_sync(0xffffffffu, vmxf[e], o));
    }
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l < VPR) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (kSumK) sk[w][vc * 8 + e] = ks[e];
      if (kSumV) sv[w][vc * 8 + e] = vs[e];
      smin[w][vc * 8 + e] = order_key(vmnf[e]);
      smax[w][vc * 8 + e] = order_key(vmxf[e]);
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += kThreads) {
    long long a = 0, b = 0;
    int mn = smin[0][c], mx = smax[0][c];
#pragma unroll
    for (int r = 0; r < NW; ++r) {
      if (kSumK) a += sk[r][c];
      if (kSumV) b += sv[r][c];
      mn = min(mn, smin[r][c]);
      mx = max(mx, smax[r][c]);
    }
    const size_t i = (size_t)hb * D + c;
    if (kSumK) atomicAdd((unsigned long long *)&st.ksum[i], (unsigned long long)a);
    if (kSumV) atomicAdd((unsigned long long *)&st.vsum[i], (unsigned long long)b);
    atomicMin(&st.vmin[i], mn);
    atomicMax(&st.vmax[i], mx);
  }
}

template <int D>
void launch_stats(dim3 grid, int flags, const void *k, const void *v, int M, StatsView st, int *status,
                  cudaStream_t stream, const VarSeq *seq, int Hkv) {
  const bool sk = (flags & SAGE_SMOOTH_K) != 0, sv = (flags & SAGE_SMOOTH_V) != 0;
  const uint4 *k4 = (const uint4 *)k, *v4 = (const uint4 *)v;
  using Kern = void (*)(const uint4 *, const uint4 *, int, StatsView, int *, const VarSeq *, int);
  Kern kern;
  if (seq)
    kern = sk ? (sv ? stats_kernel<D, true, true, true> : stats_kernel<D, true, false, true>)
              : (sv ? stats_kernel<D, false, true, true> : stats_kernel<D, false, false, true>);
  else
    kern = sk ? (sv ? stats_kernel<D, true, true, false> : stats_kernel<D, true, false, false>)
              : (sv ? stats_kernel<D, false, true, false> : stats_kernel<D, false, false, false>);
  kern<<<grid, kThreads, 0, stream>>>(k4, v4, M, st, status, seq, Hkv);
}

// ------------------------------------------------------------------ finalize
// One thread per (b, kv-head, channel): k_bar and V_m from the fixed-point
// sums (when smoothed), and delta_V = max_t |fl(V - V_m)| / 448 from the channel
// min and max (rounded subtraction is monotone).
// Packed sequences: the mean of (b, h) is over sequence b's M (a sequence
// with no keys has no mean and no use for one: 0).
__global__ void finalize_kernel(StatsView st, int n, int M, int flags, float *kbar, float *vm, float *dv,
                                const VarSeq *seq, int per_seq) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  if (seq) {
    M = seq[i / per_seq].M;
    if (M == 0) {
      kbar[i] = vm[i] = dv[i] = 0.0f;
      return;
    }
  }
  kbar[i] = (flags & SAGE_SMOOTH_K) ? mean_from_sum(st.ksum[i], M) : 0.0f;
  const float mu = (flags & SAGE_SMOOTH_V) ? mean_from_sum(st.vsum[i], M) : 0.0f;
  const float hi = order_val(st.vmax[i]), lo = order_val(st.vmin[i]);
  vm[i] = mu;
  dv[i] = __fdiv_rn(fmaxf(fabsf(__fsub_rn(hi, mu)), fabsf(__fsub_rn(lo, mu))), 448.0f);
}

// ------------------------------------------------------------------ quantize
struct QuantArgs {
  const uint4 *q, *k, *v;  // bf16 inputs, as 16-byte vectors
  int B, Hq, Hkv, N, M, N_pad, M_pad, Tm, Tn, bk;
  int mode, flags;
  uint8_t *qhat, *khat, *vhat;
  float *dq, *qbar, *dk, *kbar, *dv, *vm;
  float *dqt;  // per-row Q scales (SAGE_Q_PER_TOKEN)
  float *dvb;  // per-block V scales (SageBwd forward)
  const VarSeq *seq;  // packed sequences: per-sequence lengths and first rows (null: batched)
  StatsView st;
  int *status;
  int nq, nk;  // CTA counts of the Q and K roles (V takes the rest)
};

// The exact quotients the quantizers fall back to near a rounding tie, out of
// line: they run rarely, and inlined at every (unrolled) call site their
// divisions would fill the pre-pass kernels' instruction footprint.
__device__ __noinline__ float rint_div_exact(float x, float d) { return rintf(__fdiv_rn(x, d)); }
__device__ __noinline__ uint32_t e4m3_div_exact2(float x0, float x1, float d0, float d1) {
  return cvt_e4m3x2(__fdiv_rn(x0, d0), __fdiv_rn(x1, d1));
}

// rint(RN(x / d)) clamped to +-127, exactly as rint(__fdiv_rn(x, d)) gives it.
// q = x * RN(1/d) is within about 1.5e-5 of x/d for |x/d| <= 127, and RN(x/d)
// within 7.6e-6 of x/d; unless q lies within 1e-4 of a half-integer, both round
// to the same integer.  Near a half-integer (and for a non-finite q) the exact
// quotient decides.
__device__ __forceinline__ float int8_code(float x, float d, float rcp) {
  const float q = __fmul_rn(x, rcp);
  float c = rintf(q);
  if (__builtin_expect(!(fabsf(fabsf(__fsub_rn(q, c)) - 0.5f) > 1e-4f), 0)) c = rint_div_exact(x, d);
  return fminf(fmaxf(c, -127.0f), 127.0f);
}

// E4M3 codes of RN(x0 / d0), RN(x1 / d1) (low byte first), exactly as
// cvt(__fdiv_rn(x, d)) gives them: RN(x/d) lies between q(1 - 2^-19) and
// q(1 + 2^-19) for q = x * RN(1/d), and the conversion is monotone, so when
// both ends give the same code that is the code; otherwise the exact quotient
// decides.
__device__ __forceinline__ uint16_t e4m3_code2(float x0, float x1, float d0, float d1, float rcp0, float rcp1) {
  const float q0 = __fmul_rn(x0, rcp0), q1 = __fmul_rn(x1, rcp1);
  const float lo = 1.0f - 0x1p-19f, hi = 1.0f + 0x1p-19f;
  const uint16_t a = cvt_e4m3x2(__fmul_rn(q0, lo), __fmul_rn(q1, lo));
  const uint16_t b = cvt_e4m3x2(__fmul_rn(q0, hi), __fmul_rn(q1, hi));
  if (__builtin_expect(a == b && isfinite(q0) && isfinite(q1), 1)) return a;
  return (uint16_t)e4m3_div_exact2(x0, x1, d0, d1);
}

// Codes of 8 smoothed values g = fl(f - mu) with scale delta: 8 fp16 integers
// (INT8 mode, 16 bytes) or 8 E4M3 bytes (FP8 mode).  INT8: q = g * RN(1/delta)
// is rounded to the nearest integer; when no q of the group lies within 1e-4 of
// a half-integer that is rint(RN(g / delta)) (see int8_code), otherwise the
// group takes the exact path.  |g| <= amax keeps |q| below 127.5, so no clamp
// is reached.
template <bool kInt8>
__device__ __forceinline__ void encode8(const float (&f)[8], const float (&mu)[8], float delta, float rcp, bool on,
                                        uint8_t *dst) {
  if (kInt8) {
    uint32_t w[4] = {0, 0, 0, 0};
    if (on) {
      float g[8], c[8];
      float dmax = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 g2 = __fadd2_rn(make_float2(f[2 * i], f[2 * i + 1]), make_float2(-mu[2 * i], -mu[2 * i + 1]));
        const float2 q2 = __fmul2_rn(g2, make_float2(rcp, rcp));
        g[2 * i] = g2.x;
        g[2 * i + 1] = g2.y;
        c[2 * i] = rintf(q2.x);
        c[2 * i + 1] = rintf(q2.y);
        const float2 d2 = __fadd2_rn(q2, make_float2(-c[2 * i], -c[2 * i + 1]));
        dmax = fmaxf(dmax, fmaxf(fabsf(d2.x), fabsf(d2.y)));
      }
      if (!(dmax < 0.4999f)) {
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = int8_code(g[e], delta, rcp);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(c[2 * i], c[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t *>(&h);
      }
    }
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    uint32_t w[2] = {0, 0};
    if (on) {
      float g[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) g[e] = __fsub_rn(f[e], mu[e]);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint16_t c01 = e4m3_code2(g[4 * i], g[4 * i + 1], delta, delta, rcp, rcp);
        const uint16_t c23 = e4m3_code2(g[4 * i + 2], g[4 * i + 3], delta, delta, rcp, rcp);
        w[i] = (uint32_t)c01 | ((uint32_t)c23 << 16);
      }
    }
    *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
  }
}

// One block of `rows` rows (<= 128) of a [*, D] bf16 matrix: optional
// per-block mean (fixed point over the valid rows) or a given mean, then the
// per-block absmax scale and the codes.  Rows past `valid_rows` get code 0.
// kPerRow: each row takes its own scale, max over its channels of
// |fl(x - mu)| / 127 (or / 448), written to row_delta_out[r] (0 past
// valid_rows), and *delta_out is 0.
// The absmax max_r |fl(x_r - mu)| of a channel is taken from the channel's
// extremes (rounded subtraction is monotone), which packed bf16 min / max
// track exactly; they also carry the range check (NaN propagates).
// Shared memory of the Q/K role (fixed-point partial sums, mean, reduction)
// and of the V role (per-channel mean / scale / reciprocal, transpose tile):
// one pool, since a CTA takes one role.
template <int D>
__host__ __device__ constexpr int qk_pool_bytes() { return (kThreads / (D / 8)) * D * 8 + D * 4 + (kThreads / 32) * 4; }
template <int D>
__host__ __device__ constexpr int v_pool_bytes() { return 3 * D * 4 + D * 33 * 4; }

template <int D, bool kInt8, bool kPerRow = false>
__device__ void quant_block(const uint4 *__restrict__ src, int valid_rows, int rows, bool own_mean,
                            const float *__restrict__ given_mean, uint8_t *dst, float *delta_out,
                            float *mean_out, int *status, int site, unsigned char *pool,
                            float *row_delta_out = nullptr, int src_stride = D / 8) {
  constexpr int VPR = D / 8, RPP = kThreads / VPR, PASSES = 128 / RPP;
  long long (*ssum)[D] = reinterpret_cast<long long (*)[D]>(pool);
  float *smean = reinterpret_cast<float *>(pool + RPP * D * 8);
  float *red = smean + D;
  const int vc = threadIdx.x % VPR, rr = threadIdx.x / VPR;
  const __nv_bfloat162 pinf = __halves2bfloat162(__ushort_as_bfloat16(0x7F80), __ushort_as_bfloat16(0x7F80));
  const __nv_bfloat162 ninf = __halves2bfloat162(__ushort_as_bfloat16(0xFF80), __ushort_as_bfloat16(0xFF80));
  uint4 x[PASSES];
  __nv_bfloat162 mn[4] = {pinf, pinf, pinf, pinf}, mx[4] = {ninf, ninf, ninf, ninf};
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int r = rr + p * RPP;
    x[p] = (r < valid_rows) ? src[(size_t)r * src_stride + vc] : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int r = rr + p * RPP;
    if (r < valid_rows) {
      const uint32_t w[4] = {x[p].x, x[p].y, x[p].z, x[p].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162 *>(&w[q]);
        mn[q] = __hmin2_nan(mn[q], b2);
        mx[q] = __hmax2_nan(mx[q], b2);
      }
    }
  }
  if (own_mean) {
    long long s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      if (rr + p * RPP >= valid_rows) continue;
      float f[8];
      unpack_bf16x8(x[p], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) s[e] += fixed24(f[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) ssum[rr][vc * 8 + e] = s[e];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kThreads) {
      long long a = 0;
      for (int r = 0; r < RPP; ++r) a += ssum[r][c];
      smean[c] = mean_from_sum(a, valid_rows);
    }
  } else {
    for (int c = threadIdx.x; c < D; c += kThreads) smean[c] = given_mean ? given_mean[c] : 0.0f;
  }
  __syncthreads();
  float mu[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) mu[e] = smean[vc * 8 + e];
  float amax = 0.0f;
  if (rr < valid_rows) {  // this thread saw at least one row
    bool bad = false;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 lo = __bfloat1622float2(mn[q]), hi = __bfloat1622float2(mx[q]);
      bad |= !(lo.x > -65536.0f && lo.y > -65536.0f && hi.x < 65536.0f && hi.y < 65536.0f);
      amax = fmaxf(amax, fmaxf(fabsf(__fsub_rn(hi.x, mu[2 * q])), fabsf(__fsub_rn(lo.x, mu[2 * q]))));
      amax = fmaxf(amax, fmaxf(fabsf(__fsub_rn(hi.y, mu[2 * q + 1])), fabsf(__fsub_rn(lo.y, mu[2 * q + 1]))));
    }
    if (bad) raise_status(status, SAGE_ERR_RANGE, site);
  }
  constexpr int CB = kInt8 ? 2 : 1;  // bytes per stored code
  if constexpr (kPerRow) {
    // per-row scales: the VPR threads of a row are consecutive lanes of one
    // warp (VPR divides 32), so the row maximum is a shuffle reduction; every
    // lane runs every shuffle
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int r = rr + p * RPP;
      float f[8];
      unpack_bf16x8(x[p], f);
      float am = 0.0f;
      if (r < valid_rows) {
#pragma unroll
        for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(__fsub_rn(f[e], mu[e])));
      }
#pragma unroll
      for (int o = 1; o < VPR; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      const float dr = __fdiv_rn(am, kInt8 ? 127.0f : 448.0f);
      const float rc = __frcp_rn(dr);
      if (r < rows) {
        encode8<kInt8>(f, mu, dr, rc, r < valid_rows && dr != 0.0f, dst + ((size_t)r * D + vc * 8) * CB);
        if (vc == 0) row_delta_out[r] = dr;
      }
    }
    if (threadIdx.x == 0) *delta_out = 0.0f;
    if (mean_out)
      for (int c = threadIdx.x; c < D; c += kThreads) mean_out[c] = smean[c];
    return;
  }
  amax = block_max(amax, red);
  const float delta = __fdiv_rn(amax, kInt8 ? 127.0f : 448.0f);
  const float rcp = __frcp_rn(delta);
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int r = rr + p * RPP;
    if (r >= rows) continue;
    float f[8];
    unpack_bf16x8(x[p], f);
    encode8<kInt8>(f, mu, delta, rcp, r < valid_rows && delta != 0.0f, dst + ((size_t)r * D + vc * 8) * CB);
  }
  if (threadIdx.x == 0) *delta_out = delta;
  if (mean_out)
    for (int c = threadIdx.x; c < D; c += kThreads) mean_out[c] = smean[c];
}

// kPerRow: per-row Q scales (SAGE_Q_PER_TOKEN), an instance of its own so that
// the per-block instances keep their register allocation.  kVBlk: the SageBwd
// forward's V (per-block INT8 over 64-token blocks, fp16 integer codes).
// kVar: packed sequences (per-sequence lengths, packed [total, H, d] inputs).
template <int D, bool kInt8, bool kPerRow, bool kVBlk, bool kVar>
__global__ void __launch_bounds__(kThreads, kQuantCtas) quantize_kernel(QuantArgs a) {
  constexpr int CB = kInt8 ? 2 : 1;
  constexpr int kPool = qk_pool_bytes<D>() > v_pool_bytes<D>() ? qk_pool_bytes<D>() : v_pool_bytes<D>();
  __shared__ __align__(16) unsigned char pool[kPool];
  int cta = blockIdx.x;
  if (cta < a.nq) {
    // ---- Q block (b, h, i)
    const int i = cta % a.Tm, bh = cta / a.Tm;
    const int r0 = i * 128;
    // rows of this block in the input: batched [B, Hq, N, d], or packed [total, Hq, d]
    int Nb = a.N, stride = D / 8;
    const uint4 *src = a.q + ((size_t)bh * a.N + r0) * (D / 8);
    if constexpr (kVar) {
      const VarSeq sq = a.seq[bh / a.Hq];
      Nb = sq.N;
      stride = a.Hq * (D / 8);
      src = a.q + ((size_t)(sq.q0 + r0) * a.Hq + bh % a.Hq) * (D / 8);
    }
    const int valid = max(0, min(128, Nb - r0));
    const bool smooth = (a.flags & SAGE_SMOOTH_Q) != 0;
    float *qbar = a.qbar + ((size_t)bh * a.Tm + i) * D;
    quant_block<D, kInt8, kPerRow>(src, valid, 128, smooth && valid > 0, nullptr,
                                   a.qhat + ((size_t)bh * a.N_pad + r0) * D * CB, a.dq + (size_t)bh * a.Tm + i,
                                   qbar, a.status, 3, pool, a.dqt + (size_t)bh * a.N_pad + r0, stride);
    return;
  }
  cta -= a.nq;
  if (cta < a.nk) {
    // ---- K block (b, g, j): k_bar over all tokens from the finalize pass
    const int j = cta % a.Tn, hb = cta / a.Tn;
    const int t0 = j * a.bk;
    int Mb = a.M, stride = D / 8;
    const uint4 *src = a.k + ((size_t)hb * a.M + t0) * (D / 8);
    if constexpr (kVar) {
      const VarSeq sq = a.seq[hb / a.Hkv];
      Mb = sq.M;
      stride = a.Hkv * (D / 8);
      src = a.k + ((size_t)(sq.k0 + t0) * a.Hkv + hb % a.Hkv) * (D / 8);
    }
    const int valid = max(0, min(a.bk, Mb - t0));
    quant_block<D, kInt8>(src, valid, a.bk, false, a.kbar + (size_t)hb * D,
                          a.khat + ((size_t)hb * a.M_pad + t0) * D * CB, a.dk + (size_t)hb * a.Tn + j, nullptr,
                          a.status, 1, pool, nullptr, stride);
    return;
  }
  cta -= a.nk;
  if constexpr (kVBlk) {
    // ---- V token chunk (b, g, 128 tokens), SageBwd forward (SageAttention3
    // summary, "SageBwd Forward Pass"): the chunk holds two 64-token blocks;
    // per block s_V = max |fl(V - V_m)| / 127 over its tokens and all
    // channels, codes rint(fl(V' / s_V)) as fp16 integers written transposed
    // (token-contiguous per channel).  Work item = 4 consecutive tokens x 8
    // channels; the 32 lanes of a warp take 32 consecutive token groups of the
    // same channels, so lanes 0-15 hold block 0 and 16-31 block 1, and each
    // code store of a warp is 256 contiguous bytes.  Tokens past M get code 0
    // (the attention's masked keys read them).  The raw rows stay in
    // registers between the maximum and the codes.
    constexpr int VPR = D / 8;
    constexpr int IPT = 32 * VPR / kThreads;  // work items per thread
    static_assert(IPT >= 1 && IPT * kThreads == 32 * VPR, "whole work items per thread");
    const int nchunk = a.M_pad / 128;
    const int ch = cta % nchunk, hb = cta / nchunk;
    // this (b, kv-head)'s keys: batched rows hb * M + t, or packed (k0 + t) * Hkv + h
    int Mb = a.M;
    long long vrow = (long long)hb * a.M, vstep = 1;
    if constexpr (kVar) {
      const VarSeq sq = a.seq[hb / a.Hkv];
      Mb = sq.M;
      vrow = (long long)sq.k0 * a.Hkv + hb % a.Hkv;
      vstep = a.Hkv;
    }
    float *vmean = reinterpret_cast<float *>(pool);
    unsigned *bmax = reinterpret_cast<unsigned *>(vmean + D);  // block maxima (non-negative floats as bits)
    for (int c = threadIdx.x; c < D; c += kThreads) vmean[c] = a.vm[(size_t)hb * D + c];
    if (threadIdx.x < 2) bmax[threadIdx.x] = 0u;
    __syncthreads();
    const int t0 = ch * 128;
    const int tg = threadIdx.x & 31, blk = tg >> 4;  // token group (the lane) and its 64-token block
    uint4 raw[IPT][4];
    float am = 0.0f;
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
      const int cg = (threadIdx.x + k * kThreads) >> 5;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = t0 + 4 * tg + u;
        const size_t vi = kVar ? (size_t)(vrow + (long long)t * vstep) * VPR + cg : ((size_t)hb * a.M + t) * VPR + cg;
        raw[k][u] = (t < Mb) ? a.v[vi] : make_uint4(0, 0, 0, 0);
        if (t < Mb) {
          float f[8];
          unpack_bf16x8(raw[k][u], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(__fsub_rn(f[e], vmean[cg * 8 + e])));
        }
      }
    }
    // half-warp maxima (lanes 0-15 block 0, 16-31 block 1), then one atomic each
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if ((tg & 15) == 0) atomicMax(&bmax[blk], __float_as_uint(am));
    __syncthreads();
    const float delta = __fdiv_rn(__uint_as_float(bmax[blk]), 127.0f);
    const float rcp = __frcp_rn(delta);
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
      const int cg = (threadIdx.x + k * kThreads) >> 5;
      float f[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) unpack_bf16x8(raw[k][u], f[u]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float c4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          c4[u] = (delta != 0.0f && t0 + 4 * tg + u < Mb)
                      ? int8_code(__fsub_rn(f[u][e], vmean[cg * 8 + e]), delta, rcp) : 0.0f;
        const __half2 h01 = __floats2half2_rn(c4[0], c4[1]), h23 = __floats2half2_rn(c4[2], c4[3]);
        *reinterpret_cast<uint2 *>(a.vhat + (((size_t)hb * D + cg * 8 + e) * a.M_pad + t0 + 4 * tg) * 2) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&h01), *reinterpret_cast<const uint32_t *>(&h23));
      }
    }
    if (threadIdx.x < 2) {
      const int j = t0 / 64 + threadIdx.x;  // 64-token block index
      if (j < a.Tn) a.dvb[(size_t)hb * a.Tn + j] = __fdiv_rn(__uint_as_float(bmax[threadIdx.x]), 127.0f);
    }
    return;
  }
  // ---- V token chunk (b, g, 128 tokens): per-channel scales from the stats,
  // E4M3 codes written transposed (token-contiguous per channel).  Each work
  // item is 4 consecutive tokens x 8 channels: the 4 codes of a channel pack
  // into one 32-bit word of a shared [channel][token/4] tile (row pitch 33
  // words: the 32 items of a warp, consecutive token groups, hit 32 banks),
  // which is then written out as 128-byte channel rows.
  {
    const int nchunk = a.M_pad / 128;
    const int ch = cta % nchunk, hb = cta / nchunk;
    int Mb = a.M;
    long long vrow = (long long)hb * a.M, vstep = 1;
    if constexpr (kVar) {
      const VarSeq sq = a.seq[hb / a.Hkv];
      Mb = sq.M;
      vrow = (long long)sq.k0 * a.Hkv + hb % a.Hkv;
      vstep = a.Hkv;
    }
    float *vmean = reinterpret_cast<float *>(pool), *vdelta = vmean + D, *vrcp = vdelta + D;
    uint32_t (*tile)[33] = reinterpret_cast<uint32_t (*)[33]>(vrcp + D);
    for (int c = threadIdx.x; c < D; c += kThreads) {
      const size_t i = (size_t)hb * D + c;
      vmean[c] = a.vm[i];
      vdelta[c] = a.dv[i];
      vrcp[c] = __frcp_rn(vdelta[c]);
    }
    __syncthreads();
    constexpr int VPR = D / 8;
    const int t0 = ch * 128;
    for (int item = threadIdx.x; item < 32 * VPR; item += kThreads) {
      const int tg = item & 31, cg = item >> 5;   // 4 tokens from 4*tg, channels 8*cg..
      uint4 raw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = t0 + 4 * tg + u;
        const size_t vi = kVar ? (size_t)(vrow + (long long)t * vstep) * VPR + cg : ((size_t)hb * a.M + t) * VPR + cg;
        raw[u] = (t < Mb) ? a.v[vi] : make_uint4(0, 0, 0, 0);
      }
      uint32_t word[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (t0 + 4 * tg + u >= Mb) continue;
        float f[8];
        unpack_bf16x8(raw[u], f);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const int c = cg * 8 + e;
          const float g0 = __fsub_rn(f[e], vmean[c]), g1 = __fsub_rn(f[e + 1], vmean[c + 1]);
          // a zero scale (an all-zero channel) gives zero codes
          const uint16_t pr = e4m3_code2(vdelta[c] != 0.0f ? g0 : 0.0f, vdelta[c + 1] != 0.0f ? g1 : 0.0f,
                                         vdelta[c], vdelta[c + 1], vrcp[c], vrcp[c + 1]);
          const uint32_t lo0 = vdelta[c] != 0.0f ? (pr & 0xFF) : 0, lo1 = vdelta[c + 1] != 0.0f ? (pr >> 8) : 0;
          word[e] |= lo0 << (8 * u);
          word[e + 1] |= lo1 << (8 * u);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) tile[cg * 8 + e][tg] = word[e];
    }
    __syncthreads();
    // coalesced store: each channel row of 128 tokens is 128 contiguous bytes
    for (int idx = threadIdx.x; idx < D * 8; idx += kThreads) {
      const int c = idx / 8, part = idx % 8;
      const uint4 w = make_uint4(tile[c][4 * part], tile[c][4 * part + 1], tile[c][4 * part + 2], tile[c][4 * part + 3]);
      *reinterpret_cast<uint4 *>(a.vhat + ((size_t)hb * D + c) * a.M_pad + t0 + part * 16) = w;
    }
  }
}

// ------------------------------------------------------------------ NVFP4
// phi of the SageAttention3 summary §3.4: per 1x16 block along the reduction
// dimension, s = max|X| / 6 stored as E4M3, X^ = E2M1(X / s) with the stored s.
// Codes are packed two per byte (element 2i in the low nibble).  Scales are
// written as 512-byte atoms, one per 128 rows x 64 reduction elements: row r's
// four block scales at byte (r % 32) * 16 + (r / 32) * 4 (the layout the
// block-scaled MMA's scale copy reads).

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t h2 = cvt_e4m3x2_to_f16x2((uint16_t)(code & 0xFF));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

__device__ __noinline__ uint32_t e2m1_div_exact2(float x0, float x1, float d) {
  return cvt_e2m1x2(__fdiv_rn(x0, d), __fdiv_rn(x1, d));
}
// E2M1 codes of RN(x0 / d), RN(x1 / d) as one byte, exactly as
// cvt(__fdiv_rn(x, d)) gives them (same bracket argument as e4m3_code2).
__device__ __forceinline__ uint32_t e2m1_code2(float x0, float x1, float d, float rcp) {
  const float q0 = __fmul_rn(x0, rcp), q1 = __fmul_rn(x1, rcp);
  const float lo = 1.0f - 0x1p-19f, hi = 1.0f + 0x1p-19f;
  const uint32_t a = cvt_e2m1x2(__fmul_rn(q0, lo), __fmul_rn(q1, lo));
  const uint32_t b = cvt_e2m1x2(__fmul_rn(q0, hi), __fmul_rn(q1, hi));
  if (__builtin_expect(a == b && isfinite(q0) && isfinite(q1), 1)) return a;
  return e2m1_div_exact2(x0, x1, d);
}

// scale byte of a block with absolute maximum amax: E4M3(fl(amax / 6))
__device__ __forceinline__ uint32_t nvfp4_scale(float amax) {
  const float t = __fdiv_rn(amax, 6.0f);
  return cvt_e4m3x2(t, t) & 0xFF;
}

__device__ __forceinline__ size_t atom_off(int r, int blk) { return (size_t)(r & 31) * 16 + (r >> 5) * 4 + blk; }

// 128 rows of a [*, D] bf16 matrix -> codes [128][D/2] and scale atoms
// [D/64][512].  Mean: per-block (own_mean) or given (per channel) or none.
template <int D>
__device__ void fp4_row_block(const uint4 *__restrict__ src, int valid_rows, bool own_mean,
                              const float *__restrict__ given_mean, uint8_t *codes, uint8_t *atoms,
                              float *mean_out, int *status, int site, int src_stride = D / 8) {
  constexpr int VPR = D / 8, RPP = kThreads / VPR, PASSES = 128 / RPP;
  __shared__ long long ssum[RPP][D];
  __shared__ float smean[D];
  const int vc = threadIdx.x % VPR, rr = threadIdx.x / VPR;
  uint4 x[PASSES];
  bool bad = false;
#pragma unroll
  for (int pp = 0; pp < PASSES; ++pp) {
    const int r = rr + pp * RPP;
    x[pp] = (r < valid_rows) ? src[(size_t)r * src_stride + vc] : make_uint4(0, 0, 0, 0);
  }
  if (own_mean) {
    long long sacc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int pp = 0; pp < PASSES; ++pp) {
      if (rr + pp * RPP >= valid_rows) continue;
      float f[8];
      unpack_bf16x8(x[pp], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sacc[e] += fixed24(f[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) ssum[rr][vc * 8 + e] = sacc[e];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kThreads) {
      long long a = 0;
      for (int r = 0; r < RPP; ++r) a += ssum[r][c];
      smean[c] = mean_from_sum(a, valid_rows);
    }
  } else {
    for (int c = threadIdx.x; c < D; c += kThreads) smean[c] = given_mean ? given_mean[c] : 0.0f;
  }
  __syncthreads();
  float mu[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) mu[e] = smean[vc * 8 + e];
#pragma unroll
  for (int pp = 0; pp < PASSES; ++pp) {
    const int r = rr + pp * RPP;
    const bool valid = r < valid_rows;
    float f[8], g[8];
    unpack_bf16x8(x[pp], f);
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      bad |= valid && !in_range(f[e]);
      g[e] = __fsub_rn(f[e], mu[e]);
      amax = fmaxf(amax, fabsf(g[e]));
    }
    // the 16-channel block is this thread's 8 and its neighbour's
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const uint32_t sc = valid ? nvfp4_scale(amax) : 0;
    const float d = e4m3_value(sc);
    uint32_t w = 0;
    if (valid && d != 0.0f) {
      const float rcp = __frcp_rn(d);
#pragma unroll
      for (int e = 0; e < 8; e += 2) w |= e2m1_code2(g[e], g[e + 1], d, rcp) << (4 * e);
    }
    *reinterpret_cast<uint32_t *>(codes + (size_t)r * (D / 2) + vc * 4) = w;
    if ((vc & 1) == 0) {
      const int grp = vc >> 1;  // 16-channel block index along the row
      atoms[(size_t)(grp >> 2) * 512 + atom_off(r, grp & 3)] = (uint8_t)sc;
    }
  }
  if (bad) raise_status(status, SAGE_ERR_RANGE, site);
  if (mean_out)
    for (int c = threadIdx.x; c < D; c += kThreads) mean_out[c] = smean[c];
}

struct Fp4Args {
  const uint4 *q, *k, *v;
  int N, M, N_pad, M_pad, Tm, flags;
  int Hq, Hkv;
  const VarSeq *seq;  // packed sequences (kVar instances)
  uint8_t *qhat, *khat, *vhat, *qsf, *ksf, *vsf;
  const float *kbar, *vm;
  float *qbar;
  int *status;
  int nq, nk;
};

// kVar: packed sequences (each sequence's own lengths, packed [total, H, d] inputs)
template <int D, bool kVar>
__global__ void __launch_bounds__(kThreads) quantize_fp4_kernel(Fp4Args a) {
  int cta = blockIdx.x;
  if (cta < a.nq) {
    // ---- Q block (b, h, i) of 128 rows, optional per-block mean
    const int i = cta % a.Tm, bh = cta / a.Tm;
    const int r0 = i * 128;
    int Nb = a.N, stride = D / 8;
    const uint4 *src = a.q + ((size_t)bh * a.N + r0) * (D / 8);
    if constexpr (kVar) {
      const VarSeq sq = a.seq[bh / a.Hq];
      Nb = sq.N;
      stride = a.Hq * (D / 8);
      src = a.q + ((size_t)(sq.q0 + r0) * a.Hq + bh % a.Hq) * (D / 8);
    }
    const int valid = max(0, min(128, Nb - r0));
    fp4_row_block<D>(src, valid, (a.flags & SAGE_SMOOTH_Q) && valid > 0, nullptr,
                     a.qhat + ((size_t)bh * a.N_pad + r0) * (D / 2),
                     a.qsf + ((size_t)bh * a.Tm + i) * (D / 64) * 512, a.qbar + ((size_t)bh * a.Tm + i) * D,
                     a.status, 3, stride);
    return;
  }
  cta -= a.nq;
  const int nchunk = a.M_pad / 128;
  if (cta < a.nk) {
    // ---- K block (b, g, 128 rows) with k_bar over all tokens
    const int ch = cta % nchunk, hb = cta / nchunk;
    const int t0 = ch * 128;
    int Mb = a.M, stride = D / 8;
    const uint4 *src = a.k + ((size_t)hb * a.M + t0) * (D / 8);
    if constexpr (kVar) {
      const VarSeq sq = a.seq[hb / a.Hkv];
      Mb = sq.M;
      stride = a.Hkv * (D / 8);
      src = a.k + ((size_t)(sq.k0 + t0) * a.Hkv + hb % a.Hkv) * (D / 8);
    }
    const int valid = max(0, min(128, Mb - t0));
    fp4_row_block<D>(src, valid, false, a.kbar + (size_t)hb * D, a.khat + ((size_t)hb * a.M_pad + t0) * (D / 2),
                     a.ksf + ((size_t)hb * nchunk + ch) * (D / 64) * 512, nullptr, a.status, 1, stride);
    return;
  }
  cta -= a.nk;
  // ---- V chunk (b, g, 128 tokens): 1x16 blocks along tokens per channel,
  // codes transposed (token-contiguous per channel, two tokens per byte)
  {
    const int ch = cta % nchunk, hb = cta / nchunk;
    const int t0 = ch * 128;
    constexpr int VPR = D / 8, RPP = kThreads / VPR;
    constexpr int CA = (D + 127) / 128;  // channel atoms
    int Mb = a.M;  // this (b, kv-head)'s keys; rows hb * M + t, or (k0 + t) * Hkv + h packed
    long long vrow = (long long)hb * a.M, vstep = 1;
    if constexpr (kVar) {
      const VarSeq sq = a.seq[hb / a.Hkv];
      Mb = sq.M;
      vrow = (long long)sq.k0 * a.Hkv + hb % a.Hkv;
      vstep = a.Hkv;
    }
    __shared__ __nv_bfloat16 tile[128][D + 2];
    __shared__ float vmean[D];
    for (int c = threadIdx.x; c < D; c += kThreads) vmean[c] = a.vm[(size_t)hb * D + c];
    const int vc = threadIdx.x % VPR, rr = threadIdx.x / VPR;
    for (int r = rr; r < 128; r += RPP) {
      const int t = t0 + r;
      const size_t vi = kVar ? (size_t)(vrow + (long long)t * vstep) * VPR + vc : ((size_t)hb * a.M + t) * VPR + vc;
      const uint4 u = (t < Mb) ? a.v[vi] : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        *reinterpret_cast<uint32_t *>(&tile[r][vc * 8 + 2 * e]) = w[e];
    }
    __syncthreads();
    for (int item = threadIdx.x; item < D * 8; item += kThreads) {
      const int c = item % D, tb = item / D;  // channel, 16-token block of the chunk
      float g[16], amax = 0.0f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int t = t0 + tb * 16 + u;
        g[u] = (t < Mb) ? __fsub_rn(__bfloat162float(tile[tb * 16 + u][c]), vmean[c]) : 0.0f;
        amax = fmaxf(amax, fabsf(g[u]));
      }
      const bool any = t0 + tb * 16 < Mb;
      const uint32_t sc = any ? nvfp4_scale(amax) : 0;
      const float d = e4m3_value(sc);
      uint32_t w0 = 0, w1 = 0;
      if (d != 0.0f) {
        const float rcp = __frcp_rn(d);
#pragma unroll
        for (int u = 0; u < 8; u += 2) {
          const int t = t0 + tb * 16 + u;
          w0 |= (t < Mb ? e2m1_code2(g[u], g[u + 1], d, rcp) : 0) << (4 * u);
        }
#pragma unroll
        for (int u = 8; u < 16; u += 2) {
          const int t = t0 + tb * 16 + u;
          w1 |= (t < Mb ? e2m1_code2(g[u], g[u + 1], d, rcp) : 0) << (4 * (u - 8));
        }
      }
      // a token past M inside a pair contributes a zero nibble (its value is 0 anyway)
      *reinterpret_cast<uint2 *>(a.vhat + ((size_t)hb * D + c) * (a.M_pad / 2) + (t0 + tb * 16) / 2) =
          make_uint2(w0, w1);
      const int ts = (t0 + tb * 16) / 64, blk = ((t0 + tb * 16) % 64) / 16;
      a.vsf[(((size_t)hb * CA + c / 128) * (a.M_pad / 64) + ts) * 512 + atom_off(c % 128, blk)] = (uint8_t)sc;
    }
  }
}

}  // namespace

// Enqueue init, statistics, finalize and quantize on `stream`, with the
// statistics scratch at `st`.
// ------------------------------------------------------------------ SageBwd backward inputs
// One CTA per 128-row block of one (b, head): dO^ with the Q quantizer (no
// mean, scale fl(max|dO_i| / 127), the same binary32 steps, range check
// included), then D_r = sum_c dO[r,c] O[r,c] in fp32, the VPR threads of a row
// (consecutive lanes) combining their 8-channel partial sums by shuffles.
template <int D>
__global__ void __launch_bounds__(kThreads, kQuantCtas)
    bwd_prepare_kernel(const uint4 *__restrict__ o, const uint4 *__restrict__ dout, int N, int N_pad, int Tm,
                       uint8_t *doc, float *dos, float *drow, int *status) {
  constexpr int VPR = D / 8, RPP = kThreads / VPR;
  constexpr int kPool = qk_pool_bytes<D>();
  __shared__ __align__(16) unsigned char pool[kPool];
  const int i = blockIdx.x % Tm, bh = blockIdx.x / Tm;
  const int r0 = i * 128;
  const int valid = max(0, min(128, N - r0));
  quant_block<D, true>(dout + ((size_t)bh * N + r0) * VPR, valid, 128, false, nullptr,
                       doc + ((size_t)bh * N_pad + r0) * D * 2, dos + (size_t)bh * Tm + i, nullptr, status, 5, pool);
  const int vc = threadIdx.x % VPR, rr = threadIdx.x / VPR;
  for (int r = rr; r < 128; r += RPP) {  // every lane of a warp runs every shuffle
    float acc = 0.0f;
    if (r < valid) {
      float a[8], g[8];
      unpack_bf16x8(o[((size_t)bh * N + r0 + r) * VPR + vc], a);
      unpack_bf16x8(dout[((size_t)bh * N + r0 + r) * VPR + vc], g);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(a[e], g[e], acc);
    }
#pragma unroll
    for (int x = 1; x < VPR; x <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, x);
    if (vc == 0) drow[(size_t)bh * N_pad + r0 + r] = (r < valid) ? acc : 0.0f;
  }
}

sage_status launch_bwd_prepare(const sage_shape &s, const void *o, const void *dout, void *ws,
                               const sage_ws_layout &L, cudaStream_t stream) {
  char *w = (char *)ws;
  const unsigned grid = (unsigned)(s.B * s.Hq * L.Tm);
  auto kern = s.d == 64 ? bwd_prepare_kernel<64> : bwd_prepare_kernel<128>;
  kern<<<grid, kThreads, 0, stream>>>((const uint4 *)o, (const uint4 *)dout, s.N, L.N_pad, L.Tm,
                                      (uint8_t *)(w + L.doc), (float *)(w + L.dos), (float *)(w + L.drow),
                                      (int *)(w + L.status));
  return cudaGetLastError() == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}

// the quantize instance of a request: head dim, mode (INT8 / E4M3 Q and K;
// SageBwd V), per-row Q scales, packed sequences
template <bool kVar>
static void (*pick_quantize(int d, int mode, bool pr))(QuantArgs) {
  if (mode == SAGE_SAGEBWD_I8)
    return d == 64 ? (pr ? quantize_kernel<64, true, true, true, kVar> : quantize_kernel<64, true, false, true, kVar>)
                   : (pr ? quantize_kernel<128, true, true, true, kVar> : quantize_kernel<128, true, false, true, kVar>);
  if (mode == SAGE_Q8_PV8)
    return d == 64 ? (pr ? quantize_kernel<64, true, true, false, kVar> : quantize_kernel<64, true, false, false, kVar>)
                   : (pr ? quantize_kernel<128, true, true, false, kVar> : quantize_kernel<128, true, false, false, kVar>);
  return d == 64 ? (pr ? quantize_kernel<64, false, true, false, kVar> : quantize_kernel<64, false, false, false, kVar>)
                 : (pr ? quantize_kernel<128, false, true, false, kVar> : quantize_kernel<128, false, false, false, kVar>);
}

static sage_status enqueue_q8(const sage_shape &s, int mode, int flags, int bk, const void *q, const void *k,
                              const void *v, void *ws, const sage_ws_layout &L, StatsView st, cudaStream_t stream,
                              const VarSeq *seq = nullptr) {
  char *w = (char *)ws;
  int *status = (int *)(w + L.status);
  const int n = s.B * s.Hkv * s.d;
  init_kernel<<<(n + 255) / 256, 256, 0, stream>>>(st, n, status);
  dim3 sg((unsigned)cdiv(s.M, kStatTokens), (unsigned)(s.B * s.Hkv));
  if (s.d == 64)
    launch_stats<64>(sg, flags, k, v, s.M, st, status, stream, seq, s.Hkv);
  else
    launch_stats<128>(sg, flags, k, v, s.M, st, status, stream, seq, s.Hkv);
  finalize_kernel<<<(n + 255) / 256, 256, 0, stream>>>(st, n, s.M, flags, (float *)(w + L.kbar),
                                                        (float *)(w + L.vm), (float *)(w + L.dv), seq,
                                                        s.Hkv * s.d);
  if (mode == SAGE_NVFP4) {
    Fp4Args f;
    f.q = (const uint4 *)q;
    f.k = (const uint4 *)k;
    f.v = (const uint4 *)v;
    f.N = s.N;
    f.M = s.M;
    f.N_pad = L.N_pad;
    f.M_pad = L.M_pad;
    f.Tm = L.Tm;
    f.flags = flags;
    f.Hq = s.Hq;
    f.Hkv = s.Hkv;
    f.seq = seq;
    f.qhat = (uint8_t *)(w + L.qhat);
    f.khat = (uint8_t *)(w + L.khat);
    f.vhat = (uint8_t *)(w + L.vhat);
    f.qsf = (uint8_t *)(w + L.qsf);
    f.ksf = (uint8_t *)(w + L.ksf);
    f.vsf = (uint8_t *)(w + L.vsf);
    f.kbar = (const float *)(w + L.kbar);
    f.vm = (const float *)(w + L.vm);
    f.qbar = (float *)(w + L.qbar);
    f.status = status;
    f.nq = s.B * s.Hq * L.Tm;
    f.nk = s.B * s.Hkv * (L.M_pad / 128);
    const unsigned g4 = (unsigned)(f.nq + 2 * f.nk);  // Q blocks, K blocks, V chunks
    // the V-scale atoms of d = 64 use half their rows: clear them first
    if (s.d % 128 != 0 && cudaMemsetAsync(f.vsf, 0, L.stats - L.vsf, stream) != cudaSuccess) return SAGE_ERR_CUDA;
    auto fk = seq ? (s.d == 64 ? quantize_fp4_kernel<64, true> : quantize_fp4_kernel<128, true>)
                  : (s.d == 64 ? quantize_fp4_kernel<64, false> : quantize_fp4_kernel<128, false>);
    fk<<<g4, kThreads, 0, stream>>>(f);
    return cudaGetLastError() == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
  }
  QuantArgs a;
  a.q = (const uint4 *)q;
  a.k = (const uint4 *)k;
  a.v = (const uint4 *)v;
  a.B = s.B;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.N = s.N;
  a.M = s.M;
  a.N_pad = L.N_pad;
  a.M_pad = L.M_pad;
  a.Tm = L.Tm;
  a.Tn = L.Tn;
  a.bk = bk;
  a.mode = mode;
  a.flags = flags;
  a.qhat = (uint8_t *)(w + L.qhat);
  a.khat = (uint8_t *)(w + L.khat);
  a.vhat = (uint8_t *)(w + L.vhat);
  a.dq = (float *)(w + L.dq);
  a.dqt = (float *)(w + L.dqt);
  a.dvb = (float *)(w + L.dvb);
  a.seq = seq;
  a.qbar = (float *)(w + L.qbar);
  a.dk = (float *)(w + L.dk);
  a.kbar = (float *)(w + L.kbar);
  a.dv = (float *)(w + L.dv);
  a.vm = (float *)(w + L.vm);
  a.st = st;
  a.status = status;
  a.nq = s.B * s.Hq * L.Tm;
  a.nk = s.B * s.Hkv * L.Tn;
  const int nv = s.B * s.Hkv * (L.M_pad / 128);
  const unsigned grid = (unsigned)(a.nq + a.nk + nv);
  const bool pr = (flags & SAGE_Q_PER_TOKEN) != 0;
  void (*kern)(QuantArgs) = seq ? pick_quantize<true>(s.d, mode, pr) : pick_quantize<false>(s.d, mode, pr);
  kern<<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}

sage_status launch_quantize_q8(const sage_shape &s, int mode, int flags, int bq, int bk, const void *q,
                               const void *k, const void *v, void *ws, const sage_ws_layout &L,
                               cudaStream_t stream, const VarSeq *seq) {
  (void)bq;
  return enqueue_q8(s, mode, flags, bk, q, k, v, ws, L, stats_view(ws, L, s), stream, seq);
}

}  // namespace sage

// ---------------------------------------------------------------------------
// Pre-pass whose statistics scratch lives inside the library.
//
// The statistics pass needs B*Hkv*d * 24 bytes of device scratch (fixed-point
// column sums of K and V, V column min and max).  sage_quantize_qkv takes it
// from the caller's workspace.  This variant takes it from the fixed device
// array below instead, so a caller that is not allowed to obtain device memory
// for scratch — for example a plug-in whose host framework owns every device
// allocation, or a latency-critical caller that must not call cudaMalloc
// because it can synchronise the device — only has to provide the inputs and
// the output workspace.  The array is part of the library image: every GPU
// that loads the library holds it until the process exits.
//
// All calls share the one array and it keeps the previous call's contents: the
// init kernel clears it at the start of every call, and calls that overlap on
// the GPU (different streams, or several host threads) race on it.
namespace sage {

constexpr int kStaticStatsChannels = 32768;  // limit on B * Hkv * d
constexpr size_t kStaticStatsBytes = (size_t)kStaticStatsChannels * 24;
static __device__ __align__(256) unsigned char g_stats_scratch[kStaticStatsBytes];

// The device address of g_stats_scratch on each device, looked up once per
// device with that device current (host code cannot use the symbol's name as
// a device pointer).  The first call on a device does this look-up.
static void *static_scratch_address(int device) {
  constexpr int kMaxDevices = 64;
  static void *addr[kMaxDevices] = {};
  static std::mutex mu;
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[device]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_stats_scratch) != cudaSuccess) return nullptr;
    addr[device] = p;
  }
  return addr[device];
}

sage_status launch_quantize_q8_static_scratch(const sage_shape &s, int mode, int flags, int bq, int bk,
                                              const void *q, const void *k, const void *v, void *ws,
                                              const sage_ws_layout &L, cudaStream_t stream) {
  (void)bq;
  const int n = s.B * s.Hkv * s.d;
  if (n > kStaticStatsChannels) return SAGE_ERR_UNSUPPORTED;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return SAGE_ERR_CUDA;
  char *scratch = (char *)static_scratch_address(device);
  if (!scratch) return SAGE_ERR_CUDA;
  StatsView st;
  st.ksum = (int64_t *)scratch;
  st.vsum = (int64_t *)(scratch + (size_t)n * 8);
  st.vmin = (int *)(scratch + (size_t)n * 16);
  st.vmax = (int *)(scratch + (size_t)n * 20);

  return enqueue_q8(s, mode, flags, bk, q, k, v, ws, L, st, stream);
}

}  // namespace sage
