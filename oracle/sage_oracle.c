/*
 * Oracle for SageAttention-style quantized attention forward — TEST
 * INFRASTRUCTURE ONLY (see sage_oracle.h).  Plain loops, no blocking or
 * fusion beyond what the method itself states.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 * (contraction off so every binary32 step below rounds exactly once).
 */
#include "sage_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Codecs                                                               */
/* ------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("FN"): sign, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 is subnormal (m * 2^-9).  No infinities; S.1111.111 is NaN,
 * so the largest finite magnitude is 1.75 * 2^8 = 448 (the value the
 * SageAttention2 summary §3.4 "FP8 Quantization for P~V" scales P~ to). */
double orc_e4m3_decode(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* FP4 E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit, no inf / NaN.
 * Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} (SageAttention3 summary §3.4
 * "The NVFP4 Microscaling Format"). */
double orc_e2m1_decode(uint8_t code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double v;
  if (e == 0)
    v = 0.5 * m;
  else
    v = ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

static double e4m3_mag(int c) { return orc_e4m3_decode((uint8_t)c); }
static double e2m1_mag(int c) { return orc_e2m1_decode((uint8_t)c); }

/* Magnitude code nearest to a >= 0 among codes 0..maxcode of a format whose
 * magnitudes increase with the code; ties go to the even code (the one whose
 * mantissa lsb is 0); a at or above the largest finite value saturates. */
static int nearest_code(double a, double (*mag)(int), int maxcode) {
  int c;
  double mid;
  if (a >= mag(maxcode)) return maxcode;
  for (c = 0; c < maxcode && mag(c + 1) <= a; ++c) {
  }
  if (mag(c) == a) return c;
  mid = 0.5 * (mag(c) + mag(c + 1)); /* exact: both are short dyadic rationals */
  if (a < mid) return c;
  if (a > mid) return c + 1;
  return (c % 2 == 0) ? c : c + 1;
}

uint8_t orc_e4m3_encode(double x) {
  int sign = signbit(x) ? 0x80 : 0;
  if (isnan(x)) return 0x7F;
  return (uint8_t)(sign | nearest_code(fabs(x), e4m3_mag, 126));
}

uint8_t orc_e2m1_encode(double x) {
  int sign = signbit(x) ? 0x8 : 0;
  if (isnan(x)) return 0x7; /* no NaN in E2M1; never reached for checked inputs */
  return (uint8_t)(sign | nearest_code(fabs(x), e2m1_mag, 7));
}

double orc_bf16_decode(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* bf16: 8 significand bits, exponent range of binary32, subnormal spacing 2^-133. */
uint16_t orc_bf16_encode(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x), r, y;
  int e, ulp_exp;
  float f;
  uint32_t u;
  if (isnan(x)) return 0x7FC0;
  if (a == 0.0) return sign;
  frexp(a, &e); /* a in [2^(e-1), 2^e) */
  ulp_exp = e - 8;
  if (ulp_exp < -133) ulp_exp = -133;
  r = nearbyint(ldexp(a, -ulp_exp)); /* default rounding mode: ties to even */
  y = ldexp(r, ulp_exp);
  if (y >= 0x1p128) return (uint16_t)(sign | 0x7F80);
  f = (float)y; /* exact: y has at most 8 significant bits */
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

void orc_e4m3_encode_array(const float *x, int64_t n, uint8_t *out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = orc_e4m3_encode((double)x[i]);
}

void orc_e2m1_encode_array(const float *x, int64_t n, uint8_t *out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = orc_e2m1_encode((double)x[i]);
}

void orc_bf16_encode_array(const double *x, int64_t n, uint16_t *out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = orc_bf16_encode(x[i]);
}

static float bf16f(uint16_t bits) { return (float)orc_bf16_decode(bits); }

/* ------------------------------------------------------------------ */
/* Quantizer building blocks (binary32)                                 */
/* ------------------------------------------------------------------ */

static int in_range(float f) { return isfinite(f) && fabsf(f) < 65536.0f; }

/* Mean over tokens, used for k_bar, V_m (per head) and q_bar_i (per query
 * block) — SageAttention2 summary §3.4 "Smoothing Q": mean(K) over all tokens,
 * mean(Q_i) over the block; "Optional Smoothing of V": mean(V, axis=0).
 * To make the mean a fixed function of the inputs (independent of summation
 * order) each value is taken as a fixed-point integer with lsb 2^-24
 * (truncated toward zero, which only touches |x| < 2^-17), the integers are
 * summed exactly, and the sum is converted once to double and divided once. */
int orc_mean_bf16(const uint16_t *x, int64_t n, int64_t stride, float *mean) {
  int64_t acc = 0, i;
  for (i = 0; i < n; ++i) {
    float f = bf16f(x[i * stride]);
    if (!in_range(f)) return ORC_ERR_RANGE;
    acc += (int64_t)(f * 16777216.0f); /* exact product; cast truncates toward zero */
  }
  *mean = (n > 0) ? (float)(((double)acc * 0x1p-24) / (double)n) : 0.0f;
  return ORC_OK;
}

/* Per-block INT8: delta = max|X| / 127, X^ = round(X / delta) (SageAttention3
 * summary §3.4 "SageBwd Forward Pass"; the "Quantization for Attention"
 * page's quant_int8 / quant_sym).  Round half to even, clamp to +-127. */
float orc_int8_scale(float absmax) { return absmax / 127.0f; }

int orc_int8_code(float x, float scale) {
  float t, r;
  if (scale == 0.0f) return 0;
  t = x / scale;
  r = rintf(t);
  if (r > 127.0f) r = 127.0f;
  if (r < -127.0f) r = -127.0f;
  return (int)r;
}

/* Per-block / per-channel E4M3: delta = max|X| / 448, X^ = e4m3(X / delta)
 * (SageAttention2 summary §3.4, delta_V[c] = max|V[:,c]| / 448). */
float orc_fp8_scale(float absmax) { return absmax / 448.0f; }

uint8_t orc_fp8_code(float x, float scale) {
  if (scale == 0.0f) return 0;
  return orc_e4m3_encode((double)(x / scale));
}

/* NVFP4 phi: s = max|X| / 6 stored as E4M3, X^ = round(X / s) to E2M1
 * (SageAttention3 summary §3.4, eq. for phi).  The division uses the stored
 * (E4M3-rounded) scale, the one the block-scaled product multiplies back. */
uint8_t orc_nvfp4_scale(float absmax) { return orc_e4m3_encode((double)(absmax / 6.0f)); }

uint8_t orc_nvfp4_code(float x, uint8_t scale_code) {
  float s = (float)orc_e4m3_decode(scale_code);
  if (s == 0.0f) return 0;
  return orc_e2m1_encode((double)(x / s));
}

/* ------------------------------------------------------------------ */
/* Quantization of Q, K, V                                              */
/* ------------------------------------------------------------------ */

static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Q and K take the INT8 per-block quantizer in mode 0 and in the SageBwd
 * forward (mode 3), the E4M3 one in mode 1 */
static int int8_qk(int mode) { return mode == ORC_Q8_PV8 || mode == ORC_SAGEBWD_I8; }

static int check_shape(const orc_shape *s, int mode, int bq, int bk) {
  if (!s || s->B <= 0 || s->Hq <= 0 || s->Hkv <= 0 || s->N <= 0 || s->M <= 0 || s->d <= 0)
    return ORC_ERR_ARG;
  if (s->Hq % s->Hkv != 0 || bq <= 0 || bk <= 0) return ORC_ERR_ARG;
  if (mode < 0 || mode > 3) return ORC_ERR_ARG;
  if (mode == ORC_NVFP4 && (s->d % 16 != 0 || bk % 16 != 0)) return ORC_ERR_ARG;
  if ((int64_t)s->M > ((int64_t)1 << 23) || (int64_t)s->N > ((int64_t)1 << 23)) return ORC_ERR_ARG;
  return ORC_OK;
}

int orc_quantize(const orc_shape *s, int mode, int flags, int bq, int bk, const uint16_t *q,
                 const uint16_t *k, const uint16_t *v, orc_quant *out) {
  const int B = s->B, Hq = s->Hq, Hkv = s->Hkv, N = s->N, M = s->M, d = s->d;
  const int64_t Tm = cdiv(N, bq), Tn = cdiv(M, bk), G16 = d / 16, Mt16 = cdiv(M, 16);
  int64_t i, n;
  int b, h, c, t, rc;
  float *g; /* one smoothed row / block, binary32 */

  rc = check_shape(s, mode, bq, bk);
  if (rc) return rc;

  /* inputs must be finite and below 2^16 in magnitude */
  n = (int64_t)B * Hq * N * d;
  for (i = 0; i < n; ++i)
    if (!in_range(bf16f(q[i]))) return ORC_ERR_RANGE;
  n = (int64_t)B * Hkv * M * d;
  for (i = 0; i < n; ++i)
    if (!in_range(bf16f(k[i])) || !in_range(bf16f(v[i]))) return ORC_ERR_RANGE;

  g = (float *)malloc(sizeof(float) * (size_t)((int64_t)(bq > bk ? bq : bk) * d + (int64_t)M * d));
  if (!g) return ORC_ERR_ARG;

  for (b = 0; b < B; ++b) {
    for (h = 0; h < Hkv; ++h) {
      const int64_t hb = (int64_t)b * Hkv + h;
      const uint16_t *K = k + hb * M * d, *V = v + hb * M * d;
      float *kbar = out->kbar + hb * d, *vm = out->vm + hb * d;

      /* K: k_bar = mean over all valid tokens (SageAttention2 summary §3.4,
       * "K is smoothed once: K = K - mean(K)"), gamma(K) = K - k_bar. */
      for (c = 0; c < d; ++c) {
        kbar[c] = 0.0f;
        if (flags & ORC_SMOOTH_K) orc_mean_bf16(K + c, M, d, &kbar[c]);
      }
      if (mode == ORC_NVFP4) {
        for (t = 0; t < M; ++t) {
          int64_t gi;
          for (gi = 0; gi < G16; ++gi) {
            float amax = 0.0f, gg[16];
            uint8_t sc;
            int e;
            for (e = 0; e < 16; ++e) {
              int cc = (int)(gi * 16 + e);
              gg[e] = bf16f(K[(int64_t)t * d + cc]) - kbar[cc];
              if (fabsf(gg[e]) > amax) amax = fabsf(gg[e]);
            }
            sc = orc_nvfp4_scale(amax);
            out->ks[(hb * M + t) * G16 + gi] = sc;
            for (e = 0; e < 16; ++e)
              out->kc[(hb * M + t) * d + gi * 16 + e] = orc_nvfp4_code(gg[e], sc);
          }
        }
      } else {
        int64_t j;
        for (j = 0; j < Tn; ++j) {
          const int t0 = (int)(j * bk), t1 = (int)((j + 1) * bk < M ? (j + 1) * bk : M);
          float amax = 0.0f, sc;
          for (t = t0; t < t1; ++t)
            for (c = 0; c < d; ++c) {
              float x = bf16f(K[(int64_t)t * d + c]) - kbar[c];
              g[(int64_t)(t - t0) * d + c] = x;
              if (fabsf(x) > amax) amax = fabsf(x);
            }
          sc = int8_qk(mode) ? orc_int8_scale(amax) : orc_fp8_scale(amax);
          out->dk[hb * Tn + j] = sc;
          for (t = t0; t < t1; ++t)
            for (c = 0; c < d; ++c) {
              float x = g[(int64_t)(t - t0) * d + c];
              out->kc[(hb * M + t) * d + c] = int8_qk(mode)
                                                  ? (uint8_t)(int8_t)orc_int8_code(x, sc)
                                                  : orc_fp8_code(x, sc);
            }
        }
      }

      /* V: V_m = mean(V, axis=0) if smoothed ("Optional Smoothing of V"),
       * V' = V - V_m; FP8 modes: delta_V[c] = max over tokens |V'[:,c]| / 448;
       * NVFP4: phi over 1x16 blocks along tokens (the reduction dimension of
       * P~V), per channel. */
      for (c = 0; c < d; ++c) {
        vm[c] = 0.0f;
        if (flags & ORC_SMOOTH_V) orc_mean_bf16(V + c, M, d, &vm[c]);
      }
      for (t = 0; t < M; ++t)
        for (c = 0; c < d; ++c) g[(int64_t)t * d + c] = bf16f(V[(int64_t)t * d + c]) - vm[c];
      if (mode == ORC_NVFP4) {
        int64_t tb;
        for (c = 0; c < d; ++c)
          for (tb = 0; tb < Mt16; ++tb) {
            const int t0 = (int)(tb * 16), t1 = (int)(tb * 16 + 16 < M ? tb * 16 + 16 : M);
            float amax = 0.0f;
            uint8_t sc;
            for (t = t0; t < t1; ++t)
              if (fabsf(g[(int64_t)t * d + c]) > amax) amax = fabsf(g[(int64_t)t * d + c]);
            sc = orc_nvfp4_scale(amax);
            out->vs[(hb * Mt16 + tb) * d + c] = sc;
            for (t = t0; t < t1; ++t)
              out->vc[(hb * M + t) * d + c] = orc_nvfp4_code(g[(int64_t)t * d + c], sc);
          }
      } else if (mode == ORC_SAGEBWD_I8) {
        /* SageBwd: per-block INT8 of V' over each bk-token block and all d
         * channels, s_V = max|V'_j| / 127 (the same quantizer as Q and K) */
        int64_t j;
        for (j = 0; j < Tn; ++j) {
          const int t0 = (int)(j * bk), t1 = (int)((j + 1) * bk < M ? (j + 1) * bk : M);
          float amax = 0.0f, sc;
          for (t = t0; t < t1; ++t)
            for (c = 0; c < d; ++c)
              if (fabsf(g[(int64_t)t * d + c]) > amax) amax = fabsf(g[(int64_t)t * d + c]);
          sc = orc_int8_scale(amax);
          out->dvb[hb * Tn + j] = sc;
          for (t = t0; t < t1; ++t)
            for (c = 0; c < d; ++c)
              out->vc[(hb * M + t) * d + c] = (uint8_t)(int8_t)orc_int8_code(g[(int64_t)t * d + c], sc);
        }
      } else {
        float *dv = out->dv + hb * d;
        for (c = 0; c < d; ++c) {
          float amax = 0.0f;
          for (t = 0; t < M; ++t)
            if (fabsf(g[(int64_t)t * d + c]) > amax) amax = fabsf(g[(int64_t)t * d + c]);
          dv[c] = orc_fp8_scale(amax);
          for (t = 0; t < M; ++t)
            out->vc[(hb * M + t) * d + c] = orc_fp8_code(g[(int64_t)t * d + c], dv[c]);
        }
      }
    }

    /* Q: per block i of bq rows, q_bar_i = mean over the block's valid rows
     * if smoothed (SageAttention2 summary §3.4, gamma(Q_i) = Q_i - q_bar_i),
     * then per-block scale (modes 0, 1) or phi per 1x16 along d (mode 2). */
    for (h = 0; h < Hq; ++h) {
      const int64_t hb = (int64_t)b * Hq + h;
      const uint16_t *Q = q + hb * N * d;
      int64_t ib;
      for (ib = 0; ib < Tm; ++ib) {
        const int r0 = (int)(ib * bq), r1 = (int)((ib + 1) * bq < N ? (ib + 1) * bq : N);
        float *qbar = out->qbar + (hb * Tm + ib) * d;
        int r;
        for (c = 0; c < d; ++c) {
          qbar[c] = 0.0f;
          if (flags & ORC_SMOOTH_Q) orc_mean_bf16(Q + (int64_t)r0 * d + c, r1 - r0, d, &qbar[c]);
        }
        for (r = r0; r < r1; ++r)
          for (c = 0; c < d; ++c)
            g[(int64_t)(r - r0) * d + c] = bf16f(Q[(int64_t)r * d + c]) - qbar[c];
        if (mode == ORC_NVFP4) {
          for (r = r0; r < r1; ++r) {
            int64_t gi;
            for (gi = 0; gi < G16; ++gi) {
              float amax = 0.0f;
              uint8_t sc;
              int e;
              for (e = 0; e < 16; ++e) {
                float x = g[(int64_t)(r - r0) * d + gi * 16 + e];
                if (fabsf(x) > amax) amax = fabsf(x);
              }
              sc = orc_nvfp4_scale(amax);
              out->qs[(hb * N + r) * G16 + gi] = sc;
              for (e = 0; e < 16; ++e)
                out->qc[(hb * N + r) * d + gi * 16 + e] =
                    orc_nvfp4_code(g[(int64_t)(r - r0) * d + gi * 16 + e], sc);
            }
          }
        } else if (flags & ORC_Q_PER_TOKEN) {
          /* one scale per row of gamma(Q_i) */
          out->dq[hb * Tm + ib] = 0.0f;
          for (r = r0; r < r1; ++r) {
            float amax = 0.0f, sc;
            for (c = 0; c < d; ++c)
              if (fabsf(g[(int64_t)(r - r0) * d + c]) > amax) amax = fabsf(g[(int64_t)(r - r0) * d + c]);
            sc = int8_qk(mode) ? orc_int8_scale(amax) : orc_fp8_scale(amax);
            out->dqt[hb * N + r] = sc;
            for (c = 0; c < d; ++c) {
              float x = g[(int64_t)(r - r0) * d + c];
              out->qc[(hb * N + r) * d + c] = int8_qk(mode) ? (uint8_t)(int8_t)orc_int8_code(x, sc)
                                                                   : orc_fp8_code(x, sc);
            }
          }
        } else {
          float amax = 0.0f, sc;
          for (r = r0; r < r1; ++r)
            for (c = 0; c < d; ++c)
              if (fabsf(g[(int64_t)(r - r0) * d + c]) > amax) amax = fabsf(g[(int64_t)(r - r0) * d + c]);
          sc = int8_qk(mode) ? orc_int8_scale(amax) : orc_fp8_scale(amax);
          out->dq[hb * Tm + ib] = sc;
          for (r = r0; r < r1; ++r)
            for (c = 0; c < d; ++c) {
              float x = g[(int64_t)(r - r0) * d + c];
              out->qc[(hb * N + r) * d + c] = int8_qk(mode)
                                                  ? (uint8_t)(int8_t)orc_int8_code(x, sc)
                                                  : orc_fp8_code(x, sc);
            }
        }
      }
    }
  }
  free(g);
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Attention                                                            */
/* ------------------------------------------------------------------ */

/* key c is visible to query r: bottom-right aligned causal mask */
static int visible(int causal, int r, int c, int N, int M) {
  if (c >= M) return 0;
  if (!causal) return 1;
  return c <= r + (M - N);
}

/* Dequantized smoothed Q row (gamma(Q) reconstructed from codes and scales). */
static void deq_q_row(const orc_shape *s, int mode, int flags, int bq, const uint16_t *q,
                      const orc_quant *qz, int64_t hb, int r, double *out) {
  const int d = s->d, N = s->N;
  const int64_t Tm = cdiv(N, bq), ib = r / bq;
  const float *qbar = qz->qbar + (hb * Tm + ib) * d;
  const double sq = (flags & ORC_Q_PER_TOKEN) ? (double)qz->dqt[hb * N + r] : (double)qz->dq[hb * Tm + ib];
  int c;
  for (c = 0; c < d; ++c) {
    const int64_t e = (hb * N + r) * d + c;
    if (flags & ORC_EXACT_QK)
      out[c] = orc_bf16_decode(q[e]) - (double)qbar[c];
    else if (int8_qk(mode))
      out[c] = sq * (double)(int8_t)qz->qc[e];
    else if (mode == ORC_QF8_PV8)
      out[c] = sq * orc_e4m3_decode(qz->qc[e]);
    else
      out[c] = orc_e4m3_decode(qz->qs[(hb * N + r) * (d / 16) + c / 16]) * orc_e2m1_decode(qz->qc[e]);
  }
}

/* Dequantized smoothed K row t of kv-head hb (gamma(K) from codes and scales). */
static void deq_k_row(const orc_shape *s, int mode, int flags, int bk, const uint16_t *k,
                      const orc_quant *qz, int64_t hb, int t, double *out) {
  const int d = s->d, M = s->M;
  const int64_t Tn = cdiv(M, bk);
  int c;
  for (c = 0; c < d; ++c) {
    const int64_t e = (hb * M + t) * d + c;
    if (flags & ORC_EXACT_QK)
      out[c] = orc_bf16_decode(k[e]) - (double)qz->kbar[hb * d + c];
    else if (int8_qk(mode))
      out[c] = (double)qz->dk[hb * Tn + t / bk] * (double)(int8_t)qz->kc[e];
    else if (mode == ORC_QF8_PV8)
      out[c] = (double)qz->dk[hb * Tn + t / bk] * orc_e4m3_decode(qz->kc[e]);
    else
      out[c] = orc_e4m3_decode(qz->ks[(hb * M + t) * (d / 16) + c / 16]) * orc_e2m1_decode(qz->kc[e]);
  }
}

int orc_attn_rows_lse(const orc_shape *s, int mode, int flags, int bq, int bk, int causal,
                      double sm_scale, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const orc_quant *qz, const int64_t *rows, int64_t nrows, double *out,
                      double *lse) {
  const int Hq = s->Hq, Hkv = s->Hkv, N = s->N, M = s->M, d = s->d;
  const int64_t Tn = cdiv(M, bk), Mt16 = cdiv(M, 16);
  double *qrow, *krow, *sv, *pv, *R, *O, *vrow;
  int64_t ri;
  int rc = check_shape(s, mode, bq, bk);
  if (rc) return rc;
  if (causal && N > M) return ORC_ERR_ARG; /* bottom-right alignment needs M >= N */

  qrow = (double *)malloc(sizeof(double) * d);
  krow = (double *)malloc(sizeof(double) * d);
  vrow = (double *)malloc(sizeof(double) * d);
  sv = (double *)malloc(sizeof(double) * bk);
  pv = (double *)malloc(sizeof(double) * bk);
  R = (double *)malloc(sizeof(double) * d);
  O = (double *)malloc(sizeof(double) * d);
  if (!qrow || !krow || !vrow || !sv || !pv || !R || !O) return ORC_ERR_ARG;

  for (ri = 0; ri < nrows; ++ri) {
    const int64_t row = rows[ri];
    const int64_t bh = row / N; /* b*Hq + h */
    const int r = (int)(row % N);
    const int b = (int)(bh / Hq), h = (int)(bh % Hq);
    const int64_t hk = (int64_t)b * Hkv + h / (Hq / Hkv); /* kv head of this query head */
    const int64_t Tm = cdiv(N, bq);
    const float *qbar = qz->qbar + (bh * Tm + r / bq) * d;
    double m = -INFINITY, l = 0.0;
    int64_t j;
    int c, e;

    deq_q_row(s, mode, flags, bq, q, qz, bh, r, qrow);
    for (c = 0; c < d; ++c) O[c] = 0.0;

    for (j = 0; j < Tn; ++j) {
      const int kb = (int)(j * bk);
      double mt = -INFINITY, m_new, alpha, sP1 = 0.0, sP = 0.0;

      /* S_ij = deq(Q^_i) deq(K^_j)^T + dS_ij, dS_ij = q_bar_i deq(K^_j)^T,
       * then times sm_scale (SageAttention2 summary §3.4 "Smoothing Q"). */
      for (c = 0; c < bk; ++c) {
        const int t = kb + c;
        sv[c] = -INFINITY;
        if (visible(causal, r, t, N, M)) {
          double s0 = 0.0, ds = 0.0;
          deq_k_row(s, mode, flags, bk, k, qz, hk, t, krow);
          for (e = 0; e < d; ++e) s0 += qrow[e] * krow[e];
          if (flags & ORC_SMOOTH_Q)
            for (e = 0; e < d; ++e) ds += (double)qbar[e] * krow[e];
          sv[c] = (s0 + ds) * sm_scale;
        }
        if (sv[c] > mt) mt = sv[c];
      }

      /* online softmax: m_ij = max(m_i,j-1, rowmax S_ij), P~ = exp(S - m_ij),
       * l_ij = e^(m_i,j-1 - m_ij) l + rowsum P~ (unquantized P~). */
      m_new = (mt > m) ? mt : m;
      if (m_new == -INFINITY) {
        alpha = 1.0;
        for (c = 0; c < bk; ++c) pv[c] = 0.0;
      } else {
        alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        for (c = 0; c < bk; ++c) pv[c] = (sv[c] == -INFINITY) ? 0.0 : exp(sv[c] - m_new);
      }
      {
        double rs = 0.0;
        for (c = 0; c < bk; ++c) rs += pv[c];
        l = alpha * l + rs;
      }

      /* tile partial R_ij, accumulated over this tile's keys only */
      for (e = 0; e < d; ++e) R[e] = 0.0;
      if (flags & ORC_EXACT_PV) {
        for (c = 0; c < bk; ++c) {
          const int t = kb + c;
          if (pv[c] == 0.0) continue;
          for (e = 0; e < d; ++e)
            R[e] += pv[c] * (orc_bf16_decode(v[(hk * M + t) * d + e]) - (double)qz->vm[hk * d + e]);
        }
      } else if (mode == ORC_SAGEBWD_I8) {
        /* SageBwd per-token P~ (SageAttention3 summary, "SageBwd Forward
         * Pass"): s_P = exp(rowmax S_ij - m_ij) / 127, the row's largest P~ of
         * this tile over 127; P^ = round(P~ / s_P), ties to even; R = P^ V^ in
         * integers, dequantized by s_P s_V,j in the accumulation below */
        sP = (mt == -INFINITY) ? 0.0 : exp(mt - m_new) / 127.0;
        for (c = 0; c < bk; ++c) {
          const int t = kb + c;
          double ph;
          if (sP == 0.0 || pv[c] == 0.0) continue;
          ph = nearbyint(pv[c] / sP);
          if (ph > 127.0) ph = 127.0;
          if (ph == 0.0) continue;
          for (e = 0; e < d; ++e) R[e] += ph * (double)(int8_t)qz->vc[(hk * M + t) * d + e];
        }
      } else if (mode != ORC_NVFP4) {
        /* P^ = e4m3(P~ * 448) (static scale 1/448), R = P^ V^ */
        for (c = 0; c < bk; ++c) {
          const int t = kb + c;
          double ph = orc_e4m3_decode(orc_e4m3_encode(pv[c] * 448.0));
          if (ph == 0.0) continue;
          for (e = 0; e < d; ++e) R[e] += ph * orc_e4m3_decode(qz->vc[(hk * M + t) * d + e]);
        }
      } else {
        /* two-level P~ (SageAttention3 summary §3.4): s_P1 = rowmax(P~)/(448*6)
         * with rowmax(P~_ij) = exp(rowmax S_ij - m_ij); P2 = P~ / s_P1;
         * s_P2, P2^ = phi(P2) over 1x16 blocks; R = (P2^ s_P2)(V^ s_V).
         * ORC_P_DIRECT: s_P1 = 1, phi on P~ itself. */
        int u;
        sP1 = (mt == -INFINITY) ? 0.0 : (flags & ORC_P_DIRECT) ? 1.0 : exp(mt - m_new) / (448.0 * 6.0);
        for (u = 0; u < bk; u += 16) {
          double p2[16], amax = 0.0, s2;
          uint8_t s2c;
          for (c = 0; c < 16; ++c) {
            p2[c] = (sP1 == 0.0) ? 0.0 : pv[u + c] / sP1;
            if (p2[c] > amax) amax = p2[c];
          }
          s2c = orc_e4m3_encode(amax / 6.0);
          s2 = orc_e4m3_decode(s2c);
          for (c = 0; c < 16; ++c) {
            const int t = kb + u + c;
            double ph;
            if (s2 == 0.0 || t >= M) continue;
            ph = orc_e2m1_decode(orc_e2m1_encode(p2[c] / s2)) * s2;
            if (ph == 0.0) continue;
            for (e = 0; e < d; ++e) {
              double vv = orc_e2m1_decode(qz->vc[(hk * M + t) * d + e]) *
                          orc_e4m3_decode(qz->vs[(hk * Mt16 + t / 16) * d + e]);
              R[e] += ph * vv;
            }
          }
        }
      }

      /* two-level accumulation: O_ij = diag(e^(m_i,j-1 - m_ij)) O_i,j-1 + R_ij
       * (FP4 mode: + s_P1 R_ij; SageBwd: + s_P s_V,j R_ij) */
      {
        double rsc = 1.0;
        if (!(flags & ORC_EXACT_PV) && mode == ORC_NVFP4) rsc = sP1;
        if (!(flags & ORC_EXACT_PV) && mode == ORC_SAGEBWD_I8) rsc = sP * (double)qz->dvb[hk * Tn + j];
        for (e = 0; e < d; ++e) O[e] = alpha * O[e] + rsc * R[e];
      }
      m = m_new;
    }

    /* O_i = diag(l)^-1 O / 448 * delta_V (FP8 P~ / V), or O / l (NVFP4, whose
     * scales are inside the product), plus V_m when V was smoothed. */
    for (e = 0; e < d; ++e) {
      double o = O[e] / l;
      if (!(flags & ORC_EXACT_PV) && (mode == ORC_Q8_PV8 || mode == ORC_QF8_PV8))
        o = o / 448.0 * (double)qz->dv[hk * d + e];
      vrow[e] = o + (double)qz->vm[hk * d + e];
      out[ri * d + e] = vrow[e];
    }
    if (lse) lse[ri] = m + log(l);
  }
  free(qrow);
  free(krow);
  free(vrow);
  free(sv);
  free(pv);
  free(R);
  free(O);
  return ORC_OK;
}

int orc_attn_rows(const orc_shape *s, int mode, int flags, int bq, int bk, int causal,
                  double sm_scale, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const orc_quant *qz, const int64_t *rows, int64_t nrows, double *out) {
  return orc_attn_rows_lse(s, mode, flags, bq, bk, causal, sm_scale, q, k, v, qz, rows, nrows, out,
                           NULL);
}

int orc_attn_exact_rows(const orc_shape *s, int causal, double sm_scale, const uint16_t *q,
                        const uint16_t *k, const uint16_t *v, const int64_t *rows, int64_t nrows,
                        double *out) {
  const int Hq = s->Hq, Hkv = s->Hkv, N = s->N, M = s->M, d = s->d;
  double *sc = (double *)malloc(sizeof(double) * M);
  int64_t ri;
  if (!sc) return ORC_ERR_ARG;
  if (causal && N > M) {
    free(sc);
    return ORC_ERR_ARG;
  }
  for (ri = 0; ri < nrows; ++ri) {
    const int64_t row = rows[ri], bh = row / N;
    const int r = (int)(row % N), b = (int)(bh / Hq), h = (int)(bh % Hq);
    const int64_t hk = (int64_t)b * Hkv + h / (Hq / Hkv);
    double mx = -INFINITY, sum = 0.0;
    int t, e;
    for (t = 0; t < M; ++t) {
      sc[t] = -INFINITY;
      if (visible(causal, r, t, N, M)) {
        double acc = 0.0;
        for (e = 0; e < d; ++e)
          acc += orc_bf16_decode(q[(bh * N + r) * d + e]) * orc_bf16_decode(k[(hk * M + t) * d + e]);
        sc[t] = acc * sm_scale;
      }
      if (sc[t] > mx) mx = sc[t];
    }
    for (t = 0; t < M; ++t) {
      sc[t] = (sc[t] == -INFINITY) ? 0.0 : exp(sc[t] - mx);
      sum += sc[t];
    }
    for (e = 0; e < d; ++e) {
      double acc = 0.0;
      for (t = 0; t < M; ++t)
        if (sc[t] != 0.0) acc += sc[t] * orc_bf16_decode(v[(hk * M + t) * d + e]);
      out[ri * d + e] = acc / sum;
    }
  }
  free(sc);
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* SageBwd backward                                                     */
/* ------------------------------------------------------------------ */

/* INT8 per-block code of a value in fp64 against an fp64 scale (P and dS are
 * formed inside the backward, not in a binary32 pre-pass): round half to
 * even, clamp to +-127, 0 when the block is all zero. */
static double int8_code64(double x, double scale) {
  double r;
  if (scale == 0.0) return 0.0;
  r = nearbyint(x / scale);
  if (r > 127.0) r = 127.0;
  if (r < -127.0) r = -127.0;
  return r;
}

/* The backward's inputs of one head: dO^ per bq-row block (binary32, as Q
 * in the forward: a pre-pass quantizer) and D_r = sum_e dO[r,e] O[r,e]. */
static void sagebwd_prepare_head(const uint16_t *dO, const double *O, int N, int d, int bq, int8_t *doc,
                                 float *dos, double *Dr) {
  const int64_t Tm = cdiv(N, bq);
  int64_t i;
  int r, e;
  for (i = 0; i < Tm; ++i) {
    const int r0 = (int)(i * bq), r1 = (int)((i + 1) * bq < N ? (i + 1) * bq : N);
    float amax = 0.0f;
    for (r = r0; r < r1; ++r)
      for (e = 0; e < d; ++e)
        if (fabsf(bf16f(dO[(int64_t)r * d + e])) > amax) amax = fabsf(bf16f(dO[(int64_t)r * d + e]));
    dos[i] = orc_int8_scale(amax);
    for (r = r0; r < r1; ++r)
      for (e = 0; e < d; ++e) doc[(int64_t)r * d + e] = (int8_t)orc_int8_code(bf16f(dO[(int64_t)r * d + e]), dos[i]);
  }
  for (r = 0; r < N; ++r) {
    double acc = 0.0;
    for (e = 0; e < d; ++e) acc += orc_bf16_decode(dO[(int64_t)r * d + e]) * O[(int64_t)r * d + e];
    Dr[r] = acc;
  }
}

int orc_sagebwd_prepare(const orc_shape *s, int bq, const double *o, const uint16_t *dout, int8_t *doc,
                        float *dos, double *D) {
  const int64_t N = s->N, d = s->d, Tm = cdiv(s->N, bq);
  int64_t bh, n;
  int rc = check_shape(s, ORC_SAGEBWD_I8, bq, 64);
  if (rc) return rc;
  n = (int64_t)s->B * s->Hq * N * d;
  for (bh = 0; bh < n; ++bh)
    if (!in_range(bf16f(dout[bh]))) return ORC_ERR_RANGE;
  for (bh = 0; bh < (int64_t)s->B * s->Hq; ++bh)
    sagebwd_prepare_head(dout + bh * N * d, o + bh * N * d, (int)N, (int)d, bq, doc + bh * N * d, dos + bh * Tm,
                         D + bh * N);
  return ORC_OK;
}

int orc_sagebwd_backward(const orc_shape *s, int flags, int bq, int bk, int causal, double sm_scale,
                         const uint16_t *q, const uint16_t *k, const orc_quant *qz, const uint16_t *v,
                         const double *o, const uint16_t *dout, const double *lse, double *dq,
                         double *dk, double *dv) {
  const int B = s->B, Hq = s->Hq, Hkv = s->Hkv, N = s->N, M = s->M, d = s->d;
  const int64_t Tm = cdiv(N, bq), Tn = cdiv(M, bk);
  const int exact = (flags & ORC_EXACT_BWD) != 0;
  int8_t *doc = NULL;   /* dO codes of one head [N][d] */
  float *dos = NULL;    /* dO block scales of one head [Tm] */
  double *Dr = NULL;    /* D_r = rowsum(dO o O) of one head [N] */
  double *P = NULL, *dS = NULL, *Qd = NULL, *Kd = NULL;
  int64_t n;
  int b, h, rc = check_shape(s, ORC_SAGEBWD_I8, bq, bk);
  if (rc) return rc;
  if (causal && N > M) return ORC_ERR_ARG;

  doc = (int8_t *)malloc((size_t)N * d);
  dos = (float *)malloc(sizeof(float) * (size_t)Tm);
  Dr = (double *)malloc(sizeof(double) * (size_t)N);
  P = (double *)malloc(sizeof(double) * (size_t)bq * bk);
  dS = (double *)malloc(sizeof(double) * (size_t)bq * bk);
  Qd = (double *)malloc(sizeof(double) * (size_t)bq * d); /* deq(Q^_i) rows */
  Kd = (double *)malloc(sizeof(double) * (size_t)bk * d); /* deq(K^_j) rows */
  if (!doc || !dos || !Dr || !P || !dS || !Qd || !Kd) {
    rc = ORC_ERR_ARG;
    goto done;
  }
  n = (int64_t)B * Hq * N * d;
  for (int64_t i = 0; i < n; ++i)
    if (!in_range(bf16f(dout[i]))) {
      rc = ORC_ERR_RANGE;
      goto done;
    }
  memset(dq, 0, sizeof(double) * (size_t)n);
  n = (int64_t)B * Hkv * M * d;
  memset(dk, 0, sizeof(double) * (size_t)n);
  memset(dv, 0, sizeof(double) * (size_t)n);

  for (b = 0; b < B; ++b)
    for (h = 0; h < Hq; ++h) {
      const int64_t bh = (int64_t)b * Hq + h;
      const int64_t hk = (int64_t)b * Hkv + h / (Hq / Hkv);
      const uint16_t *dO = dout + bh * N * d;
      const float *kbar = qz->kbar + hk * d;
      int64_t i, j;
      int r, c, e;

      /* dO^ per block and D_r = rowsum(dO o O) */
      sagebwd_prepare_head(dO, o + bh * N * d, N, d, bq, doc, dos, Dr);

      for (j = 0; j < Tn; ++j) {
        const int t0 = (int)(j * bk), nk = (int)((j + 1) * bk < M ? bk : M - j * bk);
        for (c = 0; c < nk; ++c) deq_k_row(s, ORC_SAGEBWD_I8, flags, bk, k, qz, hk, t0 + c, Kd + (int64_t)c * d);

        for (i = 0; i < Tm; ++i) {
          const int r0 = (int)(i * bq), nq = (int)((i + 1) * bq < N ? bq : N - i * bq);
          const float *qbar = qz->qbar + (bh * Tm + i) * d;
          double pmax = 0.0, smax = 0.0, sP, sdS;

          for (r = 0; r < nq; ++r) deq_q_row(s, ORC_SAGEBWD_I8, flags, bq, q, qz, bh, r0 + r, Qd + (int64_t)r * d);

          /* S_ij recomputed as in the forward, P_ij = exp(S - lse) */
          for (r = 0; r < nq; ++r)
            for (c = 0; c < bk; ++c) {
              double pv = 0.0;
              if (c < nk && visible(causal, r0 + r, t0 + c, N, M)) {
                double s0 = 0.0, ds = 0.0;
                for (e = 0; e < d; ++e) s0 += Qd[(int64_t)r * d + e] * Kd[(int64_t)c * d + e];
                if (flags & ORC_SMOOTH_Q)
                  for (e = 0; e < d; ++e) ds += (double)qbar[e] * Kd[(int64_t)c * d + e];
                pv = exp((s0 + ds) * sm_scale - lse[bh * N + r0 + r]);
              }
              P[r * bk + c] = pv;
              if (pv > pmax) pmax = pv;
            }

          /* dV_j += P^T dO, P^ per tile, dO^ per block */
          sP = pmax / 127.0;
          for (c = 0; c < nk; ++c)
            for (r = 0; r < nq; ++r) {
              const double pq = exact ? P[r * bk + c] : int8_code64(P[r * bk + c], sP) * sP;
              if (pq == 0.0) continue;
              for (e = 0; e < d; ++e) {
                const double g = exact ? orc_bf16_decode(dO[(int64_t)(r0 + r) * d + e])
                                       : (double)doc[(int64_t)(r0 + r) * d + e] * (double)dos[i];
                dv[(hk * M + t0 + c) * d + e] += pq * g;
              }
            }

          /* dP = dO V^T unquantized (ORC_BWD_INT8_DP, the ablation the pages
           * measure against it: INT8 dO^ times the forward's INT8 V^, plus V_m);
           * dS = P o (dP - D) */
          for (r = 0; r < nq; ++r)
            for (c = 0; c < bk; ++c) {
              double dp = 0.0, x;
              if (P[r * bk + c] == 0.0) {
                dS[r * bk + c] = 0.0;
                continue;
              }
              if (flags & ORC_BWD_INT8_DP) {
                for (e = 0; e < d; ++e)
                  dp += (double)doc[(int64_t)(r0 + r) * d + e] * (double)dos[i] *
                        ((double)(int8_t)qz->vc[(hk * M + t0 + c) * d + e] * (double)qz->dvb[hk * Tn + j] +
                         (double)qz->vm[hk * d + e]);
              } else {
                for (e = 0; e < d; ++e)
                  dp += orc_bf16_decode(dO[(int64_t)(r0 + r) * d + e]) *
                        orc_bf16_decode(v[(hk * M + t0 + c) * d + e]);
              }
              x = P[r * bk + c] * (dp - Dr[r0 + r]);
              dS[r * bk + c] = x;
              if (fabs(x) > smax) smax = fabs(x);
            }

          /* dQ_i += (dS^ K^) s_dS + rowsum(dS) k_bar^T and
           * dK_j += (dS^T Q^) s_dS + colsum(dS) q_bar_i^T: the INT8 products
           * take the smoothed operands, the smoothing corrections the
           * unquantized dS (in higher precision); k_bar and q_bar are 0 when K
           * or Q was not smoothed */
          sdS = smax / 127.0;
          for (r = 0; r < nq; ++r)
            for (c = 0; c < nk; ++c) {
              const double gx = dS[r * bk + c];
              const double g = exact ? gx : int8_code64(gx, sdS) * sdS;
              if (gx == 0.0) continue;
              for (e = 0; e < d; ++e) {
                dq[(bh * N + r0 + r) * d + e] += g * Kd[(int64_t)c * d + e] + gx * (double)kbar[e];
                dk[(hk * M + t0 + c) * d + e] += g * Qd[(int64_t)r * d + e] + gx * (double)qbar[e];
              }
            }
        }
      }
    }

  /* the scores were S * sm_scale: dQ and dK carry that factor */
  n = (int64_t)B * Hq * N * d;
  for (int64_t i = 0; i < n; ++i) dq[i] *= sm_scale;
  n = (int64_t)B * Hkv * M * d;
  for (int64_t i = 0; i < n; ++i) dk[i] *= sm_scale;

done:
  free(doc);
  free(dos);
  free(Dr);
  free(P);
  free(dS);
  free(Qd);
  free(Kd);
  return rc;
}
