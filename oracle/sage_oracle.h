/*
 * Oracle for SageAttention-style quantized attention forward — TEST
 * INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library or its
 * binding) includes, links or calls this code; only the tests, the smoke
 * check and the bench's CPU-baseline leg do.  It shares no code, header,
 * table or constant with the CUDA path.
 *
 * What it computes (plain, single-threaded, slow on purpose):
 *   - the quantizers, in IEEE binary32 with round-to-nearest-even, so that
 *     codes and scales are a precise function of the bf16 inputs;
 *   - the tiled online-softmax attention of the method, in binary64, in the
 *     pages' order: for each query block i and key tile j = 0..Tn-1,
 *     S = deq(Q^) deq(K^)^T [+ dS], online max / sum, P~ quantization,
 *     tile partial R = P^ V^, running O = alpha O + R, then O / l scaled;
 *   - the SageBwd forward of the same loop (INT8 per-block Q, K, V; INT8 P~
 *     with a per-row scale for each key tile) and, for every mode, each row's
 *     log-sum-exp m + ln(l), the statistic a backward pass recomputes P from;
 *   - plain fp64 softmax(Q K^T sm_scale) V on the bf16 inputs.
 *
 * Sources (web pages this method is described on):
 *   SageAttention2 Technical Report summary (arXiv 2411.10958), §3.2 and
 *   §3.4: smoothing Q / K, dS, FP8 P~ with static 1/448, per-channel FP8 V,
 *   two-level accumulation, V smoothing, "The Complete Algorithm".
 *   SageAttention3 summary (arXiv 2505.11594), §3.4: NVFP4 quantizer phi,
 *   two-level quantization for P, FP4 attention algorithm; "SageBwd Forward
 *   Pass": per-block INT8 Q, K, V and per-token INT8 P.
 *   "Quantization for Attention, in depth" (aicassindra): datapath and the
 *   INT8 per-block quantizer.
 *
 * Every function is pinned by tests under -m "not gpu" (format tables from
 * the pages, closed forms, brute force on tiny inputs, identities).  The one
 * part with no independent pin is which E4M3 / E2M1 code a P~ value gets when
 * the fp64 value here and the kernel's fp32 value fall on opposite sides of a
 * rounding midpoint ("parity unpinned" for those individual codes; the
 * attention outputs stay inside the stated tolerance).
 */
#ifndef SAGE_ORACLE_H
#define SAGE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* quant modes */
#define ORC_Q8_PV8 0   /* INT8 per-block Q/K, FP8 P~ and per-channel FP8 V */
#define ORC_QF8_PV8 1  /* FP8 E4M3 per-block Q/K, FP8 P~ / V */
#define ORC_NVFP4 2    /* E2M1 1x16 blocks, E4M3 scales, two-level P~ */
/* SageBwd forward (SageAttention3 summary, "SageBwd Forward Pass"): INT8
 * per-block Q and K as in mode 0, INT8 per-block V (one scale per bk-token
 * block over all d channels), INT8 P~ with one scale per row and key tile,
 * s_P = exp(rowmax S_ij - m_ij) / 127 */
#define ORC_SAGEBWD_I8 3

/* flags */
#define ORC_SMOOTH_K 1
#define ORC_SMOOTH_Q 2
#define ORC_SMOOTH_V 4
/* ablation of the NVFP4 mode (SageAttention3 summary §3.4, two-level P): phi
 * applied to P~ itself, no level-1 scale (s_P1 = 1); no effect in the FP8 modes,
 * whose P~ quantization is already direct */
#define ORC_P_DIRECT 8
/* one Q scale per query row (modes 0, 1) instead of one per bq-row block: the
 * per-token granularity the SageAttention summaries ablate (each row of S has
 * its own dequantization scale); q_bar stays per block */
#define ORC_Q_PER_TOKEN 0x10
/* oracle-only switches used by the pins: replace a quantizer by identity */
#define ORC_EXACT_QK 0x100 /* S from the unrounded smoothed Q, K in fp64 */
#define ORC_EXACT_PV 0x200 /* R from unquantized P~ and unquantized V' in fp64 */
#define ORC_EXACT_BWD 0x400 /* backward: P, dO and dS unquantized in fp64 */
/* backward ablation (SageAttention3 summary, "SageBwd Backward Pass and the
 * Critical dOV^T Decision"): dP = dO V^T from INT8 dO^ and the forward's
 * per-block INT8 V^ instead of the unquantized operands */
#define ORC_BWD_INT8_DP 0x800

/* error codes */
#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_RANGE 4 /* |x| >= 2^16 or non-finite input */

typedef struct {
  int B, Hq, Hkv, N, M, d;
} orc_shape;

/* Quantized tensors, logical layouts (no padding), all caller-allocated.
 *   qc  [B,Hq,N,d]   codes: int8 value (mode 0), E4M3 byte (1), E2M1 nibble (2)
 *   dq  [B,Hq,Tm]    per-block Q scale (modes 0, 1)
 *   qbar[B,Hq,Tm,d]  per-block Q mean (0 unless SMOOTH_Q)
 *   kc  [B,Hkv,M,d]  codes as for Q
 *   dk  [B,Hkv,Tn]   per-block K scale (modes 0, 1)
 *   kbar[B,Hkv,d]    K mean (0 unless SMOOTH_K)
 *   vc  [B,Hkv,M,d]  E4M3 (modes 0, 1) or E2M1 nibble (mode 2)
 *   dv  [B,Hkv,d]    per-channel V scale (modes 0, 1)
 *   vm  [B,Hkv,d]    V mean (0 unless SMOOTH_V)
 *   qs  [B,Hq,N,d/16]          E4M3 block scales (mode 2)
 *   ks  [B,Hkv,M,d/16]         E4M3 block scales (mode 2)
 *   vs  [B,Hkv,ceil(M/16),d]   E4M3 block scales along tokens (mode 2)
 *   dqt [B,Hq,N]     per-token Q scale (modes 0, 1 with ORC_Q_PER_TOKEN; dq unused then)
 *   dvb [B,Hkv,Tn]   per-block V scale (mode 3; V codes are int8 values then)
 * Tm = ceil(N/bq), Tn = ceil(M/bk).  Pointers a mode does not use may be NULL. */
typedef struct {
  uint8_t *qc;
  float *dq, *qbar;
  uint8_t *kc;
  float *dk, *kbar;
  uint8_t *vc;
  float *dv, *vm;
  uint8_t *qs, *ks, *vs;
  float *dqt;
  float *dvb;
} orc_quant;

/* ---- codecs (round to nearest, ties to even; saturate to the largest
 *      finite magnitude; sign bit taken from the input's sign bit) ---- */
uint8_t orc_e4m3_encode(double x);
double orc_e4m3_decode(uint8_t code);
uint8_t orc_e2m1_encode(double x); /* 4-bit code in the low nibble */
double orc_e2m1_decode(uint8_t code);
uint16_t orc_bf16_encode(double x); /* round to nearest even, no saturation */
double orc_bf16_decode(uint16_t bits);

/* array forms of the codecs (same definitions, one call for many values) */
void orc_e4m3_encode_array(const float *x, int64_t n, uint8_t *out);
void orc_e2m1_encode_array(const float *x, int64_t n, uint8_t *out);
void orc_bf16_encode_array(const double *x, int64_t n, uint16_t *out);

/* ---- quantizer building blocks (binary32, exact definitions) ---- */
/* mean over n bf16 values with stride: fixed-point sum with lsb 2^-24
 * (each value truncated toward zero at 2^-24), then one rounding to double
 * and one division; returns ORC_ERR_RANGE for |x| >= 2^16 or non-finite. */
int orc_mean_bf16(const uint16_t *x, int64_t n, int64_t stride, float *mean);
/* INT8 per-block: scale = fl(absmax/127), code = clamp(rint(fl(x/scale))) */
float orc_int8_scale(float absmax);
int orc_int8_code(float x, float scale);
/* E4M3 per-block / per-channel: scale = fl(absmax/448), code = e4m3(fl(x/scale)) */
float orc_fp8_scale(float absmax);
uint8_t orc_fp8_code(float x, float scale);
/* NVFP4 block: s = e4m3(fl(absmax/6)), code = e2m1(fl(x/dec(s))) (0 if dec(s)==0) */
uint8_t orc_nvfp4_scale(float absmax);
uint8_t orc_nvfp4_code(float x, uint8_t scale_code);

/* ---- the method ---- */
int orc_quantize(const orc_shape *s, int mode, int flags, int bq, int bk, const uint16_t *q,
                 const uint16_t *k, const uint16_t *v, orc_quant *out);

/* Output rows of the quantized attention in fp64.  rows[i] = (b*Hq + h)*N + r.
 * out is [nrows, d]. */
int orc_attn_rows(const orc_shape *s, int mode, int flags, int bq, int bk, int causal,
                  double sm_scale, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const orc_quant *qz, const int64_t *rows, int64_t nrows, double *out);

/* As orc_attn_rows, and lse[i] = m + ln(l) of row i at the end of the key
 * loop (the softmax statistics a backward pass recomputes P from; natural log,
 * in the units of the scaled scores S * sm_scale).  lse may be NULL. */
int orc_attn_rows_lse(const orc_shape *s, int mode, int flags, int bq, int bk, int causal,
                      double sm_scale, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const orc_quant *qz, const int64_t *rows, int64_t nrows, double *out,
                      double *lse);

/* SageBwd backward (SageAttention3 summary, "SageBwd Backward Pass and the
 * Critical dOV^T Decision", eq. 8 and Algorithm 3), key blocks j outer, query
 * blocks i inner:
 *   S_ij recomputed from the forward's Q^, K^ (and dS when Q was smoothed),
 *   P_ij = exp(S_ij sm_scale - lse_i);
 *   dV_j += (P^_ij^T dO^_i) s_P s_dO    P per bq x bk tile, dO per bq-row block,
 *                                        both INT8 per-block (max / 127);
 *   dP_ij = dO_i V_j^T                   unquantized (bf16 operands, fp64 here);
 *   dS_ij = P_ij o (dP_ij - D_i), D_i = rowsum(dO_i o O_i), INT8 per tile;
 *   dQ_i += (dS^_ij K^_j) s_dS s_K,j + rowsum(dS_ij) k_bar^T
 *   dK_j += (dS^_ij^T Q^_i) s_dS s_Q,i [+ colsum(dS_ij) q_bar_i^T when Q was
 *                                        smoothed] -- the smoothing corrections
 *                                        from the unquantized dS;
 *   dQ, dK times sm_scale at the end.
 * qz is the forward's quantization (mode ORC_SAGEBWD_I8 or ORC_Q8_PV8, whose Q
 * and K codes are the same); o [B,Hq,N,d] the forward output and lse [B,Hq,N]
 * its statistics; dout bf16 [B,Hq,N,d].  Outputs fp64: dq [B,Hq,N,d],
 * dk and dv [B,Hkv,M,d] (query heads of a kv head summed).  Flags: the
 * forward's smoothing flags, ORC_EXACT_QK (unquantized smoothed Q and K) and
 * ORC_EXACT_BWD. */
int orc_sagebwd_backward(const orc_shape *s, int flags, int bq, int bk, int causal, double sm_scale,
                         const uint16_t *q, const uint16_t *k, const orc_quant *qz, const uint16_t *v,
                         const double *o, const uint16_t *dout, const double *lse, double *dq,
                         double *dk, double *dv);

/* The SageBwd backward's inputs (its pre-pass): dO^ INT8 per bq-row block
 * (binary32: scale fl(max|dO_i|/127), code clamp(rint(fl(x/scale)))), as int8
 * [B,Hq,N,d] with scales [B,Hq,Tm], and D [B,Hq,N] = rowsum(dO o O) in fp64; o is
 * the forward output [B,Hq,N,d] in fp64.  orc_sagebwd_backward forms the same. */
int orc_sagebwd_prepare(const orc_shape *s, int bq, const double *o, const uint16_t *dout, int8_t *doc,
                        float *dos, double *D);

/* Plain softmax(Q K^T sm_scale) V in fp64 on the bf16 inputs, same masks. */
int orc_attn_exact_rows(const orc_shape *s, int causal, double sm_scale, const uint16_t *q,
                        const uint16_t *k, const uint16_t *v, const int64_t *rows, int64_t nrows,
                        double *out);

#ifdef __cplusplus
}
#endif
#endif
