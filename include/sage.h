/*
 * sage.h — C ABI of the GB300 (sm_103a) quantized attention forward.
 *
 * The operation (SageAttention2 Technical Report summary, arXiv 2411.10958,
 * §3.2 "Big-Picture Architecture" and §3.4 "The Complete Algorithm";
 * SageAttention3 summary, arXiv 2505.11594, §3.4 "FP4 Attention Kernel
 * Algorithm"):
 *
 *   O = softmax(Q K^T * sm_scale) V
 *
 * computed tile by tile without materialising the N x M score matrix, with
 *   - K smoothing: K <- K - mean over tokens of K (exact under softmax);
 *   - optional Q smoothing: gamma(Q_i) = Q_i - mean(Q_i) per query block, and
 *     dS_ij = q_bar_i deq(K^_j)^T added back to the scores;
 *   - optional V smoothing: V' = V - V_m, O = O' + V_m;
 *   - Q/K quantized per block (INT8, or FP8 E4M3) or NVFP4 (E2M1 in 1x16 blocks
 *     with E4M3 scales);
 *   - P~ quantized to FP8 E4M3 with the static scale 1/448 and V per channel to
 *     FP8 E4M3 (or both NVFP4 with the two-level P~ scaling);
 *   - two-level accumulation: each key tile's P^ V^ partial is computed alone
 *     and added into an FP32 running output with the online-softmax rescale.
 *
 * Conventions
 *   - All tensors are device memory owned by the caller.  The library never
 *     allocates, frees or synchronises (except sage_read_status, which copies
 *     four words back and waits for that copy).
 *   - Inputs q [B,Hq,N,d], k and v [B,Hkv,M,d], output o [B,Hq,N,d]: bf16,
 *     contiguous, 16-byte aligned.  Query head h reads kv head h / (Hq/Hkv).
 *   - sage_quantize_qkv writes the workspace; sage_attn_fwd reads it.  Both
 *     launch on the caller's stream and return at once.
 *   - Argument errors are reported synchronously, before anything is
 *     launched.  Conditions found on the device (an input out of range, a
 *     bounded wait that gave up) are written to a status word inside the
 *     workspace; read it with sage_read_status after the stream has run.
 *     Nothing traps, aborts or throws across this boundary.
 */
#ifndef SAGE_H
#define SAGE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *sage_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  SAGE_OK = 0,
  SAGE_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad shape, bad flags */
  SAGE_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement */
  SAGE_ERR_WORKSPACE = 3,   /* workspace smaller than sage_workspace_bytes() */
  SAGE_ERR_RANGE = 4,       /* (device) an input was non-finite or |x| >= 2^16 */
  SAGE_ERR_TIMEOUT = 5,     /* (device) a bounded wait gave up; outputs undefined */
  SAGE_ERR_CUDA = 6         /* a CUDA runtime call failed (launch, copy) */
} sage_status;

/* quant_mode */
enum {
  SAGE_Q8_PV8 = 0,  /* INT8 per-block Q/K, FP8 E4M3 P~ (1/448) and per-channel FP8 V */
  SAGE_QF8_PV8 = 1, /* FP8 E4M3 per-block Q/K, FP8 P~ / V as above */
  SAGE_NVFP4 = 2,   /* NVFP4 Q/K/V (E2M1, 1x16 blocks, E4M3 scales), two-level P~ */
  /* SageBwd forward (SageAttention3 summary, "SageBwd Forward Pass"): INT8
   * per-block Q and K as in mode 0, INT8 per-block V (one scale per bk-token
   * block), INT8 P~ with one scale per row and key tile,
   * s_P = exp(rowmax S_ij - m_ij) / 127; bk = 64.  The attention also writes
   * each row's log-sum-exp (region lse), which a backward pass needs */
  SAGE_SAGEBWD_I8 = 3
};

/* flags */
enum {
  SAGE_SMOOTH_K = 1, /* subtract mean(K) over tokens (always exact) */
  SAGE_SMOOTH_Q = 2, /* subtract the per-block mean of Q, add dS back */
  SAGE_SMOOTH_V = 4, /* subtract mean(V) over tokens, add it back to O */
  /* ablation of the NVFP4 mode (SageAttention3 summary §3.4, "Two-Level
   * Quantization for P"): phi applied to P~ itself, no level-1 scale; accepted
   * and without effect in modes 0 and 1, whose P~ quantization is direct */
  SAGE_P_DIRECT = 8,
  /* one Q scale per query row instead of one per 128-row block (modes 0, 1);
   * q_bar stays per block.  Per-thread / per-token granularity is what the
   * SageAttention summaries trade against the MMA layout; on tcgen05 each
   * softmax thread owns a whole row of S, so it costs the kernel one load */
  SAGE_Q_PER_TOKEN = 0x10
};

typedef struct {
  int B, Hq, Hkv, N, M, d;
} sage_shape;

/* Byte offsets of the workspace regions (each 1024-byte aligned), for tests
 * and tools that read the quantized tensors.  Element layouts:
 *   qhat   [B*Hq*N_pad, d] codes: fp16 value of the INT8 code (mode 0: GB300's
 *          tensor cores have no INT8 path, so INT8 codes are carried as exact
 *          fp16 integers), E4M3 bytes (mode 1), packed E2M1 pairs (mode 2)
 *   dq     [B*Hq*Tm]      fp32 per-block Q scale (modes 0, 1)
 *   qbar   [B*Hq*Tm, d]   fp32 per-block Q mean (0 unless SAGE_SMOOTH_Q)
 *   khat   [B*Hkv*M_pad, d] codes as qhat
 *   dk     [B*Hkv*Tn]     fp32 per-block K scale (modes 0, 1)
 *   kbar   [B*Hkv, d]     fp32 K mean (0 unless SAGE_SMOOTH_K)
 *   vhat   [B*Hkv*d, M_pad] V codes transposed (token-contiguous): E4M3 bytes,
 *          or packed E2M1 pairs (mode 2)
 *   dv     [B*Hkv, d]     fp32 per-channel V scale (modes 0, 1)
 *   vm     [B*Hkv, d]     fp32 V mean (0 unless SAGE_SMOOTH_V)
 *   qsf, ksf, vsf         E4M3 block scales (mode 2), layouts in the .cu file
 *   stats                 reduction scratch of sage_quantize_qkv
 *   status                int32[4]: code, site, detail, spare
 *   dqt    [B*Hq*N_pad]   fp32 per-row Q scale (SAGE_Q_PER_TOKEN; 0 on pad rows)
 *   dvb    [B*Hkv*Tn]     fp32 per-block V scale (mode 3, whose vhat holds the
 *          INT8 codes as fp16 values)
 *   lse    [B*Hq*N_pad]   fp32 log-sum-exp of each row's scaled scores,
 *          ln sum_j exp(S_ij sm_scale) (mode 3; rows past N not written)
 *   doc    [B*Hq*N_pad, d] dO codes, INT8 per 128-row block held as fp16 values
 *   dos    [B*Hq*Tm]      their scales
 *   drow   [B*Hq*N_pad]   D = rowsum(dO o O), fp32
 *          (the SageBwd backward's inputs, written by sage_bwd_prepare; mode 3)
 * N_pad = N rounded up to 128, M_pad = M rounded up to 128, Tm = N_pad/bq,
 * Tn = ceil(M/bk). */
typedef struct {
  size_t qhat, dq, qbar, khat, dk, kbar, vhat, dv, vm, qsf, ksf, vsf, stats, status, total;
  int N_pad, M_pad, Tm, Tn;
  size_t dqt, dvb, lse, doc, dos, drow;
} sage_ws_layout;

/* Workspace size in bytes for a shape and mode; 0 if the request is invalid
 * or unsupported (see sage_workspace_layout for the reason). */
size_t sage_workspace_bytes(const sage_shape *shape, int quant_mode, int bq, int bk);

/* Fill *out with the workspace regions for this request. */
sage_status sage_workspace_layout(const sage_shape *shape, int quant_mode, int bq, int bk,
                                  sage_ws_layout *out);

/* Smoothing and quantization pre-pass (SageAttention2 summary §3.2 item 1 and
 * §3.4 "Smoothing Q"; SageAttention3 summary §3.4, quantizer phi).
 * Reads q, k, v (bf16, see Conventions), writes the quantized tensors, scales
 * and means into the workspace.  Supported: d in {64, 128}, bq == 128,
 * bk in {64, 128}, Hq % Hkv == 0, 1 <= N, M <= 2^23.  Every quantizer is a
 * fixed binary32 function of the inputs (round to nearest even), so codes and
 * scales are reproducible bit for bit. */
sage_status sage_quantize_qkv(const sage_shape *shape, int quant_mode, int flags, int bq, int bk,
                              const void *q, const void *k, const void *v, void *workspace,
                              size_t workspace_bytes, sage_stream_t stream);

/* The pre-pass of sage_quantize_qkv with its reduction scratch held in a fixed
 * device array inside the library instead of the caller's workspace.  The
 * pages have no counterpart: this is for callers that may not obtain device
 * memory for scratch — a plug-in whose host framework owns every device
 * allocation, or a latency-critical caller that must not call cudaMalloc
 * because it can synchronise the device.  The caller still provides q, k, v
 * and the output workspace (same size and layout as for sage_quantize_qkv, so
 * sage_attn_fwd reads it unchanged; its stats region is left untouched).
 * Limit: B * Hkv * d <= 32768 (a 768 KiB array, held on every GPU that loads
 * the library until the process exits); larger requests return
 * SAGE_ERR_UNSUPPORTED.  Every quant_mode and flag of sage_quantize_qkv is
 * accepted.  The first call on a device looks up the array's device address
 * with that device current and keeps it for the life of the process; make that
 * first call before any stream capture, and do not call this entry point again
 * after a cudaDeviceReset of that device (the kept address would be stale).
 * The call allocates and frees nothing.  Every call shares
 * the array and clears it before use; calls that overlap on the GPU race on
 * it and must be serialised by the caller. */
sage_status sage_quantize_qkv_static_scratch(const sage_shape *shape, int quant_mode, int flags, int bq,
                                             int bk, const void *q, const void *k, const void *v,
                                             void *workspace, size_t workspace_bytes,
                                             sage_stream_t stream);

/* Fused attention over the quantized workspace (SageAttention2 summary §3.4
 * "The Complete Algorithm", SageAttention3 summary §3.4 "FP4 Attention Kernel
 * Algorithm").  causal != 0 masks key j for query i when j > i + (M - N)
 * (bottom-right aligned; requires M >= N).  quant_mode, flags, bq and bk must
 * be those given to sage_quantize_qkv for this workspace.  Writes o (bf16).
 * SAGE_ERR_UNSUPPORTED for a causal INT8 / FP8 request of 2^24 or more query
 * blocks (B * Hq * ceil(N / 128)), whose work order the kernel cannot form. */
sage_status sage_attn_fwd(const sage_shape *shape, int causal, float sm_scale, int quant_mode,
                          int flags, int bq, int bk, const void *workspace, size_t workspace_bytes,
                          void *o, sage_stream_t stream);

/* End-to-end call on HOST buffers (ideally pinned): q, k, v copied in, the
 * pre-pass and the attention run, o copied back, asynchronously on `stream`.
 * The request is cut into chunks of whole kv heads of one batch element
 * (independent problems: their own means and scales, so the result is the
 * same as one call on the whole request) and the copies of one chunk overlap
 * the kernels of the others: host -> device on one internal stream, the
 * kernels of even chunks on `stream` and of odd chunks on a second internal
 * stream, device -> host on a third.  The internal streams and their events
 * are created once per device on the first call (no device memory); the call
 * is ordered after earlier work on `stream` and later work on `stream` after
 * its last copy.  Calls on one dev_buf must not overlap.  dev_buf is one
 * caller-allocated, 1024-byte aligned device buffer of at least
 * sage_host_buffer_bytes(); its first 16 bytes hold the call's device status
 * word int[4] (code, site: the first error of any chunk) once `stream` has
 * completed. */
size_t sage_host_buffer_bytes(const sage_shape *shape, int quant_mode, int bq, int bk);
sage_status sage_attn_host(const sage_shape *shape, int causal, float sm_scale, int quant_mode,
                           int flags, int bq, int bk, const void *q_host, const void *k_host,
                           const void *v_host, void *o_host, void *dev_buf, size_t dev_bytes,
                           sage_stream_t stream);

/* Packed sequences (the SageAttention production guide, "Handling Varying
 * Sequence Lengths with VarLen Kernels": sageattn_varlen).  q is bf16
 * [total_q, Hq, d], k and v bf16 [total_k, Hkv, d], o bf16 [total_q, Hq, d],
 * all contiguous; sequence s holds query rows cu_seqlens_q[s] ..
 * cu_seqlens_q[s+1] - 1 and key rows cu_seqlens_k[s] .. cu_seqlens_k[s+1] - 1.
 * cu_seqlens_q and cu_seqlens_k are HOST int32 arrays of nseq + 1 entries,
 * starting at 0 and non-decreasing; a sequence with queries needs keys, and a
 * causal mask (bottom-right aligned within each sequence) needs at least as many
 * keys as queries.  Each sequence is its own attention problem: its own means,
 * scales and query / key blocks, starting at its first token.  Every mode
 * (NVFP4 with 128-key tiles).
 * The workspace holds the batched layout of B = nseq, N = the longest query
 * run, M = the longest key run (so sage_workspace_layout of that shape
 * locates the codes), then the sequence and work-item tables; compute and
 * traffic follow the sequences' own lengths.  sage_attn_varlen runs the
 * pre-pass and the attention on `stream`; its tables reach the device by one
 * copy from pageable host memory, so the call returns only after the runtime
 * has staged them (not capturable into a CUDA graph).
 * sage_varlen_workspace_bytes returns 0 for an invalid or unsupported request. */
size_t sage_varlen_workspace_bytes(int nseq, const int *cu_seqlens_q, const int *cu_seqlens_k, int Hq, int Hkv,
                                   int d, int quant_mode, int bq, int bk);
sage_status sage_attn_varlen(int nseq, const int *cu_seqlens_q, const int *cu_seqlens_k, int Hq, int Hkv, int d,
                             int causal, float sm_scale, int quant_mode, int flags, int bq, int bk, const void *q,
                             const void *k, const void *v, void *workspace, size_t workspace_bytes, void *o,
                             sage_stream_t stream);

/* The SageBwd backward's pre-pass (SageAttention3 summary, "SageBwd Backward
 * Pass": dV takes P^T dO^ with dO INT8 per block, dS takes D = rowsum(dO o O)):
 * reads o (the forward's bf16 output) and dout (the output gradient, bf16),
 * both [B, Hq, N, d] contiguous, and writes doc / dos / drow of a mode-3
 * workspace.  dO is quantized like Q (scale fl(max|dO_i|/127) per 128-row
 * block, code rint(fl(x/scale))); D is summed in fp32.  A non-finite or
 * |x| >= 2^16 gradient sets SAGE_ERR_RANGE in the status word. */
sage_status sage_bwd_prepare(const sage_shape *shape, int quant_mode, int bq, int bk, const void *o,
                             const void *dout, void *workspace, size_t workspace_bytes, sage_stream_t stream);

/* SageBwd backward (SageAttention3 summary, "SageBwd Backward Pass and the
 * Critical dOV^T Decision", eq. 8 and Algorithm 3): dQ, dK, dV of the
 * forward that sage_attn_fwd ran on this workspace in quant_mode
 * SAGE_SAGEBWD_I8 (bk = 64), after sage_bwd_prepare wrote the dO codes and D.
 * S and P = exp(S sm_scale - lse) are recomputed from the forward's INT8 Q and K
 * codes and its log-sum-exp; P and dS go to INT8 per 128 x 64 tile (scale
 * max / 127), dO to INT8 per 128-row block; dV = P^T dO, dK = dS^T Q and
 * dQ = dS K run on those codes; dP = dO V^T stays 16-bit (bf16 operands); the
 * K and Q smoothing corrections rowsum(dS) k_bar and colsum(dS) q_bar take the
 * unquantized dS.  causal, sm_scale and flags must be the forward's
 * (SAGE_Q_PER_TOKEN is not supported: SAGE_ERR_UNSUPPORTED).
 * v: the forward's bf16 V [B,Hkv,M,d]; dout: bf16 dO [B,Hq,N,d] (the one given
 * to sage_bwd_prepare); outputs fp32, caller-allocated, 16-byte aligned:
 * dq [B,Hq,N,d], dk and dv [B,Hkv,M,d] (summed over the query heads of a kv
 * head).  Deterministic: no atomics.  A bounded wait that gives up sets
 * SAGE_ERR_TIMEOUT in the status word; the outputs are then undefined. */
sage_status sage_attn_bwd(const sage_shape *shape, int causal, float sm_scale, int quant_mode, int flags, int bq,
                          int bk, const void *workspace, size_t workspace_bytes, const void *v, const void *dout,
                          void *dq, void *dk, void *dv, sage_stream_t stream);

/* Copy the device status word back (blocking on that copy only): *code is a
 * sage_status (SAGE_OK, SAGE_ERR_RANGE or SAGE_ERR_TIMEOUT), *site says where
 * it was raised.  The status word is cleared by every sage_quantize_qkv. */
sage_status sage_read_status(const sage_shape *shape, int quant_mode, int bq, int bk, const void *workspace,
                             int *code, int *site);

const char *sage_status_str(sage_status s);

#ifdef __cplusplus
}
#endif
#endif
