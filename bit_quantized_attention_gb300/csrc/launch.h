// Kernel launchers behind the C ABI (host declarations).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sage.h"
#include "layout.h"

namespace sage {

// Packed-sequence tables in device memory (null for a batched request): the
// work item codes, their count, and the per-sequence lengths / first rows.
struct VarDev {
  const int *item_tab = nullptr;
  int items = 0;
  const VarSeq *seq = nullptr;
};

// Pre-pass for SAGE_Q8_PV8 / SAGE_QF8_PV8 (quantize.cu).
sage_status launch_quantize_q8(const sage_shape &s, int mode, int flags, int bq, int bk, const void *q,
                               const void *k, const void *v, void *ws, const sage_ws_layout &L,
                               cudaStream_t stream, const VarSeq *seq = nullptr);

// Same pre-pass with its statistics scratch in a device array inside the
// library (quantize.cu); B*Hkv*d must not exceed 32768.
sage_status launch_quantize_q8_static_scratch(const sage_shape &s, int mode, int flags, int bq, int bk,
                                              const void *q, const void *k, const void *v, void *ws,
                                              const sage_ws_layout &L, cudaStream_t stream);

// Attention for SAGE_Q8_PV8 / SAGE_QF8_PV8 (attn_q8.cu).
sage_status launch_attn_q8(const sage_shape &s, int causal, float sm_scale, int mode, int flags, int bk,
                           const void *ws, const sage_ws_layout &L, void *o, cudaStream_t stream,
                           const VarDev &var = VarDev());

// The tiles-in-turn schedule (attn_q8_ping.cu) and packed sequences
// (attn_q8_var.cu) of the same attention, called by launch_attn_q8.
sage_status launch_attn_q8_ping(const sage_shape &s, int causal, float sm_scale, int mode, int flags, int bk,
                                const void *ws, const sage_ws_layout &L, void *o, cudaStream_t stream);
sage_status launch_attn_q8_var(const sage_shape &s, int causal, float sm_scale, int mode, int flags, int bk,
                               const void *ws, const sage_ws_layout &L, void *o, cudaStream_t stream,
                               const VarDev &var);

// The SageBwd backward's pre-pass (quantize.cu): dO codes and scales, D.
sage_status launch_bwd_prepare(const sage_shape &s, const void *o, const void *dout, void *ws,
                               const sage_ws_layout &L, cudaStream_t stream);

// The two-query-block schedule of the INT8 / FP8 attention (attn_q8x2.cuh):
// batched requests, head dim 64, 64-key tiles, modes 0 and 1.
sage_status launch_attn_q8x2_64(const sage_shape &s, int causal, float sm_scale, int mode, int flags, const void *ws,
                                const sage_ws_layout &L, void *o, cudaStream_t stream);

// The SageBwd backward (attn_bwd.cu): dK and dV, then dQ, fp32 outputs.
sage_status launch_attn_bwd(const sage_shape &s, int causal, float sm_scale, int flags, const void *ws,
                            const sage_ws_layout &L, const void *v, const void *dout, float *dq, float *dk, float *dv,
                            cudaStream_t stream);

// Attention for SAGE_NVFP4 (attn_fp4.cu); bk must be 128.
sage_status launch_attn_fp4(const sage_shape &s, int causal, float sm_scale, int flags, int bk, const void *ws,
                            const sage_ws_layout &L, void *o, cudaStream_t stream, const VarDev &var = VarDev());

// The end-to-end call on host buffers, chunked and pipelined (host.cu): the
// device buffer it needs, and the call itself (arguments already checked).
sage_status host_buffer_bytes(const sage_shape &s, int mode, int bq, int bk, size_t *bytes);
sage_status run_attn_host(const sage_shape &s, int causal, float sm_scale, int mode, int flags, int bq, int bk,
                          const void *q_host, const void *k_host, const void *v_host, void *o_host, void *dev_buf,
                          cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point (api.cu).
// A 2-D byte tensor [rows][cols] with row pitch `pitch` bytes, box {box_cols, box_rows}.
sage_status make_tmap_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t pitch,
                         uint32_t box_cols, uint32_t box_rows, int swizzle_bytes);

// Spin limit (clock cycles) for bounded waits inside kernels.
long long spin_limit_cycles();

// Test hook, read at every attention launch: SAGE_TEST_STALL=1 makes the QK
// issuer of every CTA first wait on a barrier that nothing arrives on, so the
// bounded wait runs out (SAGE_ERR_TIMEOUT, site 29) and the kernel takes its
// unwind path.  Off (0) unless the variable is set.
int test_stall();

}  // namespace sage
