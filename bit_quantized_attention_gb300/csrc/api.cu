// C ABI entry points (declared in include/sage.h): argument checks, workspace
// layout, TMA descriptors and dispatch to the kernel launchers.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "layout.h"
#include "launch.h"

using namespace sage;

namespace sage {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

sage_status make_tmap_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t pitch,
                         uint32_t box_cols, uint32_t box_rows, int swizzle_bytes) {
  auto fn = encode_fn();
  if (!fn) return SAGE_ERR_CUDA;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SAGE_OK : SAGE_ERR_CUDA;
}

long long spin_limit_cycles() {
  // about two seconds at GB300 clocks unless SAGE_SPIN_LIMIT (cycles) says otherwise
  static long long v = [] {
    const char *e = getenv("SAGE_SPIN_LIMIT");
    long long x = e ? atoll(e) : 0;
    return x > 0 ? x : 4000000000LL;
  }();
  return v;
}

int test_stall() {
  const char *e = getenv("SAGE_TEST_STALL");
  return (e && e[0] == '1') ? 1 : 0;
}

}  // namespace sage

static bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

extern "C" {

// The workspace layout, and the limits of the launches built on it: every
// grid and work-item count the kernels hold in an int, and every row
// coordinate of the Q^ / K^ / V^T tensor maps (32-bit in a TMA copy), stays
// below 2^31.
static sage_status request_layout(const sage_shape *shape, int quant_mode, int bq, int bk, sage_ws_layout *L) {
  sage_status st = compute_layout(shape, quant_mode, bq, bk, L);
  if (st != SAGE_OK) return st;
  const int64_t lim = (int64_t)1 << 31;
  const int64_t bhq = (int64_t)shape->B * shape->Hq, bhk = (int64_t)shape->B * shape->Hkv;
  const int64_t items = bhq * L->Tm + bhk * ((int64_t)L->Tn + L->M_pad / 128);
  if (items >= lim || bhq * L->N_pad >= lim || bhk * L->M_pad >= lim || bhk * shape->d >= lim)
    return SAGE_ERR_UNSUPPORTED;
  return SAGE_OK;
}

size_t sage_workspace_bytes(const sage_shape *shape, int quant_mode, int bq, int bk) {
  sage_ws_layout L;
  if (request_layout(shape, quant_mode, bq, bk, &L) != SAGE_OK) return 0;
  return L.total;
}

sage_status sage_workspace_layout(const sage_shape *shape, int quant_mode, int bq, int bk, sage_ws_layout *out) {
  if (!out) return SAGE_ERR_INVALID_ARG;
  return request_layout(shape, quant_mode, bq, bk, out);
}

// Flag bits: unknown bits are an invalid argument; per-token Q scales exist in
// the INT8 / FP8 modes only (NVFP4 scales Q per 1x16 block already).
static sage_status check_flags(int quant_mode, int flags) {
  if (flags & ~(SAGE_SMOOTH_K | SAGE_SMOOTH_Q | SAGE_SMOOTH_V | SAGE_P_DIRECT | SAGE_Q_PER_TOKEN))
    return SAGE_ERR_INVALID_ARG;
  if ((flags & SAGE_Q_PER_TOKEN) && quant_mode == SAGE_NVFP4) return SAGE_ERR_UNSUPPORTED;
  return SAGE_OK;
}

sage_status sage_quantize_qkv(const sage_shape *shape, int quant_mode, int flags, int bq, int bk, const void *q,
                              const void *k, const void *v, void *workspace, size_t workspace_bytes,
                              sage_stream_t stream) {
  sage_ws_layout L;
  sage_status st = request_layout(shape, quant_mode, bq, bk, &L);
  if (st != SAGE_OK) return st;
  if ((st = check_flags(quant_mode, flags)) != SAGE_OK) return st;
  if (!q || !k || !v || !workspace) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || ((uintptr_t)workspace & 1023)) return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return SAGE_ERR_WORKSPACE;
  return launch_quantize_q8(*shape, quant_mode, flags, bq, bk, q, k, v, workspace, L, (cudaStream_t)stream);
}

// The attention call's own conditions (beyond the layout's): flags, sm_scale,
// the causal alignment, and the NVFP4 kernel's 128-key tiles.
static sage_status check_attn_args(const sage_shape *shape, int causal, float sm_scale, int quant_mode, int flags,
                                   int bk) {
  sage_status st = check_flags(quant_mode, flags);
  if (st != SAGE_OK) return st;
  if (!(sm_scale > 0.0f) || sm_scale > 1e30f) return SAGE_ERR_INVALID_ARG;
  if (causal && shape->N > shape->M) return SAGE_ERR_UNSUPPORTED;
  if (quant_mode == SAGE_NVFP4 && bk != 128) return SAGE_ERR_UNSUPPORTED;
  return SAGE_OK;
}

sage_status sage_attn_fwd(const sage_shape *shape, int causal, float sm_scale, int quant_mode, int flags, int bq,
                          int bk, const void *workspace, size_t workspace_bytes, void *o, sage_stream_t stream) {
  sage_ws_layout L;
  sage_status st = request_layout(shape, quant_mode, bq, bk, &L);
  if (st != SAGE_OK) return st;
  if ((st = check_flags(quant_mode, flags)) != SAGE_OK) return st;
  if (!workspace || !o || !aligned16(o) || ((uintptr_t)workspace & 1023)) return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return SAGE_ERR_WORKSPACE;
  st = check_attn_args(shape, causal, sm_scale, quant_mode, flags, bk);
  if (st != SAGE_OK) return st;
  if (quant_mode == SAGE_NVFP4)
    return launch_attn_fp4(*shape, causal, sm_scale, flags, bk, workspace, L, o, (cudaStream_t)stream);
  return launch_attn_q8(*shape, causal, sm_scale, quant_mode, flags, bk, workspace, L, o, (cudaStream_t)stream);
}

sage_status sage_quantize_qkv_static_scratch(const sage_shape *shape, int quant_mode, int flags, int bq, int bk,
                                             const void *q, const void *k, const void *v, void *workspace,
                                             size_t workspace_bytes, sage_stream_t stream) {
  sage_ws_layout L;
  sage_status st = request_layout(shape, quant_mode, bq, bk, &L);
  if (st != SAGE_OK) return st;
  if ((st = check_flags(quant_mode, flags)) != SAGE_OK) return st;
  if (!q || !k || !v || !workspace) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || ((uintptr_t)workspace & 1023)) return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return SAGE_ERR_WORKSPACE;
  if ((long long)shape->B * shape->Hkv * shape->d > 32768) return SAGE_ERR_UNSUPPORTED;
  return launch_quantize_q8_static_scratch(*shape, quant_mode, flags, bq, bk, q, k, v, workspace, L,
                                           (cudaStream_t)stream);
}

size_t sage_host_buffer_bytes(const sage_shape *shape, int quant_mode, int bq, int bk) {
  sage_ws_layout L;
  if (request_layout(shape, quant_mode, bq, bk, &L) != SAGE_OK) return 0;
  size_t bytes = 0;
  if (host_buffer_bytes(*shape, quant_mode, bq, bk, &bytes) != SAGE_OK) return 0;
  return bytes;
}

sage_status sage_attn_host(const sage_shape *shape, int causal, float sm_scale, int quant_mode, int flags, int bq,
                           int bk, const void *q_host, const void *k_host, const void *v_host, void *o_host,
                           void *dev_buf, size_t dev_bytes, sage_stream_t stream) {
  sage_ws_layout L;
  sage_status st = request_layout(shape, quant_mode, bq, bk, &L);
  if (st != SAGE_OK) return st;
  // every argument condition of the calls it makes, before the first copy
  st = check_attn_args(shape, causal, sm_scale, quant_mode, flags, bk);
  if (st != SAGE_OK) return st;
  if (!q_host || !k_host || !v_host || !o_host || !dev_buf) return SAGE_ERR_INVALID_ARG;
  if (((uintptr_t)dev_buf & 1023)) return SAGE_ERR_INVALID_ARG;
  size_t need = 0;
  if ((st = host_buffer_bytes(*shape, quant_mode, bq, bk, &need)) != SAGE_OK) return st;
  if (dev_bytes < need) return SAGE_ERR_WORKSPACE;
  return run_attn_host(*shape, causal, sm_scale, quant_mode, flags, bq, bk, q_host, k_host, v_host, o_host, dev_buf,
                       (cudaStream_t)stream);
}

size_t sage_varlen_workspace_bytes(int nseq, const int *cu_seqlens_q, const int *cu_seqlens_k, int Hq, int Hkv,
                                   int d, int quant_mode, int bq, int bk) {
  VarlenPlan P;
  if (plan_varlen(nseq, cu_seqlens_q, cu_seqlens_k, Hq, Hkv, d, quant_mode, bq, bk, 0, &P) != SAGE_OK) return 0;
  sage_ws_layout L;
  if (request_layout(&P.shape, quant_mode, bq, bk, &L) != SAGE_OK) return 0;
  return P.total;
}

sage_status sage_attn_varlen(int nseq, const int *cu_seqlens_q, const int *cu_seqlens_k, int Hq, int Hkv, int d,
                             int causal, float sm_scale, int quant_mode, int flags, int bq, int bk, const void *q,
                             const void *k, const void *v, void *workspace, size_t workspace_bytes, void *o,
                             sage_stream_t stream) {
  VarlenPlan P;
  sage_status st = plan_varlen(nseq, cu_seqlens_q, cu_seqlens_k, Hq, Hkv, d, quant_mode, bq, bk, causal, &P);
  if (st != SAGE_OK) return st;
  sage_ws_layout L;
  if ((st = request_layout(&P.shape, quant_mode, bq, bk, &L)) != SAGE_OK) return st;  // the int-range checks
  if ((st = check_attn_args(&P.shape, causal, sm_scale, quant_mode, flags, bk)) != SAGE_OK) return st;
  if (!q || !k || !v || !o || !workspace) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || ((uintptr_t)workspace & 1023))
    return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < P.total) return SAGE_ERR_WORKSPACE;
  // the sequence and work item tables, one host-to-device copy (from pageable
  // memory: the call returns once the source has been staged)
  char *ws = (char *)workspace;
  std::vector<char> tabs(P.total - P.seq_off, 0);
  memcpy(tabs.data(), P.seqs.data(), sizeof(VarSeq) * P.seqs.size());
  memcpy(tabs.data() + (P.item_off - P.seq_off), P.item_codes.data(), sizeof(int) * P.item_codes.size());
  cudaStream_t cs = (cudaStream_t)stream;
  if (cudaMemcpyAsync(ws + P.seq_off, tabs.data(), tabs.size(), cudaMemcpyHostToDevice, cs) != cudaSuccess)
    return SAGE_ERR_CUDA;
  const VarSeq *seq = (const VarSeq *)(ws + P.seq_off);
  st = launch_quantize_q8(P.shape, quant_mode, flags, bq, bk, q, k, v, workspace, P.L, cs, seq);
  if (st != SAGE_OK) return st;
  VarDev var;
  var.item_tab = (const int *)(ws + P.item_off);
  var.items = P.items;
  var.seq = seq;
  if (quant_mode == SAGE_NVFP4)
    return launch_attn_fp4(P.shape, causal, sm_scale, flags, bk, workspace, P.L, o, cs, var);
  return launch_attn_q8(P.shape, causal, sm_scale, quant_mode, flags, bk, workspace, P.L, o, cs, var);
}

sage_status sage_bwd_prepare(const sage_shape *shape, int quant_mode, int bq, int bk, const void *o,
                             const void *dout, void *workspace, size_t workspace_bytes, sage_stream_t stream) {
  sage_ws_layout L;
  sage_status st = request_layout(shape, quant_mode, bq, bk, &L);
  if (st != SAGE_OK) return st;
  if (quant_mode != SAGE_SAGEBWD_I8) return SAGE_ERR_UNSUPPORTED;
  if (!o || !dout || !workspace) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dout) || ((uintptr_t)workspace & 1023)) return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return SAGE_ERR_WORKSPACE;
  return launch_bwd_prepare(*shape, o, dout, workspace, L, (cudaStream_t)stream);
}

sage_status sage_attn_bwd(const sage_shape *shape, int causal, float sm_scale, int quant_mode, int flags, int bq,
                          int bk, const void *workspace, size_t workspace_bytes, const void *v, const void *dout,
                          void *dq, void *dk, void *dv, sage_stream_t stream) {
  sage_ws_layout L;
  sage_status st = request_layout(shape, quant_mode, bq, bk, &L);
  if (st != SAGE_OK) return st;
  if (quant_mode != SAGE_SAGEBWD_I8) return SAGE_ERR_UNSUPPORTED;
  if ((st = check_attn_args(shape, causal, sm_scale, quant_mode, flags, bk)) != SAGE_OK) return st;
  // per-row Q scales vary along the reduction of dK = dS^T Q: not supported here
  if (flags & SAGE_Q_PER_TOKEN) return SAGE_ERR_UNSUPPORTED;
  if (!workspace || !v || !dout || !dq || !dk || !dv) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(v) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      ((uintptr_t)workspace & 1023))
    return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return SAGE_ERR_WORKSPACE;
  return launch_attn_bwd(*shape, causal, sm_scale, flags, workspace, L, v, dout, (float *)dq, (float *)dk,
                         (float *)dv, (cudaStream_t)stream);
}

sage_status sage_read_status(const sage_shape *shape, int quant_mode, int bq, int bk, const void *workspace,
                             int *code, int *site) {
  sage_ws_layout L;
  sage_status st = request_layout(shape, quant_mode, bq, bk, &L);
  if (st != SAGE_OK) return st;
  if (!workspace || !code || !site) return SAGE_ERR_INVALID_ARG;
  int buf[4] = {0, 0, 0, 0};
  if (cudaMemcpy(buf, (const char *)workspace + L.status, sizeof(buf), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SAGE_ERR_CUDA;
  *code = buf[0];
  *site = buf[1];
  return SAGE_OK;
}

const char *sage_status_str(sage_status s) {
  switch (s) {
    case SAGE_OK: return "ok";
    case SAGE_ERR_INVALID_ARG: return "invalid argument";
    case SAGE_ERR_UNSUPPORTED: return "unsupported request";
    case SAGE_ERR_WORKSPACE: return "workspace too small";
    case SAGE_ERR_RANGE: return "input out of range (non-finite or |x| >= 2^16)";
    case SAGE_ERR_TIMEOUT: return "bounded wait gave up on the device";
    case SAGE_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

}  // extern "C"
