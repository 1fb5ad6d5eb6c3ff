// INT8 / FP8 / SageBwd attention over packed sequences (the kVar instances of
// attn_q8.cuh: work item table, per-sequence lengths, packed output rows).
#include "attn_q8.cuh"

namespace sage {

sage_status launch_attn_q8_var(const sage_shape &s, int causal, float sm_scale, int mode, int flags, int bk,
                               const void *ws, const sage_ws_layout &L, void *o, cudaStream_t stream,
                               const VarDev &var) {
  return dispatch_q8<false, true>(s, causal, sm_scale, mode, flags, bk, ws, L, o, stream, var);
}

}  // namespace sage
