// INT8 / FP8 / SageBwd attention entry (launch_attn_q8): the split softmax
// schedule for batched requests; packed sequences and the tiles-in-turn
// schedule have translation units of their own (attn_q8_var.cu,
// attn_q8_ping.cu) so that the instances compile in parallel.
#include <stdlib.h>

#include "attn_q8.cuh"

namespace sage {

sage_status launch_attn_q8(const sage_shape &s, int causal, float sm_scale, int mode, int flags, int bk,
                           const void *ws, const sage_ws_layout &L, void *o, cudaStream_t stream,
                           const VarDev &var) {
  if (var.item_tab) return launch_attn_q8_var(s, causal, sm_scale, mode, flags, bk, ws, L, o, stream, var);
  // whole key tiles in turn between the softmax warpgroups (SAGE_PINGPONG=1):
  // an alternative softmax schedule (not for the SageBwd forward)
  const char *pp = getenv("SAGE_PINGPONG");
  if (mode != SAGE_SAGEBWD_I8 && pp && pp[0] == '1')
    return launch_attn_q8_ping(s, causal, sm_scale, mode, flags, bk, ws, L, o, stream);
  // head dim 64 with 64-key tiles: two query blocks per work item (modes 0
  // and 1) unless SAGE_ATTN_SCHEDULE=split asks for the one-block schedule
  const char *sch = getenv("SAGE_ATTN_SCHEDULE");
  const bool split = sch && sch[0] == 's';
  if (!split && s.d == 64 && bk == 64 && (mode == SAGE_Q8_PV8 || mode == SAGE_QF8_PV8))
    return launch_attn_q8x2_64(s, causal, sm_scale, mode, flags, ws, L, o, stream);
  return dispatch_q8<false, false>(s, causal, sm_scale, mode, flags, bk, ws, L, o, stream, var);
}

}  // namespace sage
