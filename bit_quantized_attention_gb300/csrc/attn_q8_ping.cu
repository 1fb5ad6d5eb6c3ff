// INT8 / FP8 attention with the softmax warpgroups taking whole key tiles in
// turn (the kPing instances of attn_q8.cuh), batched requests.
#include "attn_q8.cuh"

namespace sage {

sage_status launch_attn_q8_ping(const sage_shape &s, int causal, float sm_scale, int mode, int flags, int bk,
                                const void *ws, const sage_ws_layout &L, void *o, cudaStream_t stream) {
  return dispatch_q8<true, false>(s, causal, sm_scale, mode, flags, bk, ws, L, o, stream, VarDev());
}

}  // namespace sage
