// The two-query-block INT8 / FP8 attention (attn_q8x2.cuh) at head dim 64.
#include "attn_q8x2.cuh"
