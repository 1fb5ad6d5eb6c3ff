"""Oracle for the quantized attention path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding) never does, and shares no code with it.
"""
from .oracle import (  # noqa: F401
    build, lib, quantize, attn_rows, attn_rows_lse, attn_exact_rows, attn_varlen, sagebwd_backward, sagebwd_prepare, e4m3_encode, e4m3_decode,
    e2m1_encode, e2m1_decode, bf16_encode, mean_bf16, int8_code, int8_scale,
    fp8_scale, fp8_code, nvfp4_scale, nvfp4_code, Quant, parallel_attn_rows, all_rows, bf16_round,
    MODE_Q8_PV8, MODE_QF8_PV8, MODE_NVFP4, MODE_SAGEBWD_I8, SMOOTH_K, SMOOTH_Q, SMOOTH_V,
    EXACT_QK, EXACT_PV, EXACT_BWD, BWD_INT8_DP, P_DIRECT, Q_PER_TOKEN, OracleError,
)
