"""GB300 (sm_103a) SageAttention-style quantized attention forward.

The compute path is libsage.so (CUDA kernels behind a C ABI, include/sage.h);
this package is its thin ctypes binding.  Importing it loads the library and
raises ImportError if it has not been built.
"""
from ._binding import (  # noqa: F401
    SAGE_Q8_PV8, SAGE_QF8_PV8, SAGE_NVFP4, SAGE_SAGEBWD_I8, SAGE_SMOOTH_K, SAGE_SMOOTH_Q, SAGE_SMOOTH_V, SAGE_P_DIRECT, SAGE_Q_PER_TOKEN,
    EXPORTS, LIB_PATH, SageError, Shape, Workspace, WsLayout, lib, new_workspace, sage_attn,
    sage_attn_fwd, sage_attn_host, sage_host_status, sage_lse, sage_attn_varlen, sage_varlen_workspace_bytes, sage_bwd_prepare, sage_attn_bwd, sage_host_buffer_bytes, sage_quantize_qkv, sage_read_status,
    sage_quantize_qkv_static_scratch,
    sage_status_str, sage_workspace_bytes, sage_workspace_layout, shape_of,
)
