"""The binding's own checks, which run before anything reaches the library: the
three inputs must agree (v read with k's dimensions), a reused workspace must
be for the same request, and the host call's tensors must match the shape the
library copies (it cannot see their sizes).  CPU tensors throughout: every
call below is refused before a device is needed."""
import pytest
import torch

import __graft_entry__

__graft_entry__.build_library()
import bit_quantized_attention_gb300 as sage  # noqa: E402


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def test_v_must_have_k_shape():
    q, k = _t(1, 2, 64, 64), _t(1, 2, 96, 64)
    with pytest.raises(ValueError, match="v must have k's shape"):
        sage.sage_quantize_qkv(q, k, _t(1, 2, 95, 64), 0, 1)
    with pytest.raises(ValueError, match="v must have k's shape"):
        sage.sage_quantize_qkv_static_scratch(q, k, _t(1, 1, 96, 64), 0, 1)


def test_inputs_dtype_layout_and_agreement():
    q, k, v = _t(1, 2, 64, 64), _t(1, 2, 96, 64), _t(1, 2, 96, 64)
    with pytest.raises(ValueError, match="bf16"):
        sage.sage_quantize_qkv(q.float(), k, v, 0, 1)
    with pytest.raises(ValueError, match="contiguous"):
        sage.sage_quantize_qkv(q.transpose(2, 3), k, v, 0, 1)
    with pytest.raises(ValueError, match="disagree"):
        sage.sage_quantize_qkv(q, _t(2, 2, 96, 64), _t(2, 2, 96, 64), 0, 1)
    with pytest.raises(ValueError, match="CUDA"):  # everything else agrees: the device is the last check
        sage.sage_quantize_qkv(q, k, v, 0, 1)


def test_reused_workspace_must_fit_the_request():
    q, k, v = _t(1, 2, 64, 64), _t(1, 2, 96, 64), _t(1, 2, 96, 64)
    other = sage.Shape(1, 2, 2, 128, 96, 64)
    L = sage.sage_workspace_layout(other, 0, 128, 64)
    ws = sage.Workspace(torch.empty(L.total, dtype=torch.uint8), other, 0, 1, 128, 64, L)
    with pytest.raises(ValueError, match="another shape"):
        sage.sage_quantize_qkv(q, k, v, 0, 1, workspace=ws)
    same = sage.Shape(1, 2, 2, 64, 96, 64)
    ws2 = sage.Workspace(torch.empty(8, dtype=torch.uint8), same, 1, 1, 128, 64, L)
    with pytest.raises(ValueError, match="another shape"):  # another quant mode
        sage.sage_quantize_qkv(q, k, v, 0, 1, workspace=ws2)


def test_output_must_fit_the_workspace():
    s = sage.Shape(1, 2, 2, 64, 96, 64)
    L = sage.sage_workspace_layout(s, 0, 128, 64)
    ws = sage.Workspace(torch.empty(8, dtype=torch.uint8), s, 0, 1, 128, 64, L)
    with pytest.raises(ValueError, match=r"\[B, Hq, N, d\]"):
        sage.sage_attn_fwd(ws, False, 0.125, out=_t(1, 2, 63, 64))


def test_host_call_tensors_match_the_shape():
    s = sage.Shape(1, 2, 2, 64, 96, 64)
    q, k, v, o = _t(1, 2, 64, 64), _t(1, 2, 96, 64), _t(1, 2, 96, 64), _t(1, 2, 64, 64)
    buf = torch.empty(16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="k_host"):
        sage.sage_attn_host(s, False, 0.125, 0, 1, 128, 64, q, _t(1, 2, 95, 64), v, o, buf)
    with pytest.raises(ValueError, match="o_host"):
        sage.sage_attn_host(s, False, 0.125, 0, 1, 128, 64, q, k, v, _t(1, 2, 64, 32), buf)
    with pytest.raises(ValueError, match="bf16"):
        sage.sage_attn_host(s, False, 0.125, 0, 1, 128, 64, q.float(), k, v, o, buf)
    with pytest.raises(ValueError, match="dev_buf"):  # host tensors right: the device buffer is checked next
        sage.sage_attn_host(s, False, 0.125, 0, 1, 128, 64, q, k, v, o, buf)


def test_lse_only_from_the_sagebwd_forward():
    s = sage.Shape(1, 2, 2, 64, 96, 64)
    L = sage.sage_workspace_layout(s, 0, 128, 64)
    ws = sage.Workspace(torch.empty(L.total, dtype=torch.uint8), s, 0, 1, 128, 64, L)
    with pytest.raises(ValueError, match="mode 3"):
        sage.sage_lse(ws)
    L3 = sage.sage_workspace_layout(s, 3, 128, 64)
    ws3 = sage.Workspace(torch.zeros(L3.total, dtype=torch.uint8), s, 3, 1, 128, 64, L3)
    assert tuple(sage.sage_lse(ws3).shape) == (1, 2, 64)


def test_backward_inputs_need_a_sagebwd_workspace():
    s = sage.Shape(1, 2, 2, 64, 96, 64)
    L = sage.sage_workspace_layout(s, 0, 128, 64)
    ws = sage.Workspace(torch.empty(L.total, dtype=torch.uint8), s, 0, 1, 128, 64, L)
    with pytest.raises(ValueError, match="mode 3"):
        sage.sage_bwd_prepare(ws, _t(1, 2, 64, 64), _t(1, 2, 64, 64))
    L3 = sage.sage_workspace_layout(s, 3, 128, 64)
    ws3 = sage.Workspace(torch.empty(L3.total, dtype=torch.uint8), s, 3, 1, 128, 64, L3)
    with pytest.raises(ValueError, match="CUDA"):
        sage.sage_bwd_prepare(ws3, _t(1, 2, 64, 64), _t(1, 2, 64, 64))
    assert L3.drow - L3.doc >= 1 * 2 * L3.N_pad * 64 * 2
