"""The pre-pass entry point whose reduction scratch lives inside the library.

Some callers may not obtain device memory for scratch (a plug-in whose host
framework owns every device allocation, or a latency-critical caller that must
not call cudaMalloc because it can synchronise the device).  For them
sage_quantize_qkv_static_scratch takes the statistics scratch from a fixed
device array in the library.  This file checks, through the C ABI, that two
calls in a row give exactly what sage_quantize_qkv gives (codes, scales and
means bit for bit, and the attention output read from each workspace), with
different inputs on the two calls so that state left in the shared array by
the first call cannot pass unnoticed.  It sits last in collection order.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from workload import make_inputs
from workload.configs import Config

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sage():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_quantized_attention_gb300 as s
    return s


def _cfg(seed):
    return Config(name="no_alloc", B=2, Hq=4, Hkv=2, N=300, M=520, d=128, causal=True, sm_scale=0.0884,
                  mode=0, flags=1 | 2 | 4, bq=128, bk=64, seed=seed, k_offset_std=3.0, q_offset_std=1.0,
                  v_bias_std=2.0)


def _regions(ws):
    L = ws.layout
    names = ["qhat", "dq", "qbar", "khat", "dk", "kbar", "vhat", "dv", "vm"]
    bounds = [getattr(L, n) for n in names] + [L.qsf]
    return {n: ws.buf[bounds[i]:bounds[i + 1]].cpu().numpy() for i, n in enumerate(names)}


def test_static_scratch_matches_workspace_scratch(sage):
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    for call, seed in enumerate((101, 202)):      # two calls in a row, different inputs
        cfg = _cfg(seed)
        q, k, v = (t.to(dev) for t in make_inputs(cfg))
        ref_ws = sage.sage_quantize_qkv(q, k, v, cfg.mode, cfg.flags, cfg.bq, cfg.bk)
        ref_o = sage.sage_attn_fwd(ref_ws, cfg.causal, cfg.sm_scale)

        shape = sage.shape_of(q, k)
        ws = sage.new_workspace(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, dev)
        ws.buf.fill_(0xA5)                           # outputs must all be written
        rc = sage.lib.sage_quantize_qkv_static_scratch(
            C.byref(shape), cfg.mode, cfg.flags, cfg.bq, cfg.bk, C.c_void_p(q.data_ptr()),
            C.c_void_p(k.data_ptr()), C.c_void_p(v.data_ptr()), C.c_void_p(ws.buf.data_ptr()),
            ws.buf.numel(), C.c_void_p(stream.cuda_stream))
        assert rc == 0, sage.sage_status_str(rc)
        o = sage.sage_attn_fwd(ws, cfg.causal, cfg.sm_scale)
        torch.cuda.synchronize()
        assert sage.sage_read_status(ws) == (0, 0)
        assert sage.sage_read_status(ref_ws) == (0, 0)

        got, want = _regions(ws), _regions(ref_ws)
        L = ws.layout
        B, Hq, Hkv, d = shape.B, shape.Hq, shape.Hkv, shape.d
        # the bytes the kernels own in each region: Q codes for all N_pad rows,
        # K codes for the Tn*bk rows the key tiles cover (rows up to M_pad beyond
        # them are layout padding nobody writes or reads), V codes for all M_pad
        views = {
            "qhat": lambda a: a[:B * Hq * L.N_pad * d * 2],
            "khat": lambda a: a[:B * Hkv * L.M_pad * d * 2].reshape(B * Hkv, L.M_pad, d * 2)[:, :L.Tn * cfg.bk],
            "vhat": lambda a: a[:B * Hkv * d * L.M_pad],
            "dq": lambda a: a[:B * Hq * L.Tm * 4], "qbar": lambda a: a[:B * Hq * L.Tm * d * 4],
            "dk": lambda a: a[:B * Hkv * L.Tn * 4], "kbar": lambda a: a[:B * Hkv * d * 4],
            "dv": lambda a: a[:B * Hkv * d * 4], "vm": lambda a: a[:B * Hkv * d * 4],
        }
        for name, view in views.items():
            assert np.array_equal(view(got[name]), view(want[name])), (call, name)

        # attention from either workspace: the parity bar of the attention tests
        a = o.float().cpu().numpy().ravel()
        b = ref_o.float().cpu().numpy().ravel()
        err = np.abs(a - b)
        assert err.max() <= 1e-2 * np.abs(b).max()
        assert err.sum() <= 2e-3 * np.abs(b).sum()


def test_static_scratch_nvfp4_matches_workspace_scratch(sage):
    """The NVFP4 pre-pass through the same entry point: packed E2M1 codes, E4M3
    block-scale atoms and the means bit for bit, two calls in a row."""
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    for call, seed in enumerate((303, 404)):
        cfg = _cfg(seed).with_(mode=2, bk=128, flags=1 | 2)
        q, k, v = (t.to(dev) for t in make_inputs(cfg))
        ref_ws = sage.sage_quantize_qkv(q, k, v, cfg.mode, cfg.flags, cfg.bq, cfg.bk)
        shape = sage.shape_of(q, k)
        ws = sage.new_workspace(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, dev)
        ws.buf.fill_(0xA5)
        rc = sage.lib.sage_quantize_qkv_static_scratch(
            C.byref(shape), cfg.mode, cfg.flags, cfg.bq, cfg.bk, C.c_void_p(q.data_ptr()),
            C.c_void_p(k.data_ptr()), C.c_void_p(v.data_ptr()), C.c_void_p(ws.buf.data_ptr()),
            ws.buf.numel(), C.c_void_p(stream.cuda_stream))
        assert rc == 0, sage.sage_status_str(rc)
        o = sage.sage_attn_fwd(ws, cfg.causal, cfg.sm_scale)
        ref_o = sage.sage_attn_fwd(ref_ws, cfg.causal, cfg.sm_scale)
        torch.cuda.synchronize()
        assert sage.sage_read_status(ws) == (0, 0)
        L = ws.layout
        B, Hq, Hkv, d = shape.B, shape.Hq, shape.Hkv, shape.d
        spans = {"qhat": B * Hq * L.N_pad * d // 2, "khat": B * Hkv * L.M_pad * d // 2,
                 "vhat": B * Hkv * d * L.M_pad // 2, "qbar": B * Hq * L.Tm * d * 4, "kbar": B * Hkv * d * 4,
                 "vm": B * Hkv * d * 4, "qsf": B * Hq * L.Tm * (d // 64) * 512,
                 "ksf": B * Hkv * (L.M_pad // 128) * (d // 64) * 512, "vsf": B * Hkv * (L.M_pad // 64) * 512}
        for name, n in spans.items():
            off = getattr(L, name)
            assert torch.equal(ws.buf[off:off + n], ref_ws.buf[off:off + n]), (call, name)
        a = o.float().cpu().numpy().ravel()
        b = ref_o.float().cpu().numpy().ravel()
        assert np.array_equal(a, b), call  # same workspace bytes, same kernel


def test_static_scratch_rejects_oversized_requests(sage):
    # B * Hkv * d = 4 * 64 * 128 = 32768 is the limit; one more kv-head is refused
    # before anything touches the device
    shape = sage.Shape(4, 65, 65, 128, 128, 128)
    fake = C.c_void_p(1 << 20)
    need = sage.sage_workspace_bytes(shape, 0, 128, 64)
    rc = sage.lib.sage_quantize_qkv_static_scratch(C.byref(shape), 0, 1, 128, 64, fake, fake, fake, fake, need, None)
    assert rc == 2
