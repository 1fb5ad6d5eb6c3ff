"""ctypes binding of libsage.so with the C ABI's names (include/sage.h).

Argument marshalling only: torch supplies device memory and the current
stream; every step of the path runs in the library's CUDA kernels.  There is
no fallback: if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsage.so")

SAGE_Q8_PV8, SAGE_QF8_PV8, SAGE_NVFP4, SAGE_SAGEBWD_I8 = 0, 1, 2, 3
SAGE_SMOOTH_K, SAGE_SMOOTH_Q, SAGE_SMOOTH_V = 1, 2, 4
SAGE_P_DIRECT, SAGE_Q_PER_TOKEN = 8, 0x10
STATUS = {0: "SAGE_OK", 1: "SAGE_ERR_INVALID_ARG", 2: "SAGE_ERR_UNSUPPORTED", 3: "SAGE_ERR_WORKSPACE",
          4: "SAGE_ERR_RANGE", 5: "SAGE_ERR_TIMEOUT", 6: "SAGE_ERR_CUDA"}

EXPORTS = ["sage_workspace_bytes", "sage_workspace_layout", "sage_quantize_qkv", "sage_attn_fwd",
           "sage_host_buffer_bytes", "sage_attn_host", "sage_read_status", "sage_status_str",
           "sage_quantize_qkv_static_scratch", "sage_varlen_workspace_bytes", "sage_attn_varlen",
           "sage_bwd_prepare", "sage_attn_bwd"]


class SageError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s" % (where, STATUS.get(code, code)))


class Shape(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("B", "Hq", "Hkv", "N", "M", "d")]

    def __iter__(self):
        return iter((self.B, self.Hq, self.Hkv, self.N, self.M, self.d))


class WsLayout(C.Structure):
    _fields_ = [(n, C.c_size_t) for n in ("qhat", "dq", "qbar", "khat", "dk", "kbar", "vhat", "dv", "vm",
                                          "qsf", "ksf", "vsf", "stats", "status", "total")] + \
               [(n, C.c_int) for n in ("N_pad", "M_pad", "Tm", "Tn")] + \
               [(n, C.c_size_t) for n in ("dqt", "dvb", "lse", "doc", "dos", "drow")]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libsage.so is not built (run __graft_entry__.build() or "
                          "python -m bit_quantized_attention_gb300.build); there is no fallback path")
    L = C.CDLL(LIB_PATH)
    P, vp, sz, i32, f32 = C.POINTER, C.c_void_p, C.c_size_t, C.c_int, C.c_float
    L.sage_workspace_bytes.argtypes, L.sage_workspace_bytes.restype = [P(Shape), i32, i32, i32], sz
    L.sage_workspace_layout.argtypes, L.sage_workspace_layout.restype = [P(Shape), i32, i32, i32, P(WsLayout)], i32
    L.sage_quantize_qkv.argtypes = [P(Shape), i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    L.sage_quantize_qkv.restype = i32
    L.sage_quantize_qkv_static_scratch.argtypes = [P(Shape), i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    L.sage_quantize_qkv_static_scratch.restype = i32
    L.sage_attn_fwd.argtypes = [P(Shape), i32, f32, i32, i32, i32, i32, vp, sz, vp, vp]
    L.sage_attn_fwd.restype = i32
    L.sage_host_buffer_bytes.argtypes, L.sage_host_buffer_bytes.restype = [P(Shape), i32, i32, i32], sz
    L.sage_attn_host.argtypes = [P(Shape), i32, f32, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    L.sage_attn_host.restype = i32
    L.sage_read_status.argtypes = [P(Shape), i32, i32, i32, vp, P(i32), P(i32)]
    L.sage_varlen_workspace_bytes.argtypes = [i32, vp, vp, i32, i32, i32, i32, i32, i32]
    L.sage_varlen_workspace_bytes.restype = sz
    L.sage_attn_varlen.argtypes = [i32, vp, vp, i32, i32, i32, i32, f32, i32, i32, i32, i32, vp, vp, vp, vp, sz,
                                   vp, vp]
    L.sage_attn_varlen.restype = i32
    L.sage_bwd_prepare.argtypes = [P(Shape), i32, i32, i32, vp, vp, vp, sz, vp]
    L.sage_bwd_prepare.restype = i32
    L.sage_attn_bwd.argtypes = [P(Shape), i32, f32, i32, i32, i32, i32, vp, sz, vp, vp, vp, vp, vp, vp]
    L.sage_attn_bwd.restype = i32
    L.sage_read_status.restype = i32
    L.sage_status_str.argtypes, L.sage_status_str.restype = [i32], C.c_char_p
    return L


lib = _load()


def _check(rc: int, where: str):
    if rc != 0:
        raise SageError(rc, where)


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: torch.Tensor) -> C.c_void_p:
    return C.c_void_p(t.data_ptr())


def _bf16_4d(t: torch.Tensor, name: str):
    if not (t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 4):
        raise ValueError("%s must be a contiguous 4-D bf16 tensor" % name)


def _bf16_cuda(t: torch.Tensor, name: str):
    _bf16_4d(t, name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)


def _qkv_shape(q, k, v) -> "Shape":
    """The shape the three inputs agree on (v must have k's shape: the library
    reads v with k's dimensions)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _bf16_4d(t, n)
    shape = shape_of(q, k)
    if tuple(v.shape) != tuple(k.shape):
        raise ValueError("v must have k's shape [B, Hkv, M, d]")
    return shape


def _same_request(ws: "Workspace", shape: "Shape", mode: int, bq: int, bk: int):
    if (tuple(ws.shape) != tuple(shape) or ws.mode != mode or ws.bq != bq or ws.bk != bk):
        raise ValueError("the workspace was made for another shape, mode or tiling")


def shape_of(q: torch.Tensor, k: torch.Tensor) -> Shape:
    B, Hq, N, d = q.shape
    Bk, Hkv, M, dk = k.shape
    if B != Bk or d != dk:
        raise ValueError("q and k disagree on batch or head dim")
    return Shape(B, Hq, Hkv, N, M, d)


def sage_workspace_layout(shape: Shape, mode: int, bq: int, bk: int) -> WsLayout:
    L = WsLayout()
    _check(lib.sage_workspace_layout(C.byref(shape), mode, bq, bk, C.byref(L)), "sage_workspace_layout")
    return L


def sage_workspace_bytes(shape: Shape, mode: int, bq: int, bk: int) -> int:
    return int(lib.sage_workspace_bytes(C.byref(shape), mode, bq, bk))


@dataclass
class Workspace:
    """A caller-owned device workspace for one (shape, mode, bq, bk, flags)."""
    buf: torch.Tensor
    shape: Shape
    mode: int
    flags: int
    bq: int
    bk: int
    layout: WsLayout

    def region(self, name: str, nbytes: int) -> torch.Tensor:
        off = getattr(self.layout, name)
        return self.buf[off:off + nbytes]


def new_workspace(shape: Shape, mode: int, flags: int, bq: int = 128, bk: int = 64, device=None) -> Workspace:
    L = sage_workspace_layout(shape, mode, bq, bk)
    buf = torch.empty(L.total + 1024, dtype=torch.uint8, device=device or "cuda")
    off = (-buf.data_ptr()) % 1024  # the library wants a 1024-byte aligned base
    return Workspace(buf[off:off + L.total], shape, mode, flags, bq, bk, L)


def sage_quantize_qkv(q, k, v, mode: int, flags: int, bq: int = 128, bk: int = 64, workspace=None,
                      stream=None) -> Workspace:
    shape = _qkv_shape(q, k, v)
    if workspace is not None:
        _same_request(workspace, shape, mode, bq, bk)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _bf16_cuda(t, n)
    ws = workspace or new_workspace(shape, mode, flags, bq, bk, q.device)
    ws.flags = flags
    _check(lib.sage_quantize_qkv(C.byref(shape), mode, flags, bq, bk, _ptr(q), _ptr(k), _ptr(v), _ptr(ws.buf),
                                 ws.buf.numel(), _stream(stream)), "sage_quantize_qkv")
    return ws


def sage_quantize_qkv_static_scratch(q, k, v, mode: int, flags: int, bq: int = 128, bk: int = 64,
                                     workspace=None, stream=None) -> Workspace:
    """The pre-pass with its reduction scratch inside the library (no scratch
    region is needed from the caller; see include/sage.h for the limit)."""
    shape = _qkv_shape(q, k, v)
    if workspace is not None:
        _same_request(workspace, shape, mode, bq, bk)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _bf16_cuda(t, n)
    ws = workspace or new_workspace(shape, mode, flags, bq, bk, q.device)
    ws.flags = flags
    _check(lib.sage_quantize_qkv_static_scratch(C.byref(shape), mode, flags, bq, bk, _ptr(q), _ptr(k), _ptr(v),
                                                _ptr(ws.buf), ws.buf.numel(), _stream(stream)),
           "sage_quantize_qkv_static_scratch")
    return ws


def sage_attn_fwd(ws: Workspace, causal: bool, sm_scale: float, out=None, stream=None) -> torch.Tensor:
    s = ws.shape
    if out is None:
        out = torch.empty((s.B, s.Hq, s.N, s.d), dtype=torch.bfloat16, device=ws.buf.device)
    else:
        _bf16_4d(out, "out")
        if tuple(out.shape) != (s.B, s.Hq, s.N, s.d) or out.device != ws.buf.device:
            raise ValueError("out must be [B, Hq, N, d] on the workspace's device")
    _check(lib.sage_attn_fwd(C.byref(s), int(bool(causal)), float(sm_scale), ws.mode, ws.flags, ws.bq, ws.bk,
                             _ptr(ws.buf), ws.buf.numel(), _ptr(out), _stream(stream)), "sage_attn_fwd")
    return out


def sage_read_status(ws: Workspace):
    code, site = C.c_int(0), C.c_int(0)
    _check(lib.sage_read_status(C.byref(ws.shape), ws.mode, ws.bq, ws.bk, _ptr(ws.buf), C.byref(code),
                                C.byref(site)), "sage_read_status")
    return code.value, site.value


def sage_host_buffer_bytes(shape: Shape, mode: int, bq: int, bk: int) -> int:
    return int(lib.sage_host_buffer_bytes(C.byref(shape), mode, bq, bk))


def sage_attn_host(shape: Shape, causal: bool, sm_scale: float, mode: int, flags: int, bq: int, bk: int,
                   q_host: torch.Tensor, k_host: torch.Tensor, v_host: torch.Tensor, o_host: torch.Tensor,
                   dev_buf: torch.Tensor, stream=None):
    """End-to-end call on host tensors (pinned for asynchronous copies)."""
    qs, ks = (shape.B, shape.Hq, shape.N, shape.d), (shape.B, shape.Hkv, shape.M, shape.d)
    for t, n, want in ((q_host, "q_host", qs), (k_host, "k_host", ks), (v_host, "v_host", ks), (o_host, "o_host", qs)):
        _bf16_4d(t, n)
        if t.is_cuda or tuple(t.shape) != want:
            raise ValueError("%s must be a host tensor of shape %s" % (n, want))
    if not dev_buf.is_cuda or (dev_buf.data_ptr() % 1024) != 0:
        raise ValueError("dev_buf must be a 1024-byte aligned CUDA buffer")
    _check(lib.sage_attn_host(C.byref(shape), int(bool(causal)), float(sm_scale), mode, flags, bq, bk,
                              _ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(o_host), _ptr(dev_buf),
                              dev_buf.numel(), _stream(stream)), "sage_attn_host")


def sage_host_status(dev_buf: torch.Tensor):
    """(code, site) of the last sage_attn_host call on dev_buf: the status word
    at its start (read after the call's stream has completed)."""
    st = dev_buf[:16].view(torch.int32).cpu().tolist()
    return st[0], st[1]


def sage_status_str(code: int) -> str:
    return lib.sage_status_str(code).decode()


def _cu(cu, name: str):
    """cu_seqlens (ints, or a CPU int tensor) -> (ctypes int32 array, list)"""
    if isinstance(cu, torch.Tensor):
        if cu.is_cuda:
            raise ValueError("%s must be on the host (the library sizes the work from it)" % name)
        cu = cu.tolist()
    vals = [int(x) for x in cu]
    if len(vals) < 2:
        raise ValueError("%s needs nseq + 1 >= 2 entries" % name)
    return (C.c_int * len(vals))(*vals), vals


def sage_varlen_workspace_bytes(cu_seqlens_q, cu_seqlens_k, Hq: int, Hkv: int, d: int, mode: int, bq: int = 128,
                                bk: int = 64) -> int:
    aq, lq = _cu(cu_seqlens_q, "cu_seqlens_q")
    ak, lk = _cu(cu_seqlens_k, "cu_seqlens_k")
    if len(lq) != len(lk):
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    return int(lib.sage_varlen_workspace_bytes(len(lq) - 1, aq, ak, Hq, Hkv, d, mode, bq, bk))


def sage_attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool, sm_scale: float, mode: int = SAGE_Q8_PV8,
                     flags: int = SAGE_SMOOTH_K, bq: int = 128, bk: int = 64, out=None, stream=None):
    """Packed sequences: q [total_q, Hq, d], k and v [total_k, Hkv, d] (bf16, CUDA,
    contiguous), cu_seqlens on the host.  Returns (o [total_q, Hq, d], the
    Workspace: the batched layout of (nseq, Hq, Hkv, longest query run, longest
    key run, d), for sage_read_status and sage_lse)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not (t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 3 and t.is_cuda):
            raise ValueError("%s must be a contiguous 3-D bf16 CUDA tensor [total, H, d]" % n)
    if tuple(v.shape) != tuple(k.shape) or q.shape[2] != k.shape[2]:
        raise ValueError("v must have k's shape and q, k the same head dim")
    aq, lq = _cu(cu_seqlens_q, "cu_seqlens_q")
    ak, lk = _cu(cu_seqlens_k, "cu_seqlens_k")
    if len(lq) != len(lk) or lq[-1] != q.shape[0] or lk[-1] != k.shape[0]:
        raise ValueError("cu_seqlens must end at the packed lengths and have the same number of entries")
    nseq, Hq, Hkv, d = len(lq) - 1, q.shape[1], k.shape[1], q.shape[2]
    need = sage_varlen_workspace_bytes(lq, lk, Hq, Hkv, d, mode, bq, bk)
    if need == 0:
        raise SageError(2, "sage_varlen_workspace_bytes")
    shape = Shape(nseq, Hq, Hkv, max(b - a for a, b in zip(lq, lq[1:])), max(b - a for a, b in zip(lk, lk[1:])), d)
    L = sage_workspace_layout(shape, mode, bq, bk)
    buf = torch.empty(need + 1024, dtype=torch.uint8, device=q.device)
    off = (-buf.data_ptr()) % 1024
    ws = Workspace(buf[off:off + need], shape, mode, flags, bq, bk, L)
    if out is None:
        out = torch.empty_like(q)
    elif not (out.dtype == torch.bfloat16 and out.is_contiguous() and tuple(out.shape) == tuple(q.shape)
              and out.device == q.device):
        raise ValueError("out must be a contiguous bf16 tensor shaped and placed like q")
    _check(lib.sage_attn_varlen(nseq, aq, ak, Hq, Hkv, d, int(bool(causal)), float(sm_scale), mode, flags, bq, bk,
                                _ptr(q), _ptr(k), _ptr(v), _ptr(ws.buf), need, _ptr(out), _stream(stream)),
           "sage_attn_varlen")
    return out, ws


def sage_bwd_prepare(ws: Workspace, o, dout, stream=None):
    """The SageBwd backward's inputs into a mode-3 workspace: dO codes and
    scales, D = rowsum(dO o O); o and dout bf16 [B, Hq, N, d] on the device.
    Returns views (dO codes as fp16 [B, Hq, N, d], scales [B, Hq, Tm], D [B, Hq, N])."""
    if ws.mode != SAGE_SAGEBWD_I8:
        raise ValueError("the backward's inputs live in a mode 3 (SageBwd) workspace")
    s, L = ws.shape, ws.layout
    want = (s.B, s.Hq, s.N, s.d)
    for t, n in ((o, "o"), (dout, "dout")):
        _bf16_cuda(t, n)
        if tuple(t.shape) != want:
            raise ValueError("%s must have the shape [B, Hq, N, d] = %s" % (n, want))
    _check(lib.sage_bwd_prepare(C.byref(s), ws.mode, ws.bq, ws.bk, _ptr(o), _ptr(dout), _ptr(ws.buf),
                                ws.buf.numel(), _stream(stream)), "sage_bwd_prepare")
    doc = ws.region("doc", s.B * s.Hq * L.N_pad * s.d * 2).view(torch.float16).view(s.B, s.Hq, L.N_pad, s.d)
    dos = ws.region("dos", s.B * s.Hq * L.Tm * 4).view(torch.float32).view(s.B, s.Hq, L.Tm)
    drow = ws.region("drow", s.B * s.Hq * L.N_pad * 4).view(torch.float32).view(s.B, s.Hq, L.N_pad)
    return doc[:, :, :s.N], dos, drow[:, :, :s.N]


def sage_attn_bwd(ws: Workspace, causal: bool, sm_scale: float, v, dout, dq=None, dk=None, dv=None,
                  stream=None):
    """The SageBwd backward on a mode-3 workspace that sage_attn_fwd and
    sage_bwd_prepare have filled: v the forward's bf16 V [B, Hkv, M, d], dout
    the bf16 dO [B, Hq, N, d].  Returns (dq, dk, dv) as float32 tensors
    (dq [B, Hq, N, d]; dk, dv [B, Hkv, M, d]), into the given ones if any."""
    if ws.mode != SAGE_SAGEBWD_I8:
        raise ValueError("the backward runs on a mode 3 (SageBwd) workspace")
    s = ws.shape
    qshape, kshape = (s.B, s.Hq, s.N, s.d), (s.B, s.Hkv, s.M, s.d)
    _bf16_cuda(v, "v")
    _bf16_cuda(dout, "dout")
    if tuple(v.shape) != kshape or tuple(dout.shape) != qshape:
        raise ValueError("v must be [B, Hkv, M, d] = %s and dout [B, Hq, N, d] = %s" % (kshape, qshape))
    dev = ws.buf.device
    outs = []
    for t, shp, n in ((dq, qshape, "dq"), (dk, kshape, "dk"), (dv, kshape, "dv")):
        if t is None:
            t = torch.empty(shp, dtype=torch.float32, device=dev)
        elif t.dtype != torch.float32 or tuple(t.shape) != shp or not t.is_contiguous() or t.device != dev:
            raise ValueError("%s must be a contiguous float32 tensor %s on the workspace's device" % (n, shp))
        outs.append(t)
    _check(lib.sage_attn_bwd(C.byref(s), int(bool(causal)), float(sm_scale), ws.mode, ws.flags, ws.bq, ws.bk,
                             _ptr(ws.buf), ws.buf.numel(), _ptr(v), _ptr(dout), _ptr(outs[0]), _ptr(outs[1]),
                             _ptr(outs[2]), _stream(stream)), "sage_attn_bwd")
    return tuple(outs)


def sage_lse(ws: Workspace) -> torch.Tensor:
    """The per-row log-sum-exp the SageBwd forward (mode 3) wrote into the
    workspace, ln sum_j exp(S_ij sm_scale), as a float32 view [B, Hq, N]."""
    if ws.mode != SAGE_SAGEBWD_I8:
        raise ValueError("the log-sum-exp is written by the SageBwd forward (mode 3) only")
    s, L = ws.shape, ws.layout
    t = ws.region("lse", s.B * s.Hq * L.N_pad * 4).view(torch.float32)
    return t.view(s.B, s.Hq, L.N_pad)[:, :, :s.N]


def sage_attn(q, k, v, causal: bool, sm_scale: float, mode: int = SAGE_Q8_PV8, flags: int = SAGE_SMOOTH_K,
              bq: int = 128, bk: int = 64, stream=None) -> torch.Tensor:
    """Quantize + attend: the two library calls in order on one stream."""
    ws = sage_quantize_qkv(q, k, v, mode, flags, bq, bk, stream=stream)
    return sage_attn_fwd(ws, causal, sm_scale, stream=stream)
