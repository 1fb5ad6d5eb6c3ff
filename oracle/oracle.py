"""ctypes wrapper of the C oracle (sage_oracle.c) — TEST INFRASTRUCTURE ONLY.

``build()`` compiles the plain C file with gcc (no vendor code, no CUDA) into
``oracle/liborc.so`` next to the source.  All array marshalling is numpy.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "sage_oracle.c")
LIB = os.path.join(HERE, "liborc.so")

MODE_Q8_PV8, MODE_QF8_PV8, MODE_NVFP4 = 0, 1, 2
MODE_SAGEBWD_I8 = 3  # SageBwd forward: INT8 per-block Q, K, V; INT8 per-token P~
SMOOTH_K, SMOOTH_Q, SMOOTH_V = 1, 2, 4
P_DIRECT = 8  # NVFP4 ablation: phi on P~ directly (no level-1 scale)
Q_PER_TOKEN = 0x10  # one Q scale per query row (INT8 / E4M3 modes)
EXACT_QK, EXACT_PV = 0x100, 0x200
EXACT_BWD = 0x400  # backward: P, dO, dS unquantized
BWD_INT8_DP = 0x800  # backward ablation: dP = dO V^T from INT8 dO^ and V^

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle; contraction off so each binary32 step rounds once."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(
            os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "sage_oracle.h"))):
        return LIB
    tmp = LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


class _Shape(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("B", "Hq", "Hkv", "N", "M", "d")]


class _Quant(C.Structure):
    _fields_ = [("qc", C.c_void_p), ("dq", C.c_void_p), ("qbar", C.c_void_p),
                ("kc", C.c_void_p), ("dk", C.c_void_p), ("kbar", C.c_void_p),
                ("vc", C.c_void_p), ("dv", C.c_void_p), ("vm", C.c_void_p),
                ("qs", C.c_void_p), ("ks", C.c_void_p), ("vs", C.c_void_p), ("dqt", C.c_void_p),
                ("dvb", C.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            vp, i64, dbl, i32 = C.c_void_p, C.c_int64, C.c_double, C.c_int
            L.orc_e4m3_encode.argtypes, L.orc_e4m3_encode.restype = [dbl], C.c_uint8
            L.orc_e4m3_decode.argtypes, L.orc_e4m3_decode.restype = [C.c_uint8], dbl
            L.orc_e2m1_encode.argtypes, L.orc_e2m1_encode.restype = [dbl], C.c_uint8
            L.orc_e2m1_decode.argtypes, L.orc_e2m1_decode.restype = [C.c_uint8], dbl
            L.orc_bf16_encode.argtypes, L.orc_bf16_encode.restype = [dbl], C.c_uint16
            for f in ("orc_e4m3_encode_array", "orc_e2m1_encode_array", "orc_bf16_encode_array"):
                getattr(L, f).argtypes, getattr(L, f).restype = [vp, i64, vp], None
            L.orc_mean_bf16.argtypes, L.orc_mean_bf16.restype = [vp, i64, i64, vp], i32
            L.orc_int8_scale.argtypes, L.orc_int8_scale.restype = [C.c_float], C.c_float
            L.orc_int8_code.argtypes, L.orc_int8_code.restype = [C.c_float, C.c_float], i32
            L.orc_fp8_scale.argtypes, L.orc_fp8_scale.restype = [C.c_float], C.c_float
            L.orc_fp8_code.argtypes, L.orc_fp8_code.restype = [C.c_float, C.c_float], C.c_uint8
            L.orc_nvfp4_scale.argtypes, L.orc_nvfp4_scale.restype = [C.c_float], C.c_uint8
            L.orc_nvfp4_code.argtypes, L.orc_nvfp4_code.restype = [C.c_float, C.c_uint8], C.c_uint8
            L.orc_quantize.argtypes = [C.POINTER(_Shape), i32, i32, i32, i32, vp, vp, vp,
                                       C.POINTER(_Quant)]
            L.orc_quantize.restype = i32
            L.orc_attn_rows.argtypes = [C.POINTER(_Shape), i32, i32, i32, i32, i32, dbl, vp, vp, vp,
                                        C.POINTER(_Quant), vp, i64, vp]
            L.orc_attn_rows.restype = i32
            L.orc_attn_rows_lse.argtypes = L.orc_attn_rows.argtypes + [vp]
            L.orc_attn_rows_lse.restype = i32
            L.orc_sagebwd_backward.argtypes = [C.POINTER(_Shape), i32, i32, i32, i32, dbl, vp, vp,
                                               C.POINTER(_Quant), vp, vp, vp, vp, vp, vp, vp]
            L.orc_sagebwd_backward.restype = i32
            L.orc_sagebwd_prepare.argtypes = [C.POINTER(_Shape), i32, vp, vp, vp, vp, vp]
            L.orc_sagebwd_prepare.restype = i32
            L.orc_attn_exact_rows.argtypes = [C.POINTER(_Shape), i32, dbl, vp, vp, vp, vp, i64, vp]
            L.orc_attn_exact_rows.restype = i32
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------- codecs
def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def e2m1_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, np.uint8)
    lib().orc_e2m1_encode_array(_p(x), x.size, _p(out))
    return out


def bf16_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_encode_array(_p(x), x.size, _p(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    tab = np.array([lib().orc_e4m3_decode(i) for i in range(256)], np.float64)
    return tab[c]


def e2m1_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    tab = np.array([lib().orc_e2m1_decode(i) for i in range(16)], np.float64)
    return tab[c]


def mean_bf16(bits: np.ndarray) -> float:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.zeros(1, np.float32)
    rc = lib().orc_mean_bf16(_p(bits), bits.size, 1, _p(out))
    if rc:
        raise OracleError("orc_mean_bf16 rc=%d" % rc)
    return float(out[0])


def int8_scale(absmax: float) -> float:
    return lib().orc_int8_scale(absmax)


def int8_code(x: float, scale: float) -> int:
    return lib().orc_int8_code(x, scale)


def fp8_scale(absmax: float) -> float:
    return lib().orc_fp8_scale(absmax)


def fp8_code(x: float, scale: float) -> int:
    return lib().orc_fp8_code(x, scale)


def nvfp4_scale(absmax: float) -> int:
    return lib().orc_nvfp4_scale(absmax)


def nvfp4_code(x: float, sc: int) -> int:
    return lib().orc_nvfp4_code(x, sc)


# ---------------------------------------------------------------- the method
@dataclass
class Quant:
    """Quantized Q, K, V in logical (unpadded) layouts; see sage_oracle.h."""
    qc: np.ndarray
    dq: np.ndarray
    qbar: np.ndarray
    kc: np.ndarray
    dk: np.ndarray
    kbar: np.ndarray
    vc: np.ndarray
    dv: np.ndarray
    vm: np.ndarray
    qs: np.ndarray
    ks: np.ndarray
    vs: np.ndarray
    dqt: np.ndarray  # per-token Q scales (Q_PER_TOKEN)
    dvb: np.ndarray  # per-block V scales (MODE_SAGEBWD_I8)

    def _struct(self):
        return _Quant(*[_p(getattr(self, f)) for f, _ in _Quant._fields_])


def _shape(B, Hq, Hkv, N, M, d):
    return _Shape(B, Hq, Hkv, N, M, d)


def _bits(t) -> np.ndarray:
    """bf16 torch tensor or uint16 array -> contiguous uint16 bit array."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def quantize(shape, mode, flags, bq, bk, q, k, v) -> Quant:
    B, Hq, Hkv, N, M, d = shape
    Tm, Tn = -(-N // bq), -(-M // bk)
    G = max(d // 16, 1)
    Mt16 = -(-M // 16)
    qz = Quant(
        qc=np.zeros((B, Hq, N, d), np.uint8), dq=np.zeros((B, Hq, Tm), np.float32),
        qbar=np.zeros((B, Hq, Tm, d), np.float32),
        kc=np.zeros((B, Hkv, M, d), np.uint8), dk=np.zeros((B, Hkv, Tn), np.float32),
        kbar=np.zeros((B, Hkv, d), np.float32),
        vc=np.zeros((B, Hkv, M, d), np.uint8), dv=np.zeros((B, Hkv, d), np.float32),
        vm=np.zeros((B, Hkv, d), np.float32),
        qs=np.zeros((B, Hq, N, G), np.uint8), ks=np.zeros((B, Hkv, M, G), np.uint8),
        vs=np.zeros((B, Hkv, Mt16, d), np.uint8), dqt=np.zeros((B, Hq, N), np.float32),
        dvb=np.zeros((B, Hkv, Tn), np.float32))
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    assert qb.size == B * Hq * N * d and kb.size == B * Hkv * M * d and vb.size == kb.size
    st = qz._struct()
    rc = lib().orc_quantize(C.byref(_shape(*shape)), mode, flags, bq, bk, _p(qb), _p(kb), _p(vb),
                            C.byref(st))
    if rc:
        raise OracleError("orc_quantize rc=%d" % rc)
    return qz


def attn_rows(shape, mode, flags, bq, bk, causal, sm_scale, q, k, v, qz: Quant, rows) -> np.ndarray:
    """fp64 output rows of the quantized attention; rows are (b*Hq+h)*N + r."""
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    d = shape[5]
    out = np.zeros((rows.size, d), np.float64)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    st = qz._struct()
    rc = lib().orc_attn_rows(C.byref(_shape(*shape)), mode, flags, bq, bk, int(bool(causal)),
                             float(sm_scale), _p(qb), _p(kb), _p(vb), C.byref(st), _p(rows),
                             rows.size, _p(out))
    if rc:
        raise OracleError("orc_attn_rows rc=%d" % rc)
    return out


def attn_rows_lse(shape, mode, flags, bq, bk, causal, sm_scale, q, k, v, qz: Quant, rows):
    """(out, lse): the fp64 output rows and each row's m + ln(l) after the last key tile."""
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    d = shape[5]
    out = np.zeros((rows.size, d), np.float64)
    lse = np.zeros(rows.size, np.float64)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    st = qz._struct()
    rc = lib().orc_attn_rows_lse(C.byref(_shape(*shape)), mode, flags, bq, bk, int(bool(causal)),
                                 float(sm_scale), _p(qb), _p(kb), _p(vb), C.byref(st), _p(rows),
                                 rows.size, _p(out), _p(lse))
    if rc:
        raise OracleError("orc_attn_rows_lse rc=%d" % rc)
    return out, lse


def sagebwd_backward(shape, flags, bq, bk, causal, sm_scale, q, k, v, qz: Quant, o, dout, lse):
    """(dq, dk, dv) fp64 of the SageBwd backward; o fp64 [B,Hq,N,d] and lse fp64
    [B,Hq,N] from the forward, dout bf16 [B,Hq,N,d]; see sage_oracle.h."""
    B, Hq, Hkv, N, M, d = shape
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
    o = np.ascontiguousarray(o, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    assert o.size == B * Hq * N * d and lse.size == B * Hq * N and db.size == o.size
    dq = np.zeros((B, Hq, N, d), np.float64)
    dk = np.zeros((B, Hkv, M, d), np.float64)
    dv = np.zeros((B, Hkv, M, d), np.float64)
    st = qz._struct()
    rc = lib().orc_sagebwd_backward(C.byref(_shape(*shape)), flags, bq, bk, int(bool(causal)),
                                    float(sm_scale), _p(qb), _p(kb), C.byref(st), _p(vb), _p(o), _p(db),
                                    _p(lse), _p(dq), _p(dk), _p(dv))
    if rc:
        raise OracleError("orc_sagebwd_backward rc=%d" % rc)
    return dq, dk, dv


def sagebwd_prepare(shape, bq, o, dout):
    """(dO codes int8 [B,Hq,N,d], dO block scales [B,Hq,Tm], D [B,Hq,N]) of the
    SageBwd backward; o fp64 [B,Hq,N,d], dout bf16 [B,Hq,N,d]."""
    B, Hq, Hkv, N, M, d = shape
    Tm = -(-N // bq)
    db = _bits(dout)
    o = np.ascontiguousarray(o, dtype=np.float64)
    assert o.size == B * Hq * N * d and db.size == o.size
    doc = np.zeros((B, Hq, N, d), np.int8)
    dos = np.zeros((B, Hq, Tm), np.float32)
    D = np.zeros((B, Hq, N), np.float64)
    rc = lib().orc_sagebwd_prepare(C.byref(_shape(*shape)), bq, _p(o), _p(db), _p(doc), _p(dos), _p(D))
    if rc:
        raise OracleError("orc_sagebwd_prepare rc=%d" % rc)
    return doc, dos, D


def attn_exact_rows(shape, causal, sm_scale, q, k, v, rows) -> np.ndarray:
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    d = shape[5]
    out = np.zeros((rows.size, d), np.float64)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    rc = lib().orc_attn_exact_rows(C.byref(_shape(*shape)), int(bool(causal)), float(sm_scale),
                                   _p(qb), _p(kb), _p(vb), _p(rows), rows.size, _p(out))
    if rc:
        raise OracleError("orc_attn_exact_rows rc=%d" % rc)
    return out


def all_rows(shape) -> np.ndarray:
    B, Hq, _, N, _, _ = shape
    return np.arange(B * Hq * N, dtype=np.int64)


def parallel_attn_rows(shape, mode, flags, bq, bk, causal, sm_scale, q, k, v, qz, rows,
                       threads: int | None = None) -> np.ndarray:
    """Same as attn_rows, with independent row chunks on several host threads
    (ctypes releases the GIL; the C code has no shared mutable state)."""
    from concurrent.futures import ThreadPoolExecutor
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    threads = threads or os.cpu_count() or 1
    chunks = [c for c in np.array_split(rows, max(1, min(threads * 4, rows.size))) if c.size]
    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda c: attn_rows(shape, mode, flags, bq, bk, causal, sm_scale,
                                                  q, k, v, qz, c), chunks))
    return np.concatenate(parts, axis=0)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 (nearest even) -> fp64: the method's final output rounding."""
    bits = bf16_encode(x)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)




# ---------------------------------------------------------------- varlen (packed sequences)
def _packed_bits(x) -> np.ndarray:
    """bf16 [total, H, d] tensor or uint16 array -> contiguous uint16 [total, H, d]."""
    b = _bits(x)
    assert b.ndim == 3
    return b


def _seq_lens(cu, name):
    cu = np.asarray(cu, dtype=np.int64)
    if cu.ndim != 1 or cu.size < 2 or cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise OracleError("%s must start at 0 and not decrease" % name)
    return cu


def attn_varlen(mode, flags, bq, bk, causal, sm_scale, q, k, v, cu_seqlens_q, cu_seqlens_k):
    """Quantized attention over packed sequences (the varlen interface of the
    SageAttention production guide, "Handling Varying Sequence Lengths with
    VarLen Kernels"): q [total_q, Hq, d], k and v [total_k, Hkv, d], sequence s
    holding rows cu_seqlens_q[s]:cu_seqlens_q[s+1] and keys
    cu_seqlens_k[s]:cu_seqlens_k[s+1].  Each sequence is its own attention
    problem: its own means, its own query and key blocks starting at its first
    token, its own bottom-right causal mask.  Returns (out [total_q, Hq, d] fp64,
    lse [total_q, Hq], one Quant per sequence or None for a sequence with no
    query).  A sequence with queries but no keys is an argument error."""
    qb, kb, vb = _packed_bits(q), _packed_bits(k), _packed_bits(v)
    cq, ck = _seq_lens(cu_seqlens_q, "cu_seqlens_q"), _seq_lens(cu_seqlens_k, "cu_seqlens_k")
    Hq, d, Hkv = qb.shape[1], qb.shape[2], kb.shape[1]
    if cq.size != ck.size or cq[-1] != qb.shape[0] or ck[-1] != kb.shape[0] or vb.shape != kb.shape:
        raise OracleError("cu_seqlens and packed tensors disagree")
    out = np.zeros((qb.shape[0], Hq, d), np.float64)
    lse = np.zeros((qb.shape[0], Hq), np.float64)
    quants = []
    for s in range(cq.size - 1):
        Lq, Lk = int(cq[s + 1] - cq[s]), int(ck[s + 1] - ck[s])
        if Lq == 0:
            quants.append(None)
            continue
        if Lk == 0:
            raise OracleError("sequence %d has queries but no keys" % s)
        shape = (1, Hq, Hkv, Lq, Lk, d)
        qs = np.ascontiguousarray(qb[cq[s]:cq[s + 1]].transpose(1, 0, 2))
        ks = np.ascontiguousarray(kb[ck[s]:ck[s + 1]].transpose(1, 0, 2))
        vs = np.ascontiguousarray(vb[ck[s]:ck[s + 1]].transpose(1, 0, 2))
        qz = quantize(shape, mode, flags & 0xFF, bq, bk, qs, ks, vs)
        o, l = attn_rows_lse(shape, mode, flags, bq, bk, causal, sm_scale, qs, ks, vs, qz, all_rows(shape))
        out[cq[s]:cq[s + 1]] = o.reshape(Hq, Lq, d).transpose(1, 0, 2)
        lse[cq[s]:cq[s + 1]] = l.reshape(Hq, Lq).T
        quants.append(qz)
    return out, lse, quants
