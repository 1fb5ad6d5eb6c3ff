"""The C ABI library loads and exports every symbol include/sage.h declares;
host-side checks (layout, argument validation) behave as documented.

Every call here fails validation before anything is launched, so these tests
run without a GPU (and never hand a device a fake pointer on one that has it).
"""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sage():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_quantized_attention_gb300 as s
    return s


def declared_functions():
    src = open(os.path.join(ROOT, "include", "sage.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sage_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sage_quantize_qkv", "sage_attn_fwd", "sage_workspace_bytes", "sage_read_status"):
        assert n in names


def test_library_exports_every_declared_symbol(sage):
    lib = C.CDLL(sage.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(sage.EXPORTS) == set(declared_functions())


def test_workspace_layout_is_aligned_and_ordered(sage):
    for shp, mode, bk in [((4, 32, 32, 4096, 4096, 128), 0, 64), ((2, 48, 48, 17776, 17776, 64), 0, 64),
                          ((1, 32, 8, 4096, 65536, 128), 1, 128), ((1, 2, 2, 256, 256, 64), 0, 64)]:
        s = sage.Shape(*shp)
        L = sage.sage_workspace_layout(s, mode, 128, bk).as_dict()
        offs = [L[k] for k in ("qhat", "dq", "qbar", "khat", "dk", "kbar", "vhat", "dv", "vm", "qsf", "ksf",
                               "vsf", "stats", "status", "dqt", "total")]
        assert all(o % 1024 == 0 for o in offs)
        assert offs == sorted(offs)
        assert L["N_pad"] % 128 == 0 and L["N_pad"] >= shp[3]
        assert L["M_pad"] % 128 == 0 and L["M_pad"] >= shp[4]
        assert L["Tn"] == -(-shp[4] // bk)
        code_b = 2 if mode == 0 else 1
        assert L["dq"] - L["qhat"] >= shp[0] * shp[1] * L["N_pad"] * shp[5] * code_b
        assert L["total"] - L["dqt"] >= shp[0] * shp[1] * L["N_pad"] * 4     # one Q scale per row
        assert sage.sage_workspace_bytes(s, mode, 128, bk) == L["total"]


@pytest.mark.parametrize("shp,mode,bq,bk,code", [
    ((1, 2, 2, 256, 256, 96), 0, 128, 64, 2),     # head dim not in {64, 128}
    ((1, 3, 2, 256, 256, 64), 0, 128, 64, 1),     # Hq % Hkv != 0
    ((1, 2, 2, 256, 256, 64), 0, 64, 64, 2),      # bq != 128
    ((1, 2, 2, 256, 256, 64), 0, 128, 32, 2),     # bk not in {64, 128}
    ((1, 2, 2, 0, 256, 64), 0, 128, 64, 1),       # empty query
    ((1, 2, 2, 256, 0, 64), 0, 128, 64, 1),       # empty keys
    ((1, 2, 2, 256, 256, 64), 7, 128, 64, 1),     # unknown mode
    ((1, 2, 2, 1 << 24, 256, 64), 0, 128, 64, 2),  # beyond the exact-mean token limit
    ((1024, 1024, 1024, 1 << 23, 256, 64), 0, 128, 64, 2),  # 2^36 query blocks: past the kernels' int counts
    ((1, 512, 512, 256, 1 << 23, 64), 0, 128, 64, 2),  # 2^32 K rows: past a TMA row coordinate
])
def test_invalid_requests_rejected(sage, shp, mode, bq, bk, code):
    s = sage.Shape(*shp)
    assert sage.sage_workspace_bytes(s, mode, bq, bk) == 0
    L = sage.WsLayout()
    assert sage.lib.sage_workspace_layout(C.byref(s), mode, bq, bk, C.byref(L)) == code
    fake = C.c_void_p(1 << 20)
    rc = sage.lib.sage_quantize_qkv(C.byref(s), mode, 1, bq, bk, fake, fake, fake, fake, 1 << 40, None)
    assert rc == code


def test_pointer_workspace_and_flag_checks(sage):
    s = sage.Shape(1, 2, 2, 256, 256, 64)
    need = sage.sage_workspace_bytes(s, 0, 128, 64)
    ok = C.c_void_p(1 << 20)                 # 1024-aligned, never dereferenced: every call below fails first
    q = sage.lib.sage_quantize_qkv
    a = sage.lib.sage_attn_fwd
    assert q(C.byref(s), 0, 1, 128, 64, None, ok, ok, ok, need, None) == 1            # null q
    assert q(C.byref(s), 0, 1, 128, 64, C.c_void_p((1 << 20) + 8), ok, ok, ok, need, None) == 1  # misaligned
    assert q(C.byref(s), 0, 1, 128, 64, ok, ok, ok, C.c_void_p((1 << 20) + 16), need, None) == 1  # ws align
    assert q(C.byref(s), 0, 1, 128, 64, ok, ok, ok, ok, need - 1, None) == 3          # workspace too small
    assert q(C.byref(s), 0, 64, 128, 64, ok, ok, ok, ok, need, None) == 1             # unknown flag
    assert a(C.byref(s), 0, 0.125, 0, 1, 128, 64, ok, need - 1, ok, None) == 3
    assert a(C.byref(s), 0, 0.0, 0, 1, 128, 64, ok, need, ok, None) == 1              # sm_scale <= 0
    assert a(C.byref(s), 0, float("nan"), 0, 1, 128, 64, ok, need, ok, None) == 1
    assert a(C.byref(s), 0, 0.125, 0, 1, 128, 64, ok, need, None, None) == 1          # null output
    s2 = sage.Shape(1, 2, 2, 512, 256, 64)
    need2 = sage.sage_workspace_bytes(s2, 0, 128, 64)
    assert a(C.byref(s2), 1, 0.125, 0, 1, 128, 64, ok, need2, ok, None) == 2          # causal with N > M


def test_backward_checks_before_any_launch(sage):
    """sage_attn_bwd: the SageBwd mode only, no per-token Q scales, every
    pointer present and aligned, a large enough workspace."""
    s = sage.Shape(1, 2, 2, 256, 256, 64)
    need = sage.sage_workspace_bytes(s, 3, 128, 64)
    ok = C.c_void_p(1 << 20)
    f = sage.lib.sage_attn_bwd

    def call(shape=s, causal=0, scale=0.125, mode=3, flags=1, bk=64, ws=ok, n=need, v=ok, do=ok, dq=ok, dk=ok, dv=ok):
        return f(C.byref(shape), causal, scale, mode, flags, 128, bk, ws, n, v, do, dq, dk, dv, None)
    assert call(mode=0, n=sage.sage_workspace_bytes(s, 0, 128, 64)) == 2     # not the SageBwd mode
    assert call(bk=128) == 2                                                 # SageBwd takes 64-key blocks
    assert call(flags=1 | 0x10) == 2                                         # per-token Q scales
    assert call(flags=64) == 1 and call(scale=0.0) == 1
    assert call(v=None) == 1 and call(do=None) == 1 and call(dq=None) == 1 and call(dk=None) == 1
    assert call(dv=C.c_void_p((1 << 20) + 4)) == 1                           # misaligned output
    assert call(ws=C.c_void_p((1 << 20) + 512)) == 1                         # workspace alignment
    assert call(n=need - 1) == 3
    s2 = sage.Shape(1, 2, 2, 512, 256, 64)
    assert call(shape=s2, causal=1, n=sage.sage_workspace_bytes(s2, 3, 128, 64)) == 2   # causal with N > M


def test_host_call_checks_everything_before_its_first_copy(sage):
    """sage_attn_host validates all of its own and its two calls' arguments
    before it enqueues anything (a copy attempted here, without a GPU, would
    surface as SAGE_ERR_CUDA instead of the codes below)."""
    s = sage.Shape(1, 2, 2, 256, 256, 64)
    need = sage.lib.sage_host_buffer_bytes(C.byref(s), 0, 128, 64)
    assert need > sage.sage_workspace_bytes(s, 0, 128, 64)
    h = C.c_void_p(1 << 20)                  # host pointers, never dereferenced
    dbuf = C.c_void_p(1 << 30)               # 1024-aligned, never dereferenced
    f = sage.lib.sage_attn_host

    def call(shape=s, causal=0, scale=0.125, mode=0, flags=1, bq=128, bk=64, q=h, k=h, v=h, o=h, buf=dbuf,
             n=need):
        return f(C.byref(shape), causal, scale, mode, flags, bq, bk, q, k, v, o, buf, n, None)
    assert call(q=None) == 1 and call(o=None) == 1 and call(buf=None) == 1
    assert call(buf=C.c_void_p((1 << 30) + 512)) == 1                    # device buffer alignment
    assert call(n=need - 1) == 3                                          # too small
    assert call(flags=64) == 1                                            # unknown flag
    assert call(mode=2, bk=128, flags=1 | 0x10, n=sage.lib.sage_host_buffer_bytes(C.byref(s), 2, 128, 128)) == 2
    # (per-token Q scales are for the INT8 / FP8 modes)
    assert call(scale=0.0) == 1 and call(scale=float("nan")) == 1
    s2 = sage.Shape(1, 2, 2, 512, 256, 64)
    need2 = sage.lib.sage_host_buffer_bytes(C.byref(s2), 0, 128, 64)
    assert call(shape=s2, causal=1, n=need2) == 2                         # causal with N > M
    need4 = sage.lib.sage_host_buffer_bytes(C.byref(s), 2, 128, 64)
    assert need4 > 0 and call(mode=2, bk=64, n=need4) == 2                # NVFP4 attention takes 128-key tiles
    assert call(bq=64) == 2 and call(mode=7) == 1                         # layout conditions
    assert sage.lib.sage_host_buffer_bytes(C.byref(sage.Shape(1, 3, 2, 256, 256, 64)), 0, 128, 64) == 0


def _host_chunks(B, Hq, Hkv, N):
    """The host call's chunking: about 512 query blocks per chunk, 6 to 24
    chunks, whole kv-heads of one batch element each."""
    target = max(6, min(24, B * Hq * ((N + 127) // 128) // 512))
    per_b = max(1, min(Hkv, (target + B - 1) // B))
    return [(b, k * Hkv // per_b, (k + 1) * Hkv // per_b) for b in range(B) for k in range(per_b)
            if (k + 1) * Hkv // per_b > k * Hkv // per_b]


@pytest.mark.parametrize("B,Hq,Hkv,N,M,d,mode,bk", [
    (2, 48, 48, 17776, 17776, 64, 0, 128),   # the video shape: 24 chunks of 4 kv-heads
    (4, 32, 32, 4096, 4096, 128, 0, 128),    # 8 chunks
    (1, 32, 8, 4096, 65536, 128, 0, 128),    # the minimum of 6 chunks, uneven head counts
    (1, 2, 2, 256, 256, 64, 2, 128),         # fewer kv-heads than chunks
])
def test_host_buffer_follows_the_chunking_rule(sage, B, Hq, Hkv, N, M, d, mode, bk):
    """sage_host_buffer_bytes = the status word + q, k, v, o + two workspace
    slots, each the largest chunk's workspace, rounded up to 1024 bytes."""
    G = Hq // Hkv
    al = lambda n: (n + 1023) // 1024 * 1024
    slot = max(sage.sage_workspace_bytes(sage.Shape(1, (g1 - g0) * G, g1 - g0, N, M, d), mode, 128, bk)
               for _, g0, g1 in _host_chunks(B, Hq, Hkv, N))
    io = al(B * Hq * N * d * 2) * 2 + al(B * Hkv * M * d * 2) * 2
    got = sage.lib.sage_host_buffer_bytes(C.byref(sage.Shape(B, Hq, Hkv, N, M, d)), mode, 128, bk)
    assert got == 1024 + io + 2 * al(slot)


def test_status_strings(sage):
    for code in range(7):
        assert sage.sage_status_str(code)
    assert "range" in sage.sage_status_str(4)


def test_package_has_no_fallback():
    src = open(os.path.join(ROOT, "bit_quantized_attention_gb300", "_binding.py")).read()
    assert "raise ImportError" in src
    for bad in ("import oracle", "from oracle", "sage_oracle"):
        assert bad not in src


def test_sagebwd_layout(sage):
    """Mode 3 (SageBwd forward): fp16 V codes, per-block V scales, per-row
    log-sum-exp; 64-key tiles only."""
    shp = (2, 8, 4, 1000, 1500, 128)
    s = sage.Shape(*shp)
    L = sage.sage_workspace_layout(s, 3, 128, 64).as_dict()
    B, Hq, Hkv, N, M, d = shp
    assert L["dv"] - L["vhat"] >= B * Hkv * d * L["M_pad"] * 2
    assert L["lse"] - L["dvb"] >= B * Hkv * L["Tn"] * 4
    assert L["total"] - L["lse"] >= B * Hq * L["N_pad"] * 4
    assert all(L[k] % 1024 == 0 for k in ("dqt", "dvb", "lse", "total"))
    assert sage.sage_workspace_bytes(s, 3, 128, 128) == 0
    with pytest.raises(sage.SageError):
        sage.sage_workspace_layout(s, 3, 128, 128)


def _cu(vals):
    return (C.c_int * len(vals))(*vals)


def test_varlen_workspace_plan(sage):
    """Packed sequences: the batched layout of the longest runs plus the tables;
    invalid cu_seqlens give 0 bytes."""
    f = sage.lib.sage_varlen_workspace_bytes
    cq, ck = [0, 100, 100, 400, 401], [0, 150, 160, 700, 702]
    n = f(4, _cu(cq), _cu(ck), 8, 2, 128, 0, 128, 64)
    padded = sage.sage_workspace_bytes(sage.Shape(4, 8, 2, 300, 540, 128), 0, 128, 64)
    assert n > padded and n % 1024 == 0
    assert n - padded < 1 << 16                     # the tables: 4 sequences, a few dozen work items
    assert f(4, _cu(cq), _cu(ck), 8, 2, 128, 2, 128, 128) > 0           # NVFP4 too
    assert f(2, _cu([1, 5, 9]), _cu([0, 5, 9]), 8, 2, 128, 0, 128, 64) == 0   # must start at 0
    assert f(2, _cu([0, 5, 4]), _cu([0, 5, 9]), 8, 2, 128, 0, 128, 64) == 0   # decreasing
    assert f(2, _cu([0, 5, 9]), _cu([0, 5, 5]), 8, 2, 128, 0, 128, 64) == 0   # queries without keys
    assert f(2, _cu([0, 0, 0]), _cu([0, 5, 5]), 8, 2, 128, 0, 128, 64) == 0   # no queries at all
    assert f(2, _cu([0, 5, 9]), _cu([0, 5, 9]), 3, 2, 128, 0, 128, 64) == 0   # Hq % Hkv
    assert f(2, _cu([0, 5, 9]), _cu([0, 5, 9]), 8, 2, 128, 3, 128, 128) == 0  # SageBwd: 64-key tiles


def test_varlen_call_checks_before_any_copy(sage):
    """Argument errors come back before the tables' copy (which would fail here
    without a GPU as SAGE_ERR_CUDA)."""
    g = sage.lib.sage_attn_varlen
    cq, ck = _cu([0, 64, 100]), _cu([0, 64, 200])
    need = sage.lib.sage_varlen_workspace_bytes(2, cq, ck, 4, 2, 64, 0, 128, 64)
    p = C.c_void_p(1 << 20)          # never dereferenced
    ws = C.c_void_p(1 << 30)

    def call(cqa=cq, cka=ck, causal=0, scale=0.125, mode=0, flags=1, bk=64, q=p, k=p, v=p, w=ws, n=need, o=p):
        return g(2, cqa, cka, 4, 2, 64, causal, scale, mode, flags, 128, bk, q, k, v, w, n, o, None)
    assert call(q=None) == 1 and call(o=None) == 1 and call(w=None) == 1
    assert call(w=C.c_void_p((1 << 30) + 512)) == 1          # workspace alignment
    assert call(q=C.c_void_p((1 << 20) + 8)) == 1            # 16-byte alignment of the inputs
    assert call(n=need - 1) == 3
    assert call(flags=64) == 1 and call(scale=0.0) == 1
    assert call(mode=2, bk=64) == 2                          # NVFP4 attention takes 128-key tiles
    assert call(cka=_cu([0, 32, 200]), causal=1) == 2        # causal: sequence 0 has 64 queries, 32 keys
