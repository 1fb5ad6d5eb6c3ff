"""GPU pre-pass parity: codes, scales and means bit-identical to the oracle.

Small cases run whole; the full-size workloads are checked on sampled heads
(every statistic is per (batch, head), so the oracle quantizing one kv-head
and its query heads reproduces exactly what the full tensors give there).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import compare_codes, compare_codes_fp4, read_workspace, read_workspace_fp4
from workload import CONFIGS, make_inputs
from workload.configs import Config

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sage():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_quantized_attention_gb300 as s
    return s


def _small(name, **kw):
    base = dict(name=name, B=1, Hq=2, Hkv=2, N=256, M=256, d=64, causal=False, sm_scale=0.125, mode=0,
                flags=1, bq=128, bk=64, seed=11, k_offset_std=3.0, q_offset_std=1.0, v_bias_std=1.0)
    base.update(kw)
    return Config(**base)


SMALL = [
    CONFIGS["tiny"],
    _small("ragged_all_smooth", N=200, M=333, flags=7),
    _small("fp8_qk", mode=1, flags=7, N=130, M=70),
    _small("gqa_d128", B=2, Hq=4, Hkv=2, N=300, M=520, d=128, flags=3, bk=128),
    _small("d128_bk64_i8", d=128, N=129, M=1000, flags=5, k_outliers=3, k_outlier_shift=20.0),
    _small("fp8_d128", d=128, mode=1, N=64, M=64, flags=0),
    _small("single_token", N=1, M=1, flags=7),
    # per-token Q scales (one per query row, q_bar still per block)
    _small("per_token_q_i8", N=200, M=333, flags=7 | 0x10),
    _small("per_token_q_fp8_d128", mode=1, N=130, M=300, d=128, bk=128, flags=3 | 0x10),
    _small("per_token_q_i8_d128", d=128, N=257, M=129, flags=1 | 0x10, q_offset_std=4.0),
]


def _run(sage, cfg, q, k, v):
    dev = torch.device("cuda")
    ws = sage.sage_quantize_qkv(q.to(dev), k.to(dev), v.to(dev), cfg.mode, cfg.flags, cfg.bq, cfg.bk)
    torch.cuda.synchronize()
    assert sage.sage_read_status(ws) == (0, 0)
    return ws


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
def test_quantize_bit_exact_small(sage, cfg):
    q, k, v = make_inputs(cfg)
    ws = _run(sage, cfg, q, k, v)
    got = read_workspace(ws, cfg.mode)
    ref = oracle.quantize((cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d), cfg.mode, cfg.flags, cfg.bq, cfg.bk,
                          q, k, v)
    res = compare_codes(got, ref, cfg.mode, cfg.flags)
    assert all(res.values()), res


def test_quantize_twice_identical(sage):
    cfg = SMALL[1]
    q, k, v = make_inputs(cfg)
    a = read_workspace(_run(sage, cfg, q, k, v), cfg.mode)
    b = read_workspace(_run(sage, cfg, q, k, v), cfg.mode)
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_range_error_reported(sage):
    cfg = SMALL[0]
    q, k, v = make_inputs(cfg)
    k[0, 1, 5, 7] = 70000.0
    dev = torch.device("cuda")
    ws = sage.sage_quantize_qkv(q.to(dev), k.to(dev), v.to(dev), cfg.mode, cfg.flags, cfg.bq, cfg.bk)
    torch.cuda.synchronize()
    code, site = sage.sage_read_status(ws)
    assert code == 4 and site == 1
    v[0, 0, 0, 0] = float("nan")
    k[0, 1, 5, 7] = 1.0
    ws = sage.sage_quantize_qkv(q.to(dev), k.to(dev), v.to(dev), cfg.mode, cfg.flags, cfg.bq, cfg.bk)
    torch.cuda.synchronize()
    assert sage.sage_read_status(ws) == (4, 2)


@pytest.mark.parametrize("name", ["llm_prefill", "video", "chunked_gqa"])
def test_quantize_bit_exact_full_size_sampled_heads(sage, name):
    cfg = CONFIGS[name]
    q, k, v = make_inputs(cfg)
    ws = _run(sage, cfg, q, k, v)
    got = read_workspace(ws, cfg.mode)
    G = cfg.Hq // cfg.Hkv
    for b, g in {(0, 0), (cfg.B - 1, cfg.Hkv - 1)}:
        hs = slice(g * G, (g + 1) * G)
        qs, ks, vs = q[b:b + 1, hs].contiguous(), k[b:b + 1, g:g + 1].contiguous(), v[b:b + 1, g:g + 1].contiguous()
        ref = oracle.quantize((1, G, 1, cfg.N, cfg.M, cfg.d), cfg.mode, cfg.flags, cfg.bq, cfg.bk, qs, ks, vs)
        sub = {key: (val[b:b + 1, hs] if key in ("qc", "dq", "qbar") else
                     (val[b:b + 1, g:g + 1] if key in ("kc", "dk", "kbar", "vc", "dv", "vm") else val))
               for key, val in got.items()}
        res = compare_codes(sub, ref, cfg.mode, cfg.flags)
        assert all(res.values()), (b, g, res)


FP4_SMALL = [
    _small("fp4_tiny", mode=2, flags=1, bk=128),
    _small("fp4_ragged_all_smooth", mode=2, flags=7, N=200, M=333, bk=128),
    _small("fp4_d128_gqa", mode=2, flags=3, B=2, Hq=4, Hkv=2, N=130, M=515, d=128, bk=128,
           k_outliers=2, k_outlier_shift=20.0),
    _small("fp4_single_token", mode=2, flags=5, N=1, M=1, bk=128),
]


@pytest.mark.parametrize("cfg", FP4_SMALL, ids=[c.name for c in FP4_SMALL])
def test_quantize_fp4_bit_exact_small(sage, cfg):
    q, k, v = make_inputs(cfg)
    ws = _run(sage, cfg, q, k, v)
    got = read_workspace_fp4(ws)
    ref = oracle.quantize((cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d), cfg.mode, cfg.flags, cfg.bq, cfg.bk,
                          q, k, v)
    res = compare_codes_fp4(got, ref)
    assert all(res.values()), res


def test_quantize_fp4_bit_exact_full_size_sampled_heads(sage):
    cfg = CONFIGS["nvfp4"].with_(bk=128)
    q, k, v = make_inputs(cfg)
    ws = _run(sage, cfg, q, k, v)
    got = read_workspace_fp4(ws)
    G = cfg.Hq // cfg.Hkv
    for b, g in {(0, 0), (cfg.B - 1, cfg.Hkv - 1)}:
        hs = slice(g * G, (g + 1) * G)
        qs, ks, vs = q[b:b + 1, hs].contiguous(), k[b:b + 1, g:g + 1].contiguous(), v[b:b + 1, g:g + 1].contiguous()
        ref = oracle.quantize((1, G, 1, cfg.N, cfg.M, cfg.d), cfg.mode, cfg.flags, cfg.bq, cfg.bk, qs, ks, vs)
        sub = {key: (val[b:b + 1, hs] if key in ("qc", "qs", "qbar") else val[b:b + 1, g:g + 1])
               for key, val in got.items()}
        res = compare_codes_fp4(sub, ref)
        assert all(res.values()), (b, g, res)
