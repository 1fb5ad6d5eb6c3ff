"""GPU attention parity against the oracle (INT8 / FP8 / NVFP4 modes).

Bar (per element, the method's output in bf16): max|dO| <= 1e-2 * max|O| and
mean relative L1 <= 2e-3 against the oracle's output rounded to bf16, on the
same quantized workspace; and cosine >= 0.999 against unquantized fp64
attention for INT8 Q/K (0.998 for the E4M3 Q/K mode, whose 3-bit mantissas
cost that much on these inputs in the oracle itself).  NVFP4 keeps the same
bar against the oracle; against fp64 attention its cosine must reach 0.975 and
fall no more than 2e-3 below the oracle's own (E2M1 with 16-element blocks
loses that much on Gaussian inputs in the oracle too).
Small cases compare every row; the full-size workloads compare sampled rows:
the first and last query blocks of two heads plus scattered rows.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import output_metrics
from test_gpu_quantize import FP4_SMALL, SMALL, _small
from workload import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu

ATTN_SMALL = SMALL + [
    _small("causal_square", N=384, M=384, causal=True, flags=1),
    _small("causal_bottom_right", N=200, M=777, causal=True, flags=3, d=128, bk=128),
    _small("causal_gqa_ragged", B=1, Hq=4, Hkv=1, N=131, M=4000, causal=True, flags=7, d=128),
    _small("long_keys", N=128, M=8192, flags=1, d=64, bk=128),
    _small("fp8_causal", mode=1, N=256, M=300, causal=True, flags=7, d=128),
    # more work items than SMs: every persistent CTA walks several items of
    # different lengths, so the dS stream and the rings cross item boundaries
    _small("many_items_smooth", B=2, Hq=48, Hkv=48, N=600, M=700, causal=True, flags=7, d=64, bk=128),
    _small("many_items_fp8_gqa_d128", mode=1, B=1, Hq=40, Hkv=8, N=520, M=520, flags=3, d=128, bk=128),
    _small("per_token_q_causal_many", B=2, Hq=24, Hkv=8, N=600, M=700, causal=True, flags=7 | 0x10, d=128,
           bk=128),
    _small("per_token_q_fp8_d64_bk64", mode=1, N=300, M=450, flags=1 | 0x10, d=64, bk=64),
    # Q block 2 holds one row: its smoothed Q is zero, so is its scale, and
    # its scores are the dS term alone
    _small("smooth_q_one_row_tail", N=257, M=300, flags=3, d=64, bk=128, q_offset_std=2.0),
    _small("smooth_q_per_token_d64", N=300, M=520, causal=True, flags=3 | 0x10, d=64, bk=128, q_offset_std=2.0),
]

FP4_ATTN_SMALL = FP4_SMALL + [
    _small("fp4_causal_square", mode=2, N=384, M=384, causal=True, flags=1, d=128, bk=128),
    _small("fp4_causal_bottom_right", mode=2, N=200, M=777, causal=True, flags=3, d=128, bk=128),
    _small("fp4_causal_gqa_ragged", mode=2, B=1, Hq=4, Hkv=1, N=131, M=2000, causal=True, flags=7, d=64,
           bk=128),
    _small("fp4_long_keys", mode=2, N=128, M=4096, flags=1, d=128, bk=128),
    # direct-P~ ablation: phi on P~ itself, no level-1 scale
    _small("fp4_direct_p", mode=2, N=256, M=500, flags=1 | 8, d=128, bk=128),
    _small("fp4_direct_p_causal_smooth", mode=2, N=200, M=777, causal=True, flags=3 | 8, d=64, bk=128),
]


@pytest.fixture(scope="module")
def sage():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_quantized_attention_gb300 as s
    return s


def gpu_attention(sage, cfg, q, k, v):
    dev = torch.device("cuda")
    ws = sage.sage_quantize_qkv(q.to(dev), k.to(dev), v.to(dev), cfg.mode, cfg.flags, cfg.bq, cfg.bk)
    o = sage.sage_attn_fwd(ws, cfg.causal, cfg.sm_scale)
    torch.cuda.synchronize()
    assert sage.sage_read_status(ws) == (0, 0)
    return o.float().cpu().numpy()


def check(cfg, got_rows, q, k, v, rows, threads=None):
    shape = (cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d)
    qz = oracle.quantize(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, q, k, v)
    ref = oracle.parallel_attn_rows(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, cfg.causal, cfg.sm_scale,
                                    q, k, v, qz, rows, threads=threads)
    exact = oracle.attn_exact_rows(shape, cfg.causal, cfg.sm_scale, q, k, v, rows) if len(rows) <= 4096 else None
    m = output_metrics(got_rows, oracle.bf16_round(ref))
    assert m["max_rel"] <= 1e-2, m
    assert m["rel_l1"] <= 2e-3, m
    if exact is not None:
        e = output_metrics(got_rows, exact)
        o = output_metrics(ref, exact)
        bar = {0: 0.999, 1: 0.998, 2: 0.975, 3: 0.999}[cfg.mode]
        assert e["cos"] >= bar, (e, o)
        if cfg.mode == 2:
            assert e["cos"] >= o["cos"] - 2e-3, (e, o)
    return m


@pytest.mark.parametrize("cfg", ATTN_SMALL, ids=[c.name for c in ATTN_SMALL])
def test_attention_matches_oracle_small(sage, cfg):
    q, k, v = make_inputs(cfg)
    o = gpu_attention(sage, cfg, q, k, v)
    rows = oracle.all_rows((cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d))
    check(cfg, o.reshape(-1, cfg.d), q, k, v, rows)


@pytest.mark.parametrize("cfg", FP4_ATTN_SMALL, ids=[c.name for c in FP4_ATTN_SMALL])
def test_attention_fp4_matches_oracle_small(sage, cfg):
    q, k, v = make_inputs(cfg)
    o = gpu_attention(sage, cfg, q, k, v)
    rows = oracle.all_rows((cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d))
    check(cfg, o.reshape(-1, cfg.d), q, k, v, rows)


@pytest.mark.parametrize("mode", [0, 1])
def test_zero_scale_key_tile(sage, mode):
    """The last key tile (keys 256..332, ragged and causal-masked) is all zero
    without K smoothing, so its K scale is 0: every visible score of that tile
    is 0 and the masked keys must still drop out (no 0 * inf)."""
    cfg = _small("zero_tile", mode=mode, N=200, M=333, causal=True, flags=0, d=128, bk=128, k_offset_std=0.0)
    q, k, v = make_inputs(cfg)
    k[:, :, 256:, :] = 0
    o = gpu_attention(sage, cfg, q, k, v)
    assert np.isfinite(o).all()
    rows = oracle.all_rows((cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d))
    check(cfg, o.reshape(-1, cfg.d), q, k, v, rows)


@pytest.mark.parametrize("mode,bk", [(0, 128), (0, 64), (1, 128)])
def test_constant_query_block_with_q_smoothing(sage, mode, bk):
    """Q block 0 repeats one query row and block 2 holds a single row: with Q
    smoothing both blocks quantize to zero codes with a zero scale, and their
    scores are the dS term alone."""
    cfg = _small("constant_q_block", mode=mode, N=257, M=300, flags=3, d=64, bk=bk, q_offset_std=2.0)
    q, k, v = make_inputs(cfg)
    q[:, :, :128, :] = q[:, :, :1, :]
    o = gpu_attention(sage, cfg, q, k, v)
    assert np.isfinite(o).all()
    rows = oracle.all_rows((cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d))
    check(cfg, o.reshape(-1, cfg.d), q, k, v, rows)


def test_attention_deterministic(sage):
    cfg = next(c for c in ATTN_SMALL if c.name == "per_token_q_causal_many")
    q, k, v = make_inputs(cfg)
    a = gpu_attention(sage, cfg, q, k, v)
    b = gpu_attention(sage, cfg, q, k, v)
    assert np.array_equal(a, b)


def sampled_rows(cfg, rng, extra=64):
    rows = []
    for b, h in {(0, 0), (cfg.B - 1, cfg.Hq - 1)}:
        base = (b * cfg.Hq + h) * cfg.N
        rows += list(base + np.arange(0, min(128, cfg.N)))
        last = ((cfg.N - 1) // 128) * 128
        rows += list(base + np.arange(last, cfg.N))
    rows += list(rng.integers(0, cfg.B * cfg.Hq * cfg.N, size=extra))
    return np.unique(np.array(rows, dtype=np.int64))


@pytest.mark.parametrize("name,bk", [("llm_prefill", 64), ("llm_prefill", 128), ("video", 64), ("video", 128),
                                     ("chunked_gqa", 64), ("chunked_gqa", 128), ("nvfp4", 128)])
def test_attention_full_size_sampled_rows(sage, name, bk):
    cfg = CONFIGS[name].with_(bk=bk)
    q, k, v = make_inputs(cfg)
    o = gpu_attention(sage, cfg, q, k, v).reshape(-1, cfg.d)
    rows = sampled_rows(cfg, np.random.default_rng(5))
    check(cfg, o[rows], q, k, v, rows)


def test_nvfp4_peaked_rows_reach_099(sage):
    """The NVFP4 workload's shape with peaked rows (each query copies a key row
    of its head plus N(0, 0.5^2) noise): the GPU path matches the oracle (the
    bar above) and reaches cosine >= 0.99 against fp64 attention, the
    spec NVFP4 criterion, on sampled rows."""
    cfg = CONFIGS["nvfp4"].with_(bk=128, q_from_k_noise=0.5)
    q, k, v = make_inputs(cfg)
    o = gpu_attention(sage, cfg, q, k, v).reshape(-1, cfg.d)
    rows = sampled_rows(cfg, np.random.default_rng(7))
    check(cfg, o[rows], q, k, v, rows)
    exact = oracle.attn_exact_rows((cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d), cfg.causal, cfg.sm_scale, q, k, v,
                                   rows)
    assert output_metrics(o[rows], exact)["cos"] >= 0.99
