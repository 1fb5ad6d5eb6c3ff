"""GPU parity of the attention kernels with the softmax warpgroups taking
whole key tiles in turn (SAGE_PINGPONG=1), with and without Q smoothing, in
the INT8 / FP8 and NVFP4 modes: the same bar as the split schedule against the
oracle."""
import pytest

import oracle
from test_gpu_attn import ATTN_SMALL, FP4_ATTN_SMALL, check, gpu_attention
from test_gpu_quantize import _small
from workload import make_inputs

pytestmark = pytest.mark.gpu

CASES = [c for c in ATTN_SMALL if c.mode in (0, 1)] + [
    _small("ping_causal_many_d128", B=2, Hq=24, Hkv=8, N=600, M=700, causal=True, flags=1, d=128, bk=128),
    _small("ping_fp8_d64_bk64_ragged", mode=1, N=300, M=450, causal=True, flags=5, d=64, bk=64),
] + FP4_ATTN_SMALL


@pytest.fixture(scope="module")
def sage():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_quantized_attention_gb300 as s
    return s


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_pingpong_matches_oracle(sage, cfg, monkeypatch):
    monkeypatch.setenv("SAGE_PINGPONG", "1")
    q, k, v = make_inputs(cfg)
    o = gpu_attention(sage, cfg, q, k, v)
    rows = oracle.all_rows((cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d))
    check(cfg, o.reshape(-1, cfg.d), q, k, v, rows)
