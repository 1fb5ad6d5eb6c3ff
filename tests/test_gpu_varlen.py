"""GPU parity of packed-sequence attention (sage_attn_varlen) against the
oracle's per-sequence composition.

Each sequence's codes and scales must be bit-identical to the oracle
quantizing that sequence alone (they sit at its batch index of the padded
workspace); the output must meet the same bar as the batched modes against the
oracle's packed output (max|dO| <= 1e-2 max|O|, mean relative L1 <= 2e-3), and
the SageBwd forward's lse must agree within 2e-4.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import fold_neg_zero_e4m3, output_metrics, read_workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sage():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_quantized_attention_gb300 as s
    return s


def _packed(rng, total, H, d, off):
    x = rng.standard_normal((total, H, d)) + off * rng.standard_normal((1, H, d))
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)


def _cu(lens):
    return [0] + list(np.cumsum(lens).astype(int))


CASES = [
    # name, mode, flags, causal, Hq, Hkv, d, bk, query lengths, key lengths
    ("int8_ragged", 0, 1, False, 4, 2, 64, 64, [200, 0, 1, 333, 64], [130, 9, 1, 700, 64]),
    ("int8_causal_smooth", 0, 7, True, 4, 1, 128, 128, [128, 37, 300], [128, 500, 300]),
    # a one-query sequence and a 129-query one: Q blocks of one row (zero smoothed codes)
    ("int8_smooth_q_one_query", 0, 3, False, 2, 2, 64, 128, [1, 129, 200], [50, 300, 129]),
    ("fp8_gqa", 1, 3, False, 8, 2, 128, 128, [90, 256, 17], [1000, 40, 17]),
    ("sagebwd_causal", 3, 1, True, 4, 2, 64, 64, [150, 65, 1], [150, 300, 2]),
    ("int8_per_token_q", 0, 1 | 0x10, True, 2, 2, 128, 64, [129, 400], [129, 401]),
    ("nvfp4_causal_smooth", 2, 3, True, 4, 2, 128, 128, [200, 1, 300], [260, 1, 900]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_varlen_matches_oracle(sage, case):
    name, mode, flags, causal, Hq, Hkv, d, bk, lq, lk = case
    rng = np.random.default_rng(len(name))
    cq, ck = _cu(lq), _cu(lk)
    q, k, v = _packed(rng, cq[-1], Hq, d, 2.0), _packed(rng, ck[-1], Hkv, d, 3.0), _packed(rng, ck[-1], Hkv, d, 1.0)
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda")
    o, ws = sage.sage_attn_varlen(q.to(dev), k.to(dev), v.to(dev), cq, ck, causal, scale, mode, flags, 128, bk)
    torch.cuda.synchronize()
    assert sage.sage_read_status(ws) == (0, 0)
    ref, ref_lse, quants = oracle.attn_varlen(mode, flags, 128, bk, causal, scale, q, k, v, cq, ck)
    got = o.float().cpu().numpy()
    m = output_metrics(got, oracle.bf16_round(ref))
    assert m["max_rel"] <= 1e-2 and m["rel_l1"] <= 2e-3, m
    if mode == 2:
        return  # NVFP4 codes sit in scale-factor atoms; the batched tests check them
    # codes and scales, sequence by sequence, at its batch index of the padded workspace
    w = read_workspace(ws, mode)
    for s, qz in enumerate(quants):
        if qz is None:
            continue
        n, mk = lq[s], lk[s]
        fold = fold_neg_zero_e4m3 if mode == 1 else (lambda c: c)  # E4M3 +-0 both encode 0
        assert np.array_equal(fold(w["qc"][s, :, :n]), fold(qz.qc[0])), s
        assert np.array_equal(fold(w["kc"][s, :, :mk]), fold(qz.kc[0])), s
        tn = -(-mk // bk)
        assert np.array_equal(w["dk"][s, :, :tn].view(np.uint32), qz.dk[0].view(np.uint32)), s
        assert np.array_equal(w["kbar"][s].view(np.uint32), qz.kbar[0].view(np.uint32)), s
        tm = -(-n // 128)
        assert np.array_equal(w["qbar"][s, :, :tm].view(np.uint32), qz.qbar[0].view(np.uint32)), s
    if mode == 3:
        lse = sage.sage_lse(ws).cpu().numpy()
        for s in range(len(lq)):
            if lq[s]:
                got_l = lse[s, :, :lq[s]].T   # [n, Hq], the oracle's packed order
                assert np.abs(got_l - ref_lse[cq[s]:cq[s + 1]]).max() <= 2e-4 * max(1.0, np.abs(ref_lse).max())
