"""Accuracy side of the method's switches, measured with the oracle against
fp64 attention on Gaussian inputs with channel offsets (the accuracy half of
the pages' ablation tables; the timing half is bench.py's).  Each pin states
the direction the pages report and a margin that the measured values (in the
docstrings, 1 - cosine) clear comfortably.  CPU only."""
import math

import numpy as np
import pytest

from test_oracle_attention import rand_qkv

SHAPE = (1, 4, 2, 256, 256, 64)
ROWS = np.arange(4 * 256)


def err(orc, mode, flags, **offsets):
    q, k, v = rand_qkv(*SHAPE, seed=41, **offsets)
    ref = orc.attn_exact_rows(SHAPE, False, 0.125, q, k, v, ROWS)
    bk = 128 if mode == 2 else 64
    qz = orc.quantize(SHAPE, mode, flags & 0xFF, 128, bk, q, k, v)
    got = orc.attn_rows(SHAPE, mode, flags, 128, bk, False, 0.125, q, k, v, qz, ROWS)
    return 1.0 - (got * ref).sum() / math.sqrt((got * got).sum() * (ref * ref).sum())


@pytest.mark.parametrize("mode,ratio", [(0, 0.95), (1, 0.7), (2, 0.8)])
def test_q_smoothing_helps_with_q_offsets(orc, mode, ratio):
    """Q channel offsets N(0, 4^2): INT8 6.8e-4 -> 5.7e-4, E4M3 5.1e-3 -> 2.9e-3,
    NVFP4 7.2e-2 -> 4.8e-2 with Q smoothing (dS restores q_bar)."""
    assert err(orc, mode, 1 | 2, koff=3.0, qoff=4.0) < ratio * err(orc, mode, 1, koff=3.0, qoff=4.0)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_v_smoothing_helps_with_v_offsets(orc, mode):
    """V channel offsets N(0, 4^2): 7.1e-6 -> 4.6e-7 (INT8 Q/K), 7.3e-6 -> 9.2e-7
    (E4M3), 1.5e-4 -> 1.3e-5 (NVFP4): the per-channel FP8 / per-block FP4 V
    scales no longer spend their range on the mean."""
    assert err(orc, mode, 1 | 4, koff=3.0, voff=4.0) < 0.3 * err(orc, mode, 1, koff=3.0, voff=4.0)


@pytest.mark.parametrize("mode", [0, 1])
def test_per_token_q_no_worse_than_per_block(orc, mode):
    """Per-token Q scales (a finer granularity): 6.75e-4 -> 6.61e-4 (INT8),
    2.03e-3 -> 1.92e-3 (E4M3) on these inputs."""
    assert err(orc, mode, 1 | 0x10, koff=3.0, qoff=1.0) <= err(orc, mode, 1, koff=3.0, qoff=1.0)


def test_sagebwd_int8_pv_against_fp8_pv(orc):
    """The SageBwd forward's per-row INT8 P~ and per-block INT8 V against the
    static-1/448 E4M3 P~ and per-channel E4M3 V of the INT8 mode (same INT8
    Q/K): 7.2e-4 -> 1.9e-4 (relative L1 3.8 % -> 1.9 %), the uniform INT8 grid
    the SageBwd page prefers over FP8."""
    assert err(orc, 3, 1, koff=3.0) < 0.5 * err(orc, 0, 1, koff=3.0)


@pytest.mark.parametrize("mode,factor", [(0, 3.0), (2, 10.0)])
def test_k_smoothing_ablation(orc, mode, factor):
    """The pages' case for smoothing K: with channel offsets on K (shared by all
    tokens) the per-block quantizers spend their range on the offsets.  Here,
    offsets N(0, 10^2): INT8 1 - cos 2.9e-3 unsmoothed against 7.1e-4 smoothed,
    NVFP4 0.33 against 0.019; without offsets smoothing changes nothing."""
    assert err(orc, mode, 0, koff=10.0) > factor * err(orc, mode, orc.SMOOTH_K, koff=10.0)
    assert abs(err(orc, mode, 0) - err(orc, mode, orc.SMOOTH_K)) < 0.1 * err(orc, mode, orc.SMOOTH_K)
