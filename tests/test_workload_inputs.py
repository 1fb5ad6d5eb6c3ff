"""The seeded synthetic inputs: reproducible bits, bf16 rounding that agrees with
the oracle's own encoder, the workloads' shapes, and the structure each recipe
promises (checked on scaled-down copies of the configs)."""
import numpy as np
import pytest

import oracle
from workload import CONFIGS, make_inputs
from workload.gen import bf16_bits, make_qkv_float


def test_same_seed_same_bits_other_seed_other_bits():
    cfg = CONFIGS["tiny"]
    a = [bf16_bits(t) for t in make_inputs(cfg)]
    b = [bf16_bits(t) for t in make_inputs(cfg)]
    c = [bf16_bits(t) for t in make_inputs(cfg.with_(seed=cfg.seed + 1))]
    for x, y, z in zip(a, b, c):
        assert np.array_equal(x, y)
        assert not np.array_equal(x, z)
    assert not np.array_equal(a[0][:, :, :, :], a[1][:, :, :, :])  # Q and K come from different streams


def test_bf16_rounding_matches_the_oracle_encoder():
    cfg = CONFIGS["tiny"].with_(N=64, M=96)
    floats = make_qkv_float(cfg)
    for f, t in zip(floats, make_inputs(cfg)):
        want = oracle.bf16_encode(f.astype(np.float64).reshape(-1))
        assert np.array_equal(bf16_bits(t).reshape(-1), want)


@pytest.mark.parametrize("name,shape", [
    ("tiny", (1, 2, 2, 256, 256, 64, False)),
    ("llm_prefill", (4, 32, 32, 4096, 4096, 128, True)),
    ("video", (2, 48, 48, 17776, 17776, 64, False)),
    ("chunked_gqa", (1, 32, 8, 4096, 65536, 128, True)),
    ("nvfp4", (2, 24, 24, 8192, 8192, 128, False)),
])
def test_workload_shapes(name, shape):
    c = CONFIGS[name]
    assert (c.B, c.Hq, c.Hkv, c.N, c.M, c.d, c.causal) == shape


def _channel_means(x):
    return x.astype(np.float64).mean(axis=2)  # over tokens, per (b, h, channel)


def test_tiny_fixed_channels_shifted():
    q, k, v = make_qkv_float(CONFIGS["tiny"])
    m = _channel_means(k)[0, 0]
    assert abs(m[3] - 10.0) < 0.5 and abs(m[17] - 10.0) < 0.5
    others = np.delete(m, [3, 17])
    assert np.abs(others).max() < 0.5


def test_llm_outlier_channels_and_offsets():
    cfg = CONFIGS["llm_prefill"].with_(B=1, Hq=4, Hkv=4, N=256, M=512)
    q, k, v = make_qkv_float(cfg)
    m = _channel_means(k)                            # offsets N(0, 3^2) + 4 outlier channels at +20
    big = (m > 12.0).sum(axis=-1)
    assert np.all(big >= 4)
    outl = np.sort(np.argsort(-m, axis=-1)[..., :4], axis=-1)
    assert np.all(outl == outl[0, 0])                # the same four channels in every head
    spread = np.delete(m[0, 0], outl[0, 0]).std()
    assert 1.5 < spread < 5.0                        # the per-channel offsets, std about 3
    assert abs(_channel_means(q)).max() < 0.5         # Q has no offsets in this recipe


def test_video_q_block_shifts_and_ragged_tail():
    full = CONFIGS["video"]
    assert full.N % full.q_block_len == 48           # the last 64-token block holds 48 tokens
    cfg = full.with_(B=1, Hq=2, Hkv=2, N=64 * 5 + 48, M=256)
    q, k, v = make_qkv_float(cfg)
    qb = q[0, 0, :5 * 64].reshape(5, 64, -1).astype(np.float64).mean(axis=1)  # block means per channel
    # per-(64-token block, channel) shifts N(0, 1) on top of per-channel offsets: blocks differ
    assert np.std(qb - qb.mean(axis=0), axis=0).mean() > 0.5
    assert abs(_channel_means(v)).max() > 1.0        # V carries a channel bias N(0, 2^2)


def test_chunked_v_student_t_clipped():
    cfg = CONFIGS["chunked_gqa"].with_(N=128, M=4096, Hq=4, Hkv=1)
    q, k, v = make_qkv_float(cfg)
    x = v.astype(np.float64).reshape(-1)
    assert np.abs(x).max() <= 64.0
    kurt = ((x - x.mean()) ** 4).mean() / x.var() ** 2
    assert kurt > 4.0                                 # heavier tails than a Gaussian (3)
