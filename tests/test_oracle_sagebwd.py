"""Pins for the oracle's SageBwd forward mode and for the softmax statistics it
returns (CPU only).

SageBwd forward (SageAttention3 summary, "SageBwd Forward Pass"): INT8 per-block
Q and K (max/127, as in the INT8 mode), INT8 per-block V over each bk-token
block, and INT8 P~ with one scale per row and key tile,
s_P = exp(rowmax S_ij - m_ij) / 127, so that the tile's largest P~ gets code 127.

- V codes and scales: restated here with numpy binary32 arithmetic, block by block.
- One dominant key per row: the output is that key's V row exactly (s_P times
  the code 127 gives back P~, s_V of the key's own block, the rescale alpha
  removes the earlier tiles).
- Two keys: in one tile the second gets the code round(127 e^-delta) while l
  keeps the unquantized e^-delta, a closed form; in two tiles each key is its
  tile's maximum, so the result is the textbook one.
- lse = m + ln(l): the log-sum-exp of the scores actually used, in every mode.
"""
import math

import numpy as np
import pytest

from test_oracle_attention import bf16_tensor, f64, rand_qkv, textbook

MODE = 3


def _orc_mode(orc):
    assert orc.MODE_SAGEBWD_I8 == MODE
    return MODE


def textbook_lse(q, k, causal, scale):
    """log sum_j exp(s_ij) over the visible keys, fp64; GQA and masks as textbook()."""
    B, Hq, N, d = q.shape
    Hkv, M = k.shape[1], k.shape[2]
    k = np.repeat(k, Hq // Hkv, axis=1)
    s = np.einsum("bhnd,bhmd->bhnm", q, k) * scale
    if causal:
        i = np.arange(N)[:, None]
        j = np.arange(M)[None, :]
        s = np.where(j <= i + (M - N), s, -np.inf)
    mx = s.max(-1, keepdims=True)
    return mx[..., 0] + np.log(np.exp(s - mx).sum(-1))


def _all(orc, shape, mode, flags, bq, bk, causal, scale, q, k, v):
    qz = orc.quantize(shape, mode, flags & 0xFF, bq, bk, q, k, v)
    B, Hq, _, N, _, d = shape
    out, lse = orc.attn_rows_lse(shape, mode, flags, bq, bk, causal, scale, q, k, v, qz,
                                 np.arange(B * Hq * N))
    return out.reshape(B, Hq, N, d), lse.reshape(B, Hq, N), qz


# ---------------------------------------------------------------- quantizers
def test_qk_codes_and_scales_are_the_int8_modes(orc):
    """Q and K take the same per-block INT8 quantizer in both modes."""
    shape = (2, 4, 2, 70, 90, 32)
    q, k, v = rand_qkv(*shape, seed=5, koff=3.0, qoff=2.0, voff=1.0)
    flags = orc.SMOOTH_K | orc.SMOOTH_Q | orc.SMOOTH_V
    a = orc.quantize(shape, 0, flags, 32, 16, q, k, v)
    b = orc.quantize(shape, _orc_mode(orc), flags, 32, 16, q, k, v)
    for f in ("qc", "dq", "qbar", "kc", "dk", "kbar", "vm"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    assert not b.dv.any() and b.dvb.all()


@pytest.mark.parametrize("smooth_v", [False, True])
def test_v_per_block_int8_codes(orc, smooth_v):
    """s_V,j = fl(max|V'_j| / 127) over the bk tokens of block j (ragged last
    block) and all channels; code = clamp(rint(fl(V' / s_V,j))), V' = fl(V - V_m)."""
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 2, 20, 70, 32, 16, 16
    q, k, v = rand_qkv(B, Hq, Hkv, N, M, d, seed=9, voff=3.0)
    flags = orc.SMOOTH_K | (orc.SMOOTH_V if smooth_v else 0)
    qz = orc.quantize((B, Hq, Hkv, N, M, d), _orc_mode(orc), flags, bq, bk, q, k, v)
    assert bool(qz.vm.any()) == smooth_v
    g = f64(v).astype(np.float32) - qz.vm[:, :, None, :]
    codes = qz.vc.view(np.int8)
    Tn = -(-M // bk)
    assert qz.dvb.shape == (B, Hkv, Tn)
    for j in range(Tn):
        blk = g[:, :, j * bk:(j + 1) * bk, :]
        s = (np.abs(blk).max(axis=(2, 3)) / np.float32(127)).astype(np.float32)
        assert np.array_equal(qz.dvb[:, :, j], s), j
        want = np.clip(np.rint(blk / s[:, :, None, None]), -127, 127).astype(np.int8)
        assert np.array_equal(codes[:, :, j * bk:(j + 1) * bk, :], want), j


# ---------------------------------------------------------------- exact-code inputs
def _q_one_channel(B, Hq, N, d):
    """Q = 127/16 on channel 0, 0 elsewhere: per-block scale 1/16, codes exact."""
    qf = np.zeros((B, Hq, N, d))
    qf[..., 0] = 127 * 2.0 ** -4
    return qf


def _k_from_channel0(rng, c, B, Hkv, d, bk):
    """K[t, 0] = c_t / 16 (|c_t| <= 127) and one +-127/16 per bk-block on channel 1,
    which Q does not read: every block scale is 1/16 and the codes are exact."""
    M = c.size
    kf = np.zeros((B, Hkv, M, d))
    kf[..., 0] = c * 2.0 ** -4
    for t0 in range(0, M, bk):
        kf[:, :, t0, 1] = 127 * 2.0 ** -4 * rng.choice([-1, 1])
    return kf


def _v_exact(rng, B, Hkv, M, d, bk):
    """V block j = integers in [-127, 127] times 2^-(3 + j % 3), one +-127 per
    block at a random place: s_V,j = 2^-(3 + j % 3) and every code is exact."""
    c = rng.integers(-127, 128, size=(B, Hkv, M, d)).astype(np.float64)
    for j, t0 in enumerate(range(0, M, bk)):
        t1 = min(t0 + bk, M)
        t = rng.integers(t0, t1)
        c[:, :, t, rng.integers(0, d)] = 127 * rng.choice([-1, 1])
        c[:, :, t0:t1] *= 2.0 ** -(3 + j % 3)
    return c


@pytest.mark.parametrize("causal", [False, True])
def test_dominant_key_gives_its_v_row(orc, causal):
    """c_t = -127 + 3t, scale 30: consecutive keys differ by 44.6 in S, so each
    row's last visible key holds all the weight (the next one gets
    127 e^-44.6 -> code 0, and adds ~4e-20 to l).  The output is that key's V row:
    s_P 127 = P~ of the tile maximum, times s_V of that key's block."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 1, 40, 70, 16, 16, 16
    c = -127 + 3 * np.arange(M)
    qf, kf, vf = _q_one_channel(B, Hq, N, d), _k_from_channel0(rng, c, B, Hkv, d, bk), _v_exact(rng, B, Hkv, M, d, bk)
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    assert np.array_equal(f64(k), kf) and np.array_equal(f64(v), vf)
    got, _, qz = _all(orc, (B, Hq, Hkv, N, M, d), _orc_mode(orc), 0, bq, bk, causal, 30.0, q, k, v)
    assert np.array_equal(qz.dvb[0, 0], 2.0 ** -(3 + np.arange(-(-M // bk)) % 3))
    last = np.arange(N) + (M - N) if causal else np.full(N, M - 1)
    want = vf[:, np.zeros(Hq, int)][:, :, last, :]
    assert np.allclose(got, want, rtol=1e-13, atol=0)


def _two_key_case(orc, ka, kb_, scale):
    rng = np.random.default_rng(17)
    B, Hq, Hkv, N, M, d, bq, bk = 1, 1, 1, 16, 48, 16, 16, 16
    c = rng.integers(-127, 61, size=M)          # the rest at least 66 units below: weight < e^-60
    c[ka], c[kb_] = 127, 126
    qf, kf, vf = _q_one_channel(B, Hq, N, d), _k_from_channel0(rng, c, B, Hkv, d, bk), _v_exact(rng, B, Hkv, M, d, bk)
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    got, _, _ = _all(orc, (B, Hq, Hkv, N, M, d), _orc_mode(orc), 0, bq, bk, False, scale, q, k, v)
    delta = 127.0 / 256.0 * scale               # S_a - S_b: one unit of c
    return got[0, 0], vf[0, 0, ka], vf[0, 0, kb_], delta


def test_two_keys_in_one_tile_closed_form(orc):
    """Keys a, b in one tile, S_b = S_a - delta with 127 e^-delta = p = 50.3:
    P^_a = 127, P^_b = round(p) = 50, l = 1 + p/127 (unquantized), so every row
    is (127 v_a + 50 v_b) / (127 + p)."""
    scale = math.log(127.0 / 50.3) / (127.0 / 256.0)
    out, va, vb, delta = _two_key_case(orc, 5, 9, scale)
    p = 127.0 * math.exp(-delta)
    assert round(p) == 50 and abs(p - 50.3) < 1e-9
    want = (127.0 * va + 50.0 * vb) / (127.0 + p)
    assert np.allclose(out, want[None, :], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("ka,kb_", [(5, 20), (36, 3)])
def test_two_keys_in_two_tiles_are_exact(orc, ka, kb_):
    """Each key is the maximum of its own tile, so both get code 127 with their
    own s_P: the result is textbook (v_a + e^-delta v_b) / (1 + e^-delta), in
    either tile order."""
    scale = math.log(127.0 / 50.3) / (127.0 / 256.0)
    out, va, vb, delta = _two_key_case(orc, ka, kb_, scale)
    w = math.exp(-delta)
    want = (va + w * vb) / (1.0 + w)
    assert np.allclose(out, want[None, :], rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- softmax statistics
LSE_SHAPES = [
    # B, Hq, Hkv, N, M, d, bq, bk, causal
    (1, 2, 1, 17, 17, 16, 16, 16, True),
    (2, 4, 2, 64, 130, 64, 128, 64, False),
    (1, 2, 2, 17, 64, 16, 16, 16, True),
    (1, 4, 4, 64, 17, 16, 16, 64, False),
]


@pytest.mark.parametrize("shape", LSE_SHAPES)
@pytest.mark.parametrize("flags", [0, 1, 1 | 2 | 4])
@pytest.mark.parametrize("mode", [0, 2, MODE])
def test_lse_identity_quantizers(orc, shape, flags, mode):
    """With identity quantizers S = Q (K - k_bar)^T s (dS puts q_bar back), so
    lse is the log-sum-exp of those scores over the visible keys."""
    B, Hq, Hkv, N, M, d, bq, bk, causal = shape
    q, k, v = rand_qkv(B, Hq, Hkv, N, M, d, seed=N + 3 * M, koff=3.0, qoff=2.0, voff=2.0)
    scale = 1.0 / math.sqrt(d)
    _, lse, qz = _all(orc, (B, Hq, Hkv, N, M, d), mode, flags | orc.EXACT_QK | orc.EXACT_PV, bq, bk,
                      causal, scale, q, k, v)
    ks = f64(k) - qz.kbar.astype(np.float64)[:, :, None, :]
    assert np.allclose(lse, textbook_lse(f64(q), ks, causal, scale), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("mode", [0, MODE])
@pytest.mark.parametrize("causal", [False, True])
def test_lse_sums_unquantized_p(orc, mode, causal):
    """Q, K with exact INT8 codes, P~ and V quantized: l sums the unquantized P~,
    so lse is still the textbook log-sum-exp of the exact scores."""
    rng = np.random.default_rng(29 + mode)
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 1, 40, 80, 32, 16, 16
    c = rng.integers(-127, 128, size=(B, Hq, N, d)).astype(np.float64)
    c[:, :, ::bq, 0] = 127
    qf = c * 2.0 ** -4
    c = rng.integers(-127, 128, size=(B, Hkv, M, d)).astype(np.float64)
    c[:, :, ::bk, 0] = -127
    kf = c * 2.0 ** -4
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(rng.standard_normal((B, Hkv, M, d)))
    _, lse, _ = _all(orc, (B, Hq, Hkv, N, M, d), mode, 0, bq, bk, causal, 0.05, q, k, v)
    assert np.allclose(lse, textbook_lse(qf, kf, causal, 0.05), rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- accuracy
@pytest.mark.parametrize("causal", [False, True])
def test_accuracy_against_fp64(orc, causal):
    """Gaussian inputs with K channel offsets (smoothed): per-token INT8 P~ and
    per-block INT8 V stay close to fp64 attention (measured here: 1 - cos about
    2e-4, relative L1 about 0.019 non-causal)."""
    shape = (1, 4, 2, 256, 256, 64)
    q, k, v = rand_qkv(*shape, seed=41, koff=4.0)
    ref = orc.attn_exact_rows(shape, causal, 0.125, q, k, v, np.arange(4 * 256)).reshape(1, 4, 256, 64)
    got, _, _ = _all(orc, shape, MODE, orc.SMOOTH_K, 128, 64, causal, 0.125, q, k, v)
    cos = (got * ref).sum() / math.sqrt((got * got).sum() * (ref * ref).sum())
    rel_l1 = np.abs(got - ref).sum() / np.abs(ref).sum()
    assert cos > 0.9995 and rel_l1 < 0.025, (cos, rel_l1)
