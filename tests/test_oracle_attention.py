"""Pins for the oracle's attention (CPU only).

- With every quantizer replaced by identity, the tiled online-softmax path must
  equal textbook softmax(Q K^T s) V computed here with numpy on the full score
  matrix (tiling, running max / sum, rescale, masks, GQA head map, ragged tiles,
  and the smoothing identities: K-mean invariance, S = gamma(Q)gamma(K)^T + dS
  with a row-constant remainder, P~ V_m = V_m).
- With inputs the quantizers represent exactly, the quantized Q/K path must
  equal textbook attention (dequantization scales and constants).
- With constant scores (P~ = 1 everywhere) and exactly representable V, the
  quantized P~ path must equal textbook attention (the 448 scale, delta_V,
  the two-level 448*6 constant).
- Loose statistical pins from the "Quantization for Attention" simulator.
"""
import math

import numpy as np
import pytest
import torch

from conftest import golden


def textbook(q, k, v, causal, scale):
    """softmax(q k^T * scale) v over the full score matrix, fp64; q [B,Hq,N,d],
    k, v [B,Hkv,M,d]; query head h reads kv head h // (Hq/Hkv); causal masks are
    bottom-right aligned (key j visible to query i iff j <= i + M - N)."""
    B, Hq, N, d = q.shape
    Hkv, M = k.shape[1], k.shape[2]
    k = np.repeat(k, Hq // Hkv, axis=1)
    v = np.repeat(v, Hq // Hkv, axis=1)
    s = np.einsum("bhnd,bhmd->bhnm", q, k) * scale
    if causal:
        i = np.arange(N)[:, None]
        j = np.arange(M)[None, :]
        s = np.where(j <= i + (M - N), s, -np.inf)
    s = s - s.max(-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(-1, keepdims=True)
    return np.einsum("bhnm,bhmd->bhnd", p, v)


def bf16_tensor(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64).numpy()


def run_oracle(orc, shape, mode, flags, bq, bk, causal, scale, q, k, v):
    qz = orc.quantize(shape, mode, flags & 0xFF, bq, bk, q, k, v)
    B, Hq, _, N, _, d = shape
    rows = np.arange(B * Hq * N)
    out = orc.attn_rows(shape, mode, flags, bq, bk, causal, scale, q, k, v, qz, rows)
    return out.reshape(B, Hq, N, d), qz


def rand_qkv(B, Hq, Hkv, N, M, d, seed, koff=0.0, qoff=0.0, voff=0.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, Hq, N, d)) + qoff * r.standard_normal((B, Hq, 1, d))
    k = r.standard_normal((B, Hkv, M, d)) + koff * r.standard_normal((B, Hkv, 1, d))
    v = r.standard_normal((B, Hkv, M, d)) + voff * r.standard_normal((B, Hkv, 1, d))
    return bf16_tensor(q), bf16_tensor(k), bf16_tensor(v)


SHAPES = [
    # B, Hq, Hkv, N, M, d, bq, bk, causal
    (1, 1, 1, 1, 1, 16, 16, 16, False),
    (1, 2, 1, 17, 17, 16, 16, 16, True),
    (2, 4, 2, 64, 130, 64, 128, 64, False),
    (1, 4, 1, 130, 130, 64, 64, 16, True),
    (1, 2, 2, 17, 64, 16, 16, 16, True),      # N < M, bottom-right causal
    (1, 4, 4, 64, 17, 16, 16, 64, False),     # one ragged key tile
    (1, 2, 1, 130, 64, 64, 128, 16, False),   # ragged query block
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("flags", [0, 1, 1 | 2 | 4])
@pytest.mark.parametrize("mode", [0, 2])
def test_identity_quantizers_equal_textbook(orc, shape, flags, mode):
    B, Hq, Hkv, N, M, d, bq, bk, causal = shape
    q, k, v = rand_qkv(B, Hq, Hkv, N, M, d, seed=N * 31 + M, koff=3.0, qoff=2.0, voff=2.0)
    scale = 1.0 / math.sqrt(d)
    got, _ = run_oracle(orc, (B, Hq, Hkv, N, M, d), mode, flags | orc.EXACT_QK | orc.EXACT_PV,
                        bq, bk, causal, scale, q, k, v)
    ref = textbook(f64(q), f64(k), f64(v), causal, scale)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("shape", SHAPES[:5])
def test_exact_attention_equals_textbook(orc, shape):
    B, Hq, Hkv, N, M, d, bq, bk, causal = shape
    q, k, v = rand_qkv(B, Hq, Hkv, N, M, d, seed=7)
    rows = np.arange(B * Hq * N)
    got = orc.attn_exact_rows((B, Hq, Hkv, N, M, d), causal, 0.125, q, k, v, rows).reshape(B, Hq, N, d)
    ref = textbook(f64(q), f64(k), f64(v), causal, 0.125)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- exact Q/K codes
def _int8_exact(rng, shape, blk):
    """values c * 2^-4, integer c in [-127,127], every blk-row block holding +-127*2^-4"""
    B, H, L, d = shape
    c = rng.integers(-127, 128, size=shape).astype(np.float64)
    for t0 in range(0, L, blk):
        c[:, :, t0, 0] = 127 * rng.choice([-1, 1])
    return c * 2.0 ** -4


def _fp8_exact(rng, shape, blk, orc):
    mags = orc.e4m3_decode(np.arange(127))
    x = rng.choice(mags, size=shape) * rng.choice([-1, 1], size=shape)
    for t0 in range(0, shape[2], blk):
        x[:, :, t0, 0] = 448.0
    return x * 2.0 ** -6


def _nvfp4_exact_rows(rng, shape):
    """each 1x16 block along d: E2M1 values times 2^e with one element at 6*2^e"""
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    x = rng.choice(mags, size=shape) * rng.choice([-1, 1], size=shape)
    B, H, L, d = shape
    e = rng.integers(-5, 3, size=(B, H, L, d // 16))
    x = x.reshape(B, H, L, d // 16, 16)
    x[..., 3] = 6.0
    x = x * (2.0 ** e)[..., None]
    return x.reshape(shape)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_exact_qk_codes_reproduce_textbook(orc, mode, causal):
    rng = np.random.default_rng(3 + mode)
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 1, 40, 80, 32, 16, 16
    if mode == 0:
        qf = _int8_exact(rng, (B, Hq, N, d), bq)
        kf = _int8_exact(rng, (B, Hkv, M, d), bk)
    elif mode == 1:
        qf = _fp8_exact(rng, (B, Hq, N, d), bq, orc)
        kf = _fp8_exact(rng, (B, Hkv, M, d), bk, orc)
    else:
        qf = _nvfp4_exact_rows(rng, (B, Hq, N, d))
        kf = _nvfp4_exact_rows(rng, (B, Hkv, M, d))
    vf = rng.standard_normal((B, Hkv, M, d))
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    assert np.array_equal(f64(q), qf) and np.array_equal(f64(k), kf)
    scale = 0.02
    got, _ = run_oracle(orc, (B, Hq, Hkv, N, M, d), mode, orc.EXACT_PV, bq, bk, causal, scale, q, k, v)
    ref = textbook(qf, kf, f64(v), causal, scale)
    assert np.allclose(got, ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- V smoothing through the codes
@pytest.mark.parametrize("causal", [False, True])
def test_v_smoothing_exact_codes_reproduce_textbook(orc, causal):
    """V = (base + deviations) 2^e per channel, the deviations in cancelling
    token pairs from {0, +-256, +-320, +-384, +-448} (exact in E4M3) and the base
    a multiple of 64 (so every value is exact in bf16): V_m is the base exactly,
    delta_V = 2^e, the codes of V' = V - V_m are the deviations.  With constant
    scores (P~ = 1, P^ = 448 exactly) the output O / l * delta_V / 448 + V_m is
    the mean of the visible V rows: textbook attention ("Optional Smoothing of
    V", SageAttention2 summary §3.4)."""
    rng = np.random.default_rng(91)
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 2, 48, 96, 32, 16, 32
    qf = rng.standard_normal((B, Hq, N, d))
    kf = np.broadcast_to(rng.standard_normal((B, Hkv, 1, d)), (B, Hkv, M, d)).copy()
    half = rng.choice([0.0, 256.0, 320.0, 384.0, -256.0, -320.0, -384.0], size=(B, Hkv, M // 2, d))
    half[:, :, 3, :] = 448.0
    dev = np.concatenate([half, -half], axis=2)        # token t and t + M/2 cancel
    base = rng.choice([-448.0, -320.0, -64.0, 0.0, 64.0, 192.0, 448.0], size=(B, Hkv, 1, d))
    e = 2.0 ** rng.integers(-6, 0, size=(B, Hkv, 1, d))
    vf = (base + dev) * e
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    assert np.array_equal(f64(v), vf)
    got, qz = run_oracle(orc, (B, Hq, Hkv, N, M, d), 0, orc.SMOOTH_K | orc.SMOOTH_V, bq, bk, causal, 0.1,
                         q, k, v)
    assert np.array_equal(qz.vm.astype(np.float64), (base * e)[:, :, 0, :])
    assert np.array_equal(qz.dv.astype(np.float64), e[:, :, 0, :])
    assert np.array_equal(orc.e4m3_decode(qz.vc), dev)
    ref = textbook(qf, kf, vf, causal, 0.1)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- running max as the P~ reference
def test_p_quantized_against_the_running_max(orc):
    """m_ij = max(m_i,j-1, rowmax S_ij) and P~_ij = exp(S_ij - m_ij)
    (SageAttention2 summary §3.4): a tile whose own maximum lies below the
    running one quantizes P~ relative to the running maximum.  One query; tile 0
    holds the row maximum (S = 8 at key 0, S = -64 elsewhere), tile 1 sits at
    S = 4.875: its P~ = e^-3.125 becomes e4m3(448 e^-3.125) / 448 = 20 / 448.
    Exact S, V exactly representable in FP8 per channel, l over unquantized P~."""
    B, Hq, Hkv, N, M, d, bk = 1, 1, 1, 1, 32, 16, 16
    qf = np.zeros((B, Hq, N, d))
    qf[..., 0] = 1.0
    kf = np.zeros((B, Hkv, M, d))
    kf[0, 0, 0, 0] = 8.0
    kf[0, 0, 1:16, 0] = -64.0
    kf[0, 0, 16:, 0] = 4.875
    rng = np.random.default_rng(9)
    mags = orc.e4m3_decode(np.arange(127))
    vf = rng.choice(mags, size=(B, Hkv, M, d)) * rng.choice([-1, 1], size=(B, Hkv, M, d))
    vf[0, 0, 7, :] = 448.0                           # per-channel absmax 448: delta_V = 1, V^ = V
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    assert np.array_equal(f64(k), kf) and np.array_equal(f64(v), vf)
    got, _ = run_oracle(orc, (B, Hq, Hkv, N, M, d), 0, orc.EXACT_QK, 128, bk, False, 1.0, q, k, v)
    p1 = np.exp(4.875 - 8.0)
    ph1 = orc.e4m3_decode(orc.e4m3_encode(np.array([448.0 * p1])))[0] / 448.0
    assert ph1 == 20.0 / 448.0
    l = 1.0 + 16.0 * p1
    want = (vf[0, 0, 0] + ph1 * vf[0, 0, 16:].sum(axis=0)) / l
    assert np.allclose(got.reshape(-1), want, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- Q smoothing through the codes
@pytest.mark.parametrize("causal", [False, True])
def test_q_smoothing_exact_codes_reproduce_textbook(orc, causal):
    """Q rows = a per-block base (the block's exact mean) plus +-pairs of INT8
    codes times 2^-4: q_bar is the base exactly, gamma(Q) quantizes exactly
    (delta_Q = 2^-4), and with exact K codes and unquantized P~V the smoothed
    path S = (deq gamma(Q) + q_bar) deq(K)^T is textbook attention on the bf16
    inputs (SageAttention2 summary §3.4, smoothing Q with the dS correction)."""
    rng = np.random.default_rng(81)
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 1, 32, 48, 32, 16, 16
    c = np.zeros((B, Hq, N, d))
    for t0 in range(0, N, bq):                         # every block: rows r and r + bq/2 cancel
        half = rng.integers(-126, 127, size=(B, Hq, bq // 2, d)).astype(np.float64)
        half[:, :, 0, 0] = 127.0                       # the block's absmax: delta_Q = 2^-4
        c[:, :, t0:t0 + bq // 2] = half
        c[:, :, t0 + bq // 2:t0 + bq] = -half
    base = rng.integers(-64, 65, size=(B, Hq, N // bq, 1, d)).astype(np.float64)
    base = np.broadcast_to(base, (B, Hq, N // bq, bq, d)).reshape(B, Hq, N, d)
    qf = (base + c) * 2.0 ** -4
    kf = _int8_exact(rng, (B, Hkv, M, d), bk)
    vf = rng.standard_normal((B, Hkv, M, d))
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    assert np.array_equal(f64(q), qf) and np.array_equal(f64(k), kf)
    got, qz = run_oracle(orc, (B, Hq, Hkv, N, M, d), 0, orc.SMOOTH_Q | orc.EXACT_PV, bq, bk, causal, 0.02,
                         q, k, v)
    assert np.array_equal(qz.qbar.astype(np.float64), (base * 2.0 ** -4)[:, :, ::bq, :])
    assert np.array_equal(qz.qc.view(np.int8).astype(np.float64), c)
    ref = textbook(qf, kf, f64(v), causal, 0.02)
    assert np.allclose(got, ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- per-token Q scales
def _rows_exact(rng, shape, mode, orc):
    """each row: codes times its own power of two, the row's absmax at 127 (INT8)
    or 448 (E4M3) times it, so fl(absmax / 127 or 448) is the power itself"""
    B, H, L, d = shape
    if mode == 0:
        c = rng.integers(-127, 128, size=shape).astype(np.float64)
        c[..., 0] = 127 * rng.choice([-1, 1], size=(B, H, L))
    else:
        mags = orc.e4m3_decode(np.arange(127))
        c = rng.choice(mags, size=shape) * rng.choice([-1, 1], size=shape)
        c[..., 0] = 448.0
    e = rng.integers(-12, -2, size=(B, H, L, 1))
    return c, 2.0 ** e


@pytest.mark.parametrize("mode", [0, 1])
def test_per_token_q_scales_are_the_row_scales(orc, mode):
    """With Q_PER_TOKEN each row gets fl(absmax/127) (INT8) or fl(absmax/448)
    (E4M3) of its own and codes with it: rows built as codes times a power of two
    come back exactly.  Per block, the rows with the smaller powers share the
    block's largest scale and lose bits: their codes differ."""
    rng = np.random.default_rng(41 + mode)
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 1, 40, 32, 32, 16, 16
    c, s = _rows_exact(rng, (B, Hq, N, d), mode, orc)
    q = bf16_tensor(c * s)
    k = bf16_tensor(rng.standard_normal((B, Hkv, M, d)))
    v = bf16_tensor(rng.standard_normal((B, Hkv, M, d)))
    assert np.array_equal(f64(q), c * s)
    shape = (B, Hq, Hkv, N, M, d)
    tok = orc.quantize(shape, mode, orc.Q_PER_TOKEN, bq, bk, q, k, v)
    assert np.array_equal(tok.dqt.astype(np.float64), s[..., 0])
    codes = tok.qc.view(np.int8).astype(np.float64) if mode == 0 else orc.e4m3_decode(tok.qc)
    assert np.array_equal(codes, c)
    blk = orc.quantize(shape, mode, 0, bq, bk, q, k, v)
    bcodes = blk.qc.view(np.int8).astype(np.float64) if mode == 0 else orc.e4m3_decode(blk.qc)
    assert not np.array_equal(bcodes, c)


@pytest.mark.parametrize("causal", [False, True])
def test_per_token_q_exact_codes_reproduce_textbook(orc, causal):
    """Per-token Q codes that are exact, exact K codes per block and unquantized
    P~V: the oracle's attention is textbook attention on the bf16 inputs (each
    row of S dequantized with its own Q scale)."""
    rng = np.random.default_rng(61)
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 1, 40, 80, 32, 16, 16
    c, s = _rows_exact(rng, (B, Hq, N, d), 0, orc)
    qf = c * s
    kf = _int8_exact(rng, (B, Hkv, M, d), bk)
    vf = rng.standard_normal((B, Hkv, M, d))
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    got, qz = run_oracle(orc, (B, Hq, Hkv, N, M, d), 0, orc.Q_PER_TOKEN | orc.EXACT_PV, bq, bk, causal, 0.02,
                         q, k, v)
    assert np.array_equal(qz.dqt.astype(np.float64), s[..., 0])
    ref = textbook(qf, kf, f64(v), causal, 0.02)
    assert np.allclose(got, ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- exact P~ path
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_constant_scores_exact_p_path(orc, mode, causal):
    """All keys equal -> K - mean(K) = 0 -> S = 0 -> P~ = 1: e4m3(448*1) = 448
    (FP8 modes) or s_P1 = 1/2688, s_P2 = 448, code 6 (NVFP4); with V exactly
    representable the quantized output equals the mean of the visible V rows."""
    rng = np.random.default_rng(21 + mode)
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 2, 48, 96, 32, 16, 32
    qf = rng.standard_normal((B, Hq, N, d))
    kf = np.broadcast_to(rng.standard_normal((B, Hkv, 1, d)), (B, Hkv, M, d)).copy()
    if mode in (0, 1):
        mags = orc.e4m3_decode(np.arange(127))
        vf = rng.choice(mags, size=(B, Hkv, M, d)) * rng.choice([-1, 1], size=(B, Hkv, M, d))
        vf[:, :, 5, :] = 448.0                              # per-channel absmax 448*2^e
        vf = vf * (2.0 ** rng.integers(-8, 0, size=(B, Hkv, 1, d)))
    else:
        mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
        vf = rng.choice(mags, size=(B, Hkv, M, d)) * rng.choice([-1, 1], size=(B, Hkv, M, d))
        vf = vf.reshape(B, Hkv, M // 16, 16, d)
        vf[:, :, :, 2, :] = 6.0                             # each 16-token block max 6*2^e
        vf = (vf * (2.0 ** rng.integers(-4, 2, size=(B, Hkv, M // 16, 1, d)))).reshape(B, Hkv, M, d)
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    assert np.array_equal(f64(v), vf)
    got, qz = run_oracle(orc, (B, Hq, Hkv, N, M, d), mode, orc.SMOOTH_K, bq, bk, causal, 0.1, q, k, v)
    assert not qz.kc.any()
    ref = textbook(qf, kf, vf, causal, 0.1)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- direct P~ (NVFP4 ablation)
@pytest.mark.parametrize("causal", [False, True])
def test_direct_p_constant_scores_closed_form(orc, causal):
    """Constant scores make P~ = 1 for every visible key.  Quantized directly,
    each 16-key block gets s = e4m3(1/6) and code e2m1(1/s), so every P~ becomes
    e2m1(1/s) * s (6 * 0.171875 = 1.03125), while l sums the unquantized 1s: the
    output is that factor times the mean of the visible V rows (V exactly
    representable), where the two-level path returns the mean itself."""
    rng = np.random.default_rng(71)
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 2, 48, 96, 32, 16, 32
    qf = rng.standard_normal((B, Hq, N, d))
    kf = np.broadcast_to(rng.standard_normal((B, Hkv, 1, d)), (B, Hkv, M, d)).copy()
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    vf = rng.choice(mags, size=(B, Hkv, M, d)) * rng.choice([-1, 1], size=(B, Hkv, M, d))
    vf = vf.reshape(B, Hkv, M // 16, 16, d)
    vf[:, :, :, 2, :] = 6.0
    vf = (vf * (2.0 ** rng.integers(-4, 2, size=(B, Hkv, M // 16, 1, d)))).reshape(B, Hkv, M, d)
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    s1 = orc.e4m3_decode(orc.e4m3_encode(np.array([1.0 / 6.0])))[0]
    factor = orc.e2m1_decode(orc.e2m1_encode(np.array([1.0 / s1])))[0] * s1
    assert factor == 1.03125
    shape = (B, Hq, Hkv, N, M, d)
    got, _ = run_oracle(orc, shape, 2, orc.SMOOTH_K | orc.P_DIRECT, bq, bk, causal, 0.1, q, k, v)
    two, _ = run_oracle(orc, shape, 2, orc.SMOOTH_K, bq, bk, causal, 0.1, q, k, v)
    ref = textbook(qf, kf, vf, causal, 0.1)
    assert np.allclose(two, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(got, factor * ref, rtol=1e-12, atol=1e-12)


def test_direct_p_no_effect_in_fp8_modes(orc):
    """The FP8 modes quantize P~ directly already (static 1/448): the switch
    leaves them unchanged."""
    B, Hq, Hkv, N, M, d = 1, 2, 1, 64, 96, 64
    q, k, v = rand_qkv(B, Hq, Hkv, N, M, d, seed=5, koff=3.0)
    for mode in (0, 1):
        a, _ = run_oracle(orc, (B, Hq, Hkv, N, M, d), mode, orc.SMOOTH_K, 128, 64, True, 0.125, q, k, v)
        b, _ = run_oracle(orc, (B, Hq, Hkv, N, M, d), mode, orc.SMOOTH_K | orc.P_DIRECT, 128, 64, True, 0.125,
                          q, k, v)
        assert np.array_equal(a, b)


def test_direct_p_small_block_scale_underflows(orc):
    """Why the pages scale P~ in two levels (SageAttention3 summary §3.4): P~
    lies in [0, 1], so a 16-key block whose largest P~ is small gets a direct
    E4M3 scale max/6 below E4M3's smallest subnormal (2^-9) and rounds to zero:
    the block vanishes from the numerator while l, which sums the unquantized
    P~, still counts it.  One query against two key blocks (exact Q/K):
    block A at S = 0 (P~ = 1, quantized to 6 * e4m3(1/6) = 1.03125 each) and
    block B at S = -6.9375 (P~ = e^-6.9375, about 9.7e-4, scale about 1.6e-4).
    Directly quantized, the output is 1.03125 * sum_A V / (16 + 16 e^-6.9375)
    with V exactly representable; the two-level form keeps block B."""
    B, Hq, Hkv, N, M, d = 1, 1, 1, 1, 32, 16
    qf = np.zeros((B, Hq, N, d))
    qf[..., 0] = 1.0
    kf = np.zeros((B, Hkv, M, d))
    kf[0, 0, 16:, 0] = -55.5                          # S = -55.5 / 8 on block B
    rng = np.random.default_rng(5)
    mags = np.array([0.5, 1, 1.5, 2, 3, 4, 6])
    vf = rng.choice(mags, size=(B, Hkv, M, d)) * rng.choice([-1, 1], size=(B, Hkv, M, d))
    vf[0, 0, 3, :] = 6.0                              # each 16-token block's max is 6 (V exact in NVFP4)
    vf[0, 0, 19, :] = 6.0
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    assert np.array_equal(f64(k), kf) and np.array_equal(f64(v), vf)
    sB = -55.5 / 8.0
    small = np.array([np.exp(sB) / 6.0])
    assert orc.e4m3_decode(orc.e4m3_encode(small))[0] == 0.0 and small[0] < 2.0 ** -9
    shape = (B, Hq, Hkv, N, M, d)
    direct, _ = run_oracle(orc, shape, 2, orc.EXACT_QK | orc.P_DIRECT, 128, 32, False, 1.0 / 8.0, q, k, v)
    two, _ = run_oracle(orc, shape, 2, orc.EXACT_QK, 128, 32, False, 1.0 / 8.0, q, k, v)
    l = 16.0 + 16.0 * np.exp(sB)
    want = 1.03125 * vf[0, 0, :16].sum(axis=0) / l
    assert np.allclose(direct.reshape(-1), want, rtol=1e-12, atol=1e-12)
    exact = textbook(qf, kf, vf, False, 1.0 / 8.0).reshape(-1)
    # the two-level form keeps block B: it lands much closer to exact attention
    assert np.abs(two.reshape(-1) - exact).max() < 0.2 * np.abs(direct.reshape(-1) - exact).max()


# ---------------------------------------------------------------- accuracy sanity
# INT8 Q/K (the mode of the INT8/FP8 workloads) reaches 0.999.  The extra E4M3
# Q/K mode carries 3 mantissa bits per operand (about 0.9987 here).  NVFP4 on
# i.i.d. Gaussian inputs, whose attention rows are nearly flat, lands near 0.98
# (the pages' 99.5 % is measured on real video-model tensors).
@pytest.mark.parametrize("mode,min_cos", [(0, 0.999), (1, 0.998), (2, 0.975)])
def test_quantized_accuracy_against_fp64(orc, mode, min_cos):
    B, Hq, Hkv, N, M, d = 1, 2, 1, 200, 300, 64
    q, k, v = rand_qkv(B, Hq, Hkv, N, M, d, seed=99, koff=3.0)
    got, _ = run_oracle(orc, (B, Hq, Hkv, N, M, d), mode, orc.SMOOTH_K, 128, 64, True, 0.125, q, k, v)
    ref = textbook(f64(q), f64(k), f64(v), True, 0.125)
    cos = (got * ref).sum() / np.sqrt((got ** 2).sum() * (ref ** 2).sum())
    assert cos >= min_cos


def test_nvfp4_reaches_099_on_peaked_rows(orc):
    """The spec NVFP4 bar (cosine >= 0.99 against fp64 attention) where
    the method can reach it: each query copies one key row of its head (plus
    noise), so its row is peaked on that key, as attention rows of trained
    models are; on the same shape with i.i.d. Gaussian queries (nearly flat
    rows over 1024 keys) the method stays below 0.99."""
    from workload import CONFIGS, make_inputs

    def cos_of(cfg):
        q, k, v = make_inputs(cfg)
        shape = (cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d)
        qz = orc.quantize(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, q, k, v)
        rows = orc.all_rows(shape)[::8]
        got = orc.attn_rows(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, cfg.causal, cfg.sm_scale, q, k, v, qz, rows)
        ref = orc.attn_exact_rows(shape, cfg.causal, cfg.sm_scale, q, k, v, rows)
        return float((got * ref).sum() / np.sqrt((got ** 2).sum() * (ref ** 2).sum()))

    base = CONFIGS["nvfp4"].with_(B=1, Hq=2, Hkv=2, N=256, M=1024, bk=128)
    assert cos_of(base.with_(q_from_k_noise=0.5)) >= 0.99
    assert cos_of(base) < 0.99


def test_quantize_rejects_out_of_range(orc):
    q, k, v = rand_qkv(1, 1, 1, 16, 16, 16, seed=1)
    k[0, 0, 3, 3] = 70000.0
    with pytest.raises(orc.OracleError):
        orc.quantize((1, 1, 1, 16, 16, 16), 0, 1, 16, 16, q, k, v)


@pytest.mark.slow
def test_simulator_statistics(orc):
    """K smoothing roughly halves the relative L1 of per-block INT8 Q/K
    (about 2.5 % -> 1.3 %) on the simulator's synthetic recipe."""
    g = golden("p5_simulator.txt")
    B, H, N, d = 1, 8, 1024, 128
    r = np.random.default_rng(0)
    qf, kf, vf = (r.standard_normal((B, H, N, d)) for _ in range(3))
    kf[..., 7] += 8.0
    q, k, v = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf)
    shape = (B, H, H, N, N, d)
    heads = [0, 3]
    rows = np.concatenate([np.arange(h * N, (h + 1) * N) for h in heads])
    ref = orc.attn_exact_rows(shape, False, 1 / math.sqrt(d), q, k, v, rows)
    rel = {}
    for flags in (0, orc.SMOOTH_K):
        qz = orc.quantize(shape, 0, flags, 64, 64, q, k, v)
        out = orc.parallel_attn_rows(shape, 0, flags | orc.EXACT_PV, 64, 64, False, 1 / math.sqrt(d),
                                     q, k, v, qz, rows)
        rel[flags] = np.abs(out - ref).sum() / np.abs(ref).sum()
    assert 0.5 * g["rel_l1_no_smooth"] < rel[0] < 2.0 * g["rel_l1_no_smooth"]
    assert 0.5 * g["rel_l1_smooth_k"] < rel[orc.SMOOTH_K] < 2.0 * g["rel_l1_smooth_k"]
    assert rel[orc.SMOOTH_K] < 0.75 * rel[0]

