"""Pins for the oracle's SageBwd backward (CPU only).

- With every quantizer replaced by identity (unquantized Q and K, P, dO and dS),
  dQ, dK and dV equal torch autograd of fp64 softmax(Q K^T s) V: D_i, dS, the
  scale factor, the masks, the GQA sums, and the K and Q smoothing corrections.
- With inputs whose every quantized operand is exact (P = 1/2 on two equal
  dominant keys, dS and dO integers times a power of two with a +-127 in each
  block, Q and K with exact codes), the quantized backward equals autograd too:
  the INT8 divisors and the scales multiplied back.
- With an O that is not P V (D_i then leaves rowsum(dS) nonzero), identity
  quantizers give eq. 8 on the full score matrix: the smoothing corrections.
- On Gaussian inputs the quantized gradients stay close to autograd's, and
  smoothing K (with its correction from the unquantized dS) helps dQ.
"""
import math

import numpy as np
import pytest
import torch

from test_oracle_attention import bf16_tensor, f64, rand_qkv


def autograd(qf, kf, vf, dof, causal, scale):
    """fp64 torch autograd of softmax(q k^T scale) v, GQA by repetition,
    bottom-right causal; returns (dq, dk, dv, o, lse) as numpy."""
    q = torch.tensor(qf, dtype=torch.float64, requires_grad=True)
    k = torch.tensor(kf, dtype=torch.float64, requires_grad=True)
    v = torch.tensor(vf, dtype=torch.float64, requires_grad=True)
    g = q.shape[1] // k.shape[1]
    N, M = q.shape[2], k.shape[2]
    s = q @ k.repeat_interleave(g, dim=1).transpose(-1, -2) * scale
    if causal:
        vis = torch.arange(M)[None, :] <= torch.arange(N)[:, None] + (M - N)
        s = s.masked_fill(~vis, float("-inf"))
    o = torch.softmax(s, dim=-1) @ v.repeat_interleave(g, dim=1)
    o.backward(torch.tensor(dof, dtype=torch.float64))
    return (q.grad.numpy(), k.grad.numpy(), v.grad.numpy(), o.detach().numpy(),
            torch.logsumexp(s, dim=-1).detach().numpy())


def _forward(orc, shape, flags, bq, bk, causal, scale, q, k, v):
    qz = orc.quantize(shape, orc.MODE_SAGEBWD_I8, flags & 0xFF, bq, bk, q, k, v)
    B, Hq, _, N, _, d = shape
    out, lse = orc.attn_rows_lse(shape, orc.MODE_SAGEBWD_I8, flags, bq, bk, causal, scale, q, k, v, qz,
                                 orc.all_rows(shape))
    return qz, out.reshape(B, Hq, N, d), lse.reshape(B, Hq, N)


def _close(a, b, rtol):
    return np.abs(a - b).max() <= rtol * np.abs(b).max()


SHAPES = [
    # B, Hq, Hkv, N, M, d, bq, bk, causal
    (1, 1, 1, 1, 1, 16, 16, 16, False),
    (1, 2, 1, 17, 17, 16, 16, 16, True),
    (2, 4, 2, 40, 70, 32, 16, 32, False),
    (1, 4, 1, 33, 70, 16, 16, 16, True),     # N < M, bottom-right causal, ragged tiles
    (1, 2, 2, 70, 20, 16, 32, 16, False),    # ragged query and key blocks
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("flags", [0, 1, 1 | 2, 1 | 2 | 4])
def test_identity_quantizers_equal_autograd(orc, shape, flags):
    B, Hq, Hkv, N, M, d, bq, bk, causal = shape
    q, k, v = rand_qkv(B, Hq, Hkv, N, M, d, seed=N * 7 + M, koff=3.0, qoff=2.0, voff=2.0)
    dout = bf16_tensor(np.random.default_rng(N + M).standard_normal((B, Hq, N, d)))
    scale = 1.0 / math.sqrt(d)
    s = (B, Hq, Hkv, N, M, d)
    qz, _, lse = _forward(orc, s, flags | orc.EXACT_QK | orc.EXACT_PV, bq, bk, causal, scale, q, k, v)
    gq, gk, gv, o, _ = autograd(f64(q), f64(k), f64(v), f64(dout), causal, scale)
    dq, dk, dv = orc.sagebwd_backward(s, flags | orc.EXACT_QK | orc.EXACT_BWD, bq, bk, causal, scale,
                                      q, k, v, qz, o, dout, lse)
    for got, want in ((dq, gq), (dk, gk), (dv, gv)):
        assert _close(got, want, 1e-11)


@pytest.mark.parametrize("flags", [1, 1 | 2])
def test_identity_quantizers_full_matrix_with_given_o(orc, flags):
    """The backward takes D_i from the O it is given, so with an O that is not
    P V (a forward's rounded output, here a perturbed one) rowsum(dS) is not 0
    and the smoothing corrections carry weight.  Identity quantizers: dQ, dK, dV
    must equal eq. 8 on the full score matrix, P = softmax(S), dS = P o (dO V^T - D),
    D = rowsum(dO o O), dQ = dS K s, dK = dS^T Q s, dV = P^T dO (unsmoothed K, Q)."""
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 1, 40, 56, 16, 16, 16
    q, k, v = rand_qkv(B, Hq, Hkv, N, M, d, seed=23, koff=4.0, qoff=3.0)
    rng = np.random.default_rng(24)
    dout = bf16_tensor(rng.standard_normal((B, Hq, N, d)))
    scale = 0.25
    shape = (B, Hq, Hkv, N, M, d)
    qz, o, lse = _forward(orc, shape, flags | orc.EXACT_QK | orc.EXACT_PV, bq, bk, True, scale, q, k, v)
    o = o + 0.05 * rng.standard_normal(o.shape)
    dq, dk, dv = orc.sagebwd_backward(shape, flags | orc.EXACT_QK | orc.EXACT_BWD, bq, bk, True, scale,
                                      q, k, v, qz, o, dout, lse)
    qf, kf, vf, dof = f64(q), np.repeat(f64(k), Hq, axis=1), np.repeat(f64(v), Hq, axis=1), f64(dout)
    sc = np.einsum("bhnd,bhmd->bhnm", qf, kf) * scale
    sc = np.where(np.arange(M)[None, :] <= np.arange(N)[:, None] + (M - N), sc, -np.inf)
    p = np.exp(sc - sc.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    D = (dof * o).sum(-1, keepdims=True)
    ds = p * (np.einsum("bhnd,bhmd->bhnm", dof, vf) - D)
    want_q = np.einsum("bhnm,bhmd->bhnd", ds, kf) * scale
    want_k = np.einsum("bhnm,bhnd->bhmd", ds, qf).sum(1, keepdims=True) * scale
    want_v = np.einsum("bhnm,bhnd->bhmd", p, dof).sum(1, keepdims=True)
    for got, want in ((dq, want_q), (dk, want_k), (dv, want_v)):
        assert _close(got, want, 1e-11)


def _exact_case(rng, causal):
    """Q = +-127/16 on channel 0 (sign per row), K[t,0] = c_t/16 (the other
    channels integers / 16, which give dQ its values): rows of sign +
    put all weight on keys a1, a2 (c = 127), rows of sign - on b1, b2 (c = -127),
    every other key at least 3 units away (e^-44 at scale 30).  V rows a2 = a1 and
    b2 = b1 except on channel 1 (by +2 and -2), dO integers times 2^-4 with a
    +-127 on channel 1 in a + row and a - row of every query block: every
    dominant dS is +-n_i 2^-5 (n_i the row's channel-1 integer), exact on the
    INT8 grid of its tile; P = 1/2 is too."""
    B, Hq, Hkv, N, M, d, bq, bk = 1, 2, 1, 32, 48, 16, 16, 16
    a1, a2, b1, b2 = (3, 9, 20, 30) if not causal else (3, 9, 5, 12)
    sign = np.where(np.arange(N) % 2 == 0, 1.0, -1.0)
    qf = np.zeros((B, Hq, N, d))
    qf[..., 0] = 127 * 2.0 ** -4 * sign
    c = rng.integers(-124, 125, size=M).astype(np.float64)
    c[[a1, a2]], c[[b1, b2]] = 127, -127
    kf = rng.integers(-126, 127, size=(B, Hkv, M, d)) * 2.0 ** -4   # channels Q reads as 0: dQ's values
    kf[..., 0] = c * 2.0 ** -4
    for t0 in range(0, M, bk):
        kf[:, :, t0, 2] = 127 * 2.0 ** -4               # block scale 1/16 (channel 2: Q reads 0 there)
    vf = rng.integers(-100, 101, size=(B, Hkv, M, d)) * 2.0 ** -3
    vf[:, :, a2] = vf[:, :, a1]
    vf[:, :, a2, 1] += 2.0
    vf[:, :, b2] = vf[:, :, b1]
    vf[:, :, b2, 1] -= 2.0
    n = rng.integers(-126, 127, size=(B, Hq, N, d)).astype(np.float64)
    for r0 in range(0, N, bq):
        n[:, :, r0, 1], n[:, :, r0 + 1, 1] = 127, -127  # a + row and a - row per block
    dof = n * 2.0 ** -4
    return (B, Hq, Hkv, N, M, d), bq, bk, qf, kf, vf, dof


@pytest.mark.parametrize("causal", [False, True])
def test_exact_operands_quantized_equal_autograd(orc, causal):
    rng = np.random.default_rng(5 + causal)
    shape, bq, bk, qf, kf, vf, dof = _exact_case(rng, causal)
    q, k, v, dout = bf16_tensor(qf), bf16_tensor(kf), bf16_tensor(vf), bf16_tensor(dof)
    for t, x in ((q, qf), (k, kf), (v, vf), (dout, dof)):
        assert np.array_equal(f64(t), x)
    scale = 30.0
    qz, _, lse = _forward(orc, shape, 0, bq, bk, causal, scale, q, k, v)
    gq, gk, gv, o, lse_t = autograd(qf, kf, vf, dof, causal, scale)
    assert np.allclose(lse, lse_t, rtol=1e-14, atol=1e-12)
    assert np.abs(qz.dq - 2.0 ** -4 / 1.0).max() == 0 and np.abs(qz.dk - 2.0 ** -4).max() == 0
    dq, dk, dv = orc.sagebwd_backward(shape, 0, bq, bk, causal, scale, q, k, v, qz, o, dout, lse)
    for got, want in ((dq, gq), (dk, gk), (dv, gv)):
        assert np.abs(want).max() > 1.0
        assert _close(got, want, 1e-12)


def _cos_err(got, want):
    return 1.0 - (got * want).sum() / math.sqrt((got * got).sum() * (want * want).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_gaussian_gradients_close_to_autograd(orc, causal):
    """K with channel offsets N(0, 3^2), per-block INT8 P, dO, dS and the
    forward's Q^, K^, dP = dO V^T unquantized.  With K smoothed (and the k_bar
    correction from the unquantized dS) every gradient stays within 1 - cos
    < 2.5e-3 of fp64 autograd (measured 1.6e-3, 9e-4, 7e-4 for dQ, dK, dV).
    Without smoothing the INT8 dS K product carries K's offsets and dQ's error
    is several times larger (measured 8.5e-3)."""
    shape = (1, 4, 2, 128, 192, 64)
    B, Hq, Hkv, N, M, d = shape
    q, k, v = rand_qkv(*shape, seed=13, koff=3.0)
    dout = bf16_tensor(np.random.default_rng(14).standard_normal((B, Hq, N, d)))
    scale = 0.125
    gq, gk, gv, o, _ = autograd(f64(q), f64(k), f64(v), f64(dout), causal, scale)
    err = {}
    for flags in (0, orc.SMOOTH_K):
        qz, _, lse = _forward(orc, shape, flags, 64, 64, causal, scale, q, k, v)
        dq, dk, dv = orc.sagebwd_backward(shape, flags, 64, 64, causal, scale, q, k, v, qz, o, dout, lse)
        err[flags] = [_cos_err(dq, gq), _cos_err(dk, gk), _cos_err(dv, gv)]
    assert max(err[orc.SMOOTH_K]) < 2.5e-3, err
    assert err[0][0] > 3.0 * err[orc.SMOOTH_K][0], err


def test_prepare_restated(orc):
    """dO^: per bq-row block (ragged last block), scale fl(max|dO_i| / 127), codes
    clamp(rint(fl(x / scale))) -- restated here in numpy binary32; D = rowsum(dO o O)."""
    B, Hq, Hkv, N, M, d, bq = 1, 2, 1, 200, 64, 32, 64
    rng = np.random.default_rng(31)
    dout = bf16_tensor(rng.standard_normal((B, Hq, N, d)) * 3.0)
    o = rng.standard_normal((B, Hq, N, d))
    doc, dos, D = orc.sagebwd_prepare((B, Hq, Hkv, N, M, d), bq, o, dout)
    x = f64(dout).astype(np.float32)
    for i in range(-(-N // bq)):
        blk = x[:, :, i * bq:(i + 1) * bq]
        sc = (np.abs(blk).max(axis=(2, 3)) / np.float32(127)).astype(np.float32)
        assert np.array_equal(dos[:, :, i], sc), i
        want = np.clip(np.rint(blk / sc[:, :, None, None]), -127, 127).astype(np.int8)
        assert np.array_equal(doc[:, :, i * bq:(i + 1) * bq], want), i
    assert np.allclose(D, (f64(dout) * o).sum(-1), rtol=1e-13, atol=1e-13)


def test_int8_dov_ablation_hurts_dq(orc):
    """The pages' reason to keep dO V^T unquantized: with INT8 dO^ and V^ in dP,
    dQ's error grows with V's channel means (the dO dV^T term does not average
    out), while dK and dV stay put.  Measured here: dQ 1 - cos 1.6e-3 -> 2.5e-2
    (V offsets N(0, 1)) -> 0.16 (N(0, 3^2)); dK, dV within 2x."""
    shape = (1, 4, 2, 128, 192, 64)
    B, Hq, Hkv, N, M, d = shape
    q, k, v = rand_qkv(*shape, seed=13, koff=3.0, voff=3.0)
    dout = bf16_tensor(np.random.default_rng(14).standard_normal((B, Hq, N, d)))
    gq, gk, gv, o, _ = autograd(f64(q), f64(k), f64(v), f64(dout), False, 0.125)
    qz, _, lse = _forward(orc, shape, orc.SMOOTH_K, 64, 64, False, 0.125, q, k, v)
    err = {}
    for flags in (orc.SMOOTH_K, orc.SMOOTH_K | orc.BWD_INT8_DP):
        dq, dk, dv = orc.sagebwd_backward(shape, flags, 64, 64, False, 0.125, q, k, v, qz, o, dout, lse)
        err[flags] = [_cos_err(dq, gq), _cos_err(dk, gk), _cos_err(dv, gv)]
    base, int8 = err[orc.SMOOTH_K], err[orc.SMOOTH_K | orc.BWD_INT8_DP]
    assert int8[0] > 20 * base[0], err
    assert int8[1] < 2 * base[1] and int8[2] < 2 * base[2], err
