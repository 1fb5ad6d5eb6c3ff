"""Pins for the oracle's packed-sequence (varlen) attention (CPU only).

- Sequences of one length packed together give the batched result bit for bit.
- With identity quantizers, ragged packed sequences equal textbook attention
  over the whole packed score matrix with a block-diagonal mask (each query
  sees its own sequence's keys only, bottom-right causal within it).
- Changing one sequence's tokens leaves every other sequence's output unchanged
  (means, scales and blocks are per sequence).
"""
import math

import numpy as np
import pytest

from test_oracle_attention import bf16_tensor, f64


def _packed(rng, total, H, d, off=0.0):
    x = rng.standard_normal((total, H, d)) + off * rng.standard_normal((1, H, d))
    return bf16_tensor(x)


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)


def test_equal_lengths_equal_batched(orc):
    rng = np.random.default_rng(1)
    S, Hq, Hkv, L, Lk, d, bq, bk = 3, 4, 2, 40, 56, 32, 16, 16
    q, k, v = _packed(rng, S * L, Hq, d, 2.0), _packed(rng, S * Lk, Hkv, d, 3.0), _packed(rng, S * Lk, Hkv, d, 1.0)
    flags = orc.SMOOTH_K | orc.SMOOTH_Q | orc.SMOOTH_V
    out, lse, quants = orc.attn_varlen(0, flags, bq, bk, True, 0.2, q, k, v, _cu([L] * S), _cu([Lk] * S))

    def batched(x, n):
        return x.reshape(S, n, x.shape[1], d).permute(0, 2, 1, 3).contiguous()

    qb, kb, vb = batched(q, L), batched(k, Lk), batched(v, Lk)
    shape = (S, Hq, Hkv, L, Lk, d)
    qz = orc.quantize(shape, 0, flags, bq, bk, qb, kb, vb)
    o, l = orc.attn_rows_lse(shape, 0, flags, bq, bk, True, 0.2, qb, kb, vb, qz, orc.all_rows(shape))
    assert np.array_equal(out, o.reshape(S, Hq, L, d).transpose(0, 2, 1, 3).reshape(S * L, Hq, d))
    assert np.array_equal(lse, l.reshape(S, Hq, L).transpose(0, 2, 1).reshape(S * L, Hq))
    for s in range(S):
        assert np.array_equal(quants[s].kc[0], qz.kc[s]) and np.array_equal(quants[s].dq[0], qz.dq[s])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("flags", [0, 1 | 2 | 4])
def test_identity_quantizers_block_diagonal_textbook(orc, causal, flags):
    rng = np.random.default_rng(2)
    Hq, Hkv, d, bq, bk = 4, 2, 16, 16, 16
    lq = [17, 0, 1, 40, 33]
    lk = [17, 5, 30, 40, 70] if causal else [9, 5, 1, 64, 20]
    cq, ck = _cu(lq), _cu(lk)
    q, k, v = _packed(rng, cq[-1], Hq, d, 2.0), _packed(rng, ck[-1], Hkv, d, 3.0), _packed(rng, ck[-1], Hkv, d, 2.0)
    scale = 1.0 / math.sqrt(d)
    out, lse, quants = orc.attn_varlen(0, flags | orc.EXACT_QK | orc.EXACT_PV, bq, bk, causal, scale,
                                       q, k, v, cq, ck)
    assert quants[1] is None
    # textbook over the packed matrix: row i of sequence s sees key j of sequence s
    # iff (causal) j - ck[s] <= (i - cq[s]) + (lk[s] - lq[s])
    qf, kf, vf = f64(q), f64(k), f64(v)
    seq_q = np.repeat(np.arange(len(lq)), lq)
    seq_k = np.repeat(np.arange(len(lk)), lk)
    pos_q = np.arange(cq[-1]) - cq[seq_q]
    pos_k = np.arange(ck[-1]) - ck[seq_k]
    vis = seq_q[:, None] == seq_k[None, :]
    if causal:
        vis &= pos_k[None, :] <= pos_q[:, None] + (np.array(lk) - np.array(lq))[seq_q][:, None]
    g = Hq // Hkv
    for h in range(Hq):
        s = qf[:, h, :] @ kf[:, h // g, :].T * scale
        s = np.where(vis, s, -np.inf)
        mx = s.max(-1, keepdims=True)
        p = np.exp(s - mx)
        want = (p @ vf[:, h // g, :]) / p.sum(-1, keepdims=True)
        assert np.allclose(out[:, h, :], want, rtol=1e-12, atol=1e-12)
        if flags == 0:
            assert np.allclose(lse[:, h], mx[:, 0] + np.log(p.sum(-1)), rtol=1e-13, atol=1e-13)


def test_sequences_are_isolated(orc):
    """Quantized, all smoothing on: new tokens in sequence 1 change nothing
    in sequences 0 and 2 (not a bit)."""
    rng = np.random.default_rng(3)
    Hq, Hkv, d = 2, 1, 32
    lq, lk = [30, 20, 45], [30, 50, 45]
    cq, ck = _cu(lq), _cu(lk)
    q, k, v = _packed(rng, cq[-1], Hq, d, 2.0), _packed(rng, ck[-1], Hkv, d, 3.0), _packed(rng, ck[-1], Hkv, d, 1.0)
    flags = 1 | 2 | 4
    a, la, _ = orc.attn_varlen(0, flags, 16, 16, True, 0.15, q, k, v, cq, ck)
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[cq[1]:cq[2]] = _packed(rng, lq[1], Hq, d, 5.0)
    k2[ck[1]:ck[2]] = _packed(rng, lk[1], Hkv, d, 9.0)
    v2[ck[1]:ck[2]] = _packed(rng, lk[1], Hkv, d, 4.0)
    b, lb, _ = orc.attn_varlen(0, flags, 16, 16, True, 0.15, q2, k2, v2, cq, ck)
    keep = np.r_[cq[0]:cq[1], cq[2]:cq[3]]
    assert np.array_equal(a[keep], b[keep]) and np.array_equal(la[keep], lb[keep])
    assert not np.array_equal(a[cq[1]:cq[2]], b[cq[1]:cq[2]])


def test_rejects_bad_cu_seqlens(orc):
    rng = np.random.default_rng(4)
    q, k, v = _packed(rng, 10, 2, 16), _packed(rng, 12, 2, 16), _packed(rng, 12, 2, 16)
    with pytest.raises(orc.OracleError, match="no keys"):
        orc.attn_varlen(0, 1, 16, 16, False, 0.25, q, k, v, _cu([4, 6]), _cu([12, 0]))
    with pytest.raises(orc.OracleError, match="disagree"):
        orc.attn_varlen(0, 1, 16, 16, False, 0.25, q, k, v, _cu([4, 5]), _cu([6, 6]))
    with pytest.raises(orc.OracleError, match="start at 0"):
        orc.attn_varlen(0, 1, 16, 16, False, 0.25, q, k, v, np.array([1, 10]), _cu([12]))
