"""Seeded synthetic Q, K, V in bf16 for a ``Config``.

Draws come from numpy's PCG64 generator (seeded per config), are shaped and
shifted as the config's recipe says, and are rounded to bf16 (round to
nearest even).  Inputs are produced once on the host; the CUDA path receives
a device copy of the same bits, so the oracle and the kernels see identical
values.  Tensors are contiguous [B, H, L, d].
"""
from __future__ import annotations

import numpy as np
import torch

from .configs import Config


def _rng(cfg: Config, stream: int) -> np.random.Generator:
    # independent sub-streams for Q, K, V and the offset draws
    return np.random.Generator(np.random.PCG64([cfg.seed, stream]))


def make_qkv_float(cfg: Config):
    """float32 Q, K, V (before the bf16 rounding) following the config's recipe."""
    B, Hq, Hkv, N, M, d = cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d
    rq, rk, rv, ro = _rng(cfg, 1), _rng(cfg, 2), _rng(cfg, 3), _rng(cfg, 4)

    q = rq.standard_normal((B, Hq, N, d), dtype=np.float32)
    k = rk.standard_normal((B, Hkv, M, d), dtype=np.float32)
    if cfg.q_from_k_noise > 0:
        # peaked attention: query i of head h copies key pick[i] of its kv head
        g = Hq // Hkv
        pick = rq.integers(0, M, size=(B, Hq, N))
        kk = np.repeat(k, g, axis=1)
        q = np.take_along_axis(kk, pick[..., None], axis=2) + q * np.float32(cfg.q_from_k_noise)

    if cfg.v_student_t > 0:
        nu = cfg.v_student_t
        z = rv.standard_normal((B, Hkv, M, d), dtype=np.float32)
        chi = rv.chisquare(nu, size=(B, Hkv, M, d)).astype(np.float32)
        v = z / np.sqrt(chi / np.float32(nu))
    else:
        v = rv.standard_normal((B, Hkv, M, d), dtype=np.float32)
    if cfg.v_clip > 0:
        np.clip(v, -cfg.v_clip, cfg.v_clip, out=v)

    for c in cfg.k_fixed_channels:
        k[..., c] += np.float32(cfg.k_fixed_shift)
    if cfg.k_offset_std > 0:
        k += (ro.standard_normal((B, Hkv, 1, d)) * cfg.k_offset_std).astype(np.float32)
    if cfg.k_outliers > 0:
        chans = ro.choice(d, size=cfg.k_outliers, replace=False)
        for c in chans:
            k[..., int(c)] += np.float32(cfg.k_outlier_shift)
    if cfg.q_offset_std > 0:
        q += (ro.standard_normal((B, Hq, 1, d)) * cfg.q_offset_std).astype(np.float32)
    if cfg.q_block_shift_std > 0:
        L = cfg.q_block_len
        nb = (N + L - 1) // L
        sh = (ro.standard_normal((B, Hq, nb, 1, d)) * cfg.q_block_shift_std).astype(np.float32)
        sh = np.broadcast_to(sh, (B, Hq, nb, L, d)).reshape(B, Hq, nb * L, d)[:, :, :N]
        q += sh
    if cfg.v_bias_std > 0:
        v += (ro.standard_normal((B, Hkv, 1, d)) * cfg.v_bias_std).astype(np.float32)
    return q, k, v


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """float32 numpy -> bf16 torch tensor (torch's CPU cast rounds to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


def make_inputs(cfg: Config):
    """bf16 CPU tensors (q, k, v), contiguous [B, H, L, d]."""
    q, k, v = make_qkv_float(cfg)
    return to_bf16(q), to_bf16(k), to_bf16(v)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw uint16 bit patterns of a contiguous bf16 CPU tensor."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
