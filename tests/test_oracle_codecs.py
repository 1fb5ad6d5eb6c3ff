"""Pins for the oracle's codecs and quantizer building blocks (CPU only).

Each check compares the oracle with something other than itself: values the
pages print (tests/golden), a library implementation of the same format
(torch's float8_e4m3fn and bfloat16 casts), exact rational arithmetic, or a
brute-force nearest-value search written here.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import golden


def f32(x):
    return struct.unpack("f", struct.pack("f", x))[0]


# ------------------------------------------------------------------ E2M1
def test_e2m1_values_match_pages(orc):
    g = golden("e2m1_values.txt")
    vals = orc.e2m1_decode(np.arange(16))
    distinct = sorted(set(float(v) + 0.0 for v in vals))  # +0.0 folds -0 into 0
    assert distinct == sorted(g["values"])
    assert len(distinct) == int(g["distinct"])
    assert max(abs(v) for v in distinct) == g["max"]


def _nearest_even_bruteforce(x, mags):
    """Nearest magnitude by exhaustive distance, ties to the even index."""
    a = abs(x)
    if a >= mags[-1]:
        return len(mags) - 1
    dist = [abs(a - m) for m in mags]
    best = min(dist)
    cands = [i for i, dd in enumerate(dist) if dd == best]
    if len(cands) == 1:
        return cands[0]
    return [c for c in cands if c % 2 == 0][0]


def test_e2m1_encode_bruteforce(orc):
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    xs = [i / 64.0 for i in range(-512, 513)]                      # dense grid incl. all midpoints
    xs += [(mags[i] + mags[i + 1]) / 2 for i in range(7)]          # exact ties
    rng = np.random.default_rng(5)
    xs += list(rng.uniform(-8, 8, 4000).astype(np.float32).astype(float))
    xs = np.array(xs, np.float32)
    got = orc.e2m1_encode(xs)
    for x, c in zip(xs, got):
        want = _nearest_even_bruteforce(float(x), mags) | (0x8 if math.copysign(1, x) < 0 else 0)
        assert c == want, (x, c, want)


def test_e2m1_ties_by_hand(orc):
    # ties resolve to the even code: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2.0,
    # 2.5 -> 2.0, 3.5 -> 4.0, 5 -> 4.0; 7 saturates to 6
    cases = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0, 7.0: 6.0,
             100.0: 6.0, -5.0: -4.0}
    codes = orc.e2m1_encode(np.array(list(cases), np.float32))
    assert list(orc.e2m1_decode(codes)) == list(cases.values())


# ------------------------------------------------------------------ E4M3
def test_e4m3_facts_match_pages(orc):
    g = golden("e4m3_facts.txt")
    vals = orc.e4m3_decode(np.arange(256))
    fin = vals[np.isfinite(vals)]
    assert fin.max() == g["max"]
    nonneg = sorted(set(float(v) for v in fin if v >= 0))
    assert len([v for v in nonneg if v <= 448]) == int(g["count_0_448"])
    assert len([v for v in nonneg if v <= 1 / 6]) == int(g["count_0_sixth"])


def test_e4m3_decode_matches_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def _all_bf16_finite_f32():
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    return x[np.isfinite(x)]


@pytest.mark.parametrize("shift", [-12, -6, 0, 3])
def test_e4m3_encode_matches_torch(orc, shift):
    """Every bf16 value (scaled by 2^shift) inside the finite E4M3 range, encoded
    by the oracle and by torch's float32 -> float8_e4m3fn cast (RNE)."""
    x = _all_bf16_finite_f32().astype(np.float64) * 2.0 ** shift
    x = x[np.abs(x) <= 448].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode(x)
    assert np.array_equal(ref, got)


def test_e4m3_ties_and_saturation_by_hand(orc):
    # 17 lies halfway between 16 (mantissa 000) and 18 (001): even -> 16.
    # 19 between 18 (001) and 20 (010): even -> 20.  2^-10 between 0 and 2^-9: -> 0.
    # 3*2^-10 between 2^-9 (001) and 2*2^-9 (010): -> 2^-8.  Above 448: saturate.
    cases = {17.0: 16.0, 19.0: 20.0, 2.0 ** -10: 0.0, 3 * 2.0 ** -10: 2.0 ** -8, 450.0: 448.0,
             1e6: 448.0, -1e6: -448.0, 464.0: 448.0, 0.0: 0.0}
    codes = orc.e4m3_encode(np.array(list(cases), np.float32))
    assert list(orc.e4m3_decode(codes)) == list(cases.values())
    assert orc.e4m3_encode(np.array([-0.0], np.float32))[0] == 0x80


# ------------------------------------------------------------------ bf16
def test_bf16_encode_matches_torch(orc):
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-38,
                        rng.standard_normal(2000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.bf16_encode(x.astype(np.float64))
    assert np.array_equal(ref, got)


def test_bf16_encode_single_rounding(orc):
    # 1 + 2^-8 + 2^-30 is just above the midpoint between 1 and 1 + 2^-7; one
    # rounding gives 1 + 2^-7 (a float32 detour would land on the tie and give 1).
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    bits = orc.bf16_encode(np.array([x]))[0]
    assert bits == 0x3F81
    assert orc.bf16_encode(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80  # exact tie -> even


# ------------------------------------------------------------------ INT8 / scales
def test_int8_zero_threshold_and_ties(orc):
    # With scale 1 (absmax 127) an element rounds to 0 iff |x| <= absmax/254 = 0.5
    # (the INT8 analogue of the INT4 "14 times smaller" rule in the SageAttention2
    # summary §3.4 "Smoothing Q"), ties to even.
    s = orc.int8_scale(127.0)
    assert s == 1.0
    assert orc.int8_code(0.5, s) == 0
    assert orc.int8_code(-0.5, s) == 0
    assert orc.int8_code(float(np.nextafter(np.float32(0.5), np.float32(1))), s) == 1
    assert orc.int8_code(1.5, s) == 2 and orc.int8_code(2.5, s) == 2 and orc.int8_code(-3.5, s) == -4
    assert orc.int8_code(127.0, s) == 127 and orc.int8_code(-127.0, s) == -127
    assert orc.int8_code(1.0, 0.0) == 0


def test_scale_closed_forms(orc):
    assert orc.int8_scale(127.0) == 1.0
    assert orc.fp8_scale(448.0) == 1.0
    assert orc.int8_scale(9.0) == f32(9.0 / 127.0)
    assert orc.nvfp4_scale(6.0) == 0x38          # e4m3(1.0)
    assert orc.nvfp4_scale(6.0 * 448) == 0x7E    # e4m3(448)
    assert orc.nvfp4_scale(0.0) == 0
    # an element equal to the block max lands on the top code
    assert orc.fp8_code(3.7, orc.fp8_scale(3.7)) == 0x7E
    assert orc.nvfp4_code(3.7, orc.nvfp4_scale(3.7)) in (0x7,)  # 6 (scale rounded down) or sat


def test_int8_worked_example_levels(orc):
    """The per-block INT8 worked example: an offset channel at ~8 +- 1 sets the
    block scale to ~9/127 and a +-0.3 channel spans ~8 codes; subtracting the
    channel means brings the scale to ~1/127 and the span to ~76 codes."""
    g = golden("p5_worked_example.txt")
    rng = np.random.default_rng(11)
    T, d = 64, 128
    base = np.linspace(-1, 1, T)
    k = np.stack([rng.permutation(base) for _ in range(d)], axis=1)[None, None].astype(np.float32)
    k[..., 5] = g["offset"] + np.linspace(-1, 1, T)       # offset channel, spread +-1
    k[..., 9] = np.linspace(-0.3, 0.3, T)                  # the +-0.3 channel
    kb = torch.from_numpy(k).to(torch.bfloat16)
    q = torch.zeros(1, 1, 128, d, dtype=torch.bfloat16)
    shape = (1, 1, 1, 128, T, d)
    res = {}
    for flags in (0, orc.SMOOTH_K):
        qz = orc.quantize(shape, orc.MODE_Q8_PV8, flags, 128, 64, q, kb, kb)
        codes = qz.kc[0, 0, :, 9].view(np.int8).astype(int)
        res[flags] = (float(qz.dk[0, 0, 0]), int(codes.max() - codes.min()))
    s0, l0 = res[0]
    s1, l1 = res[orc.SMOOTH_K]
    assert abs(s0 - g["scale_before"]) / g["scale_before"] < 0.02 and abs(l0 - g["levels_before"]) <= 1
    assert abs(s1 - g["scale_after"]) / g["scale_after"] < 0.1
    assert abs(l1 - g["levels_after"]) / g["levels_after"] < 0.1


# ------------------------------------------------------------------ means
def _exact_mean_f32(vals):
    fr = sum((Fraction(float(v)) for v in vals), Fraction(0)) / len(vals)
    return fr


@pytest.mark.parametrize("scale", [1.0, 1e-3, 300.0])
def test_mean_matches_exact_rational(orc, scale):
    rng = np.random.default_rng(int(scale * 1000) % 97)
    for n in (1, 2, 7, 64, 1000, 4097):
        x = (rng.standard_normal(n) * scale + 0.3 * scale).astype(np.float32)
        bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        vals = (bits.astype(np.uint32) << 16).view(np.float32)
        exact = _exact_mean_f32(vals)
        got = orc.mean_bf16(bits)
        # one rounding to double then to float: within one float ulp of the exact
        # mean, plus the 2^-24 truncation for tiny elements
        ulp = float(np.spacing(np.float32(abs(float(exact)))))
        assert abs(Fraction(got) - exact) <= Fraction(ulp) + Fraction(2.0 ** -24), (n, got, float(exact))


def test_mean_closed_forms(orc):
    for c in (1.5, -3.25, 1000.0, 2.0 ** -10):
        bits = np.full(777, np.float32(c)).view(np.uint32) >> 16
        assert orc.mean_bf16(bits.astype(np.uint16)) == c
    pair = np.array([0x4040, 0xC040], np.uint16)  # 3, -3
    assert orc.mean_bf16(pair) == 0.0


def test_mean_range_errors(orc):
    big = np.array([0x4780], np.uint16)  # 65536
    with pytest.raises(orc.OracleError):
        orc.mean_bf16(big)
    inf = np.array([0x7F80], np.uint16)
    with pytest.raises(orc.OracleError):
        orc.mean_bf16(inf)
