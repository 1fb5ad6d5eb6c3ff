"""The oracle's pins catch plausible mistakes in it.

Each case plants one mistake in a copy of the oracle's C source (a dropped or
flipped term, a wrong index, a wrong constant, the other tie rule), builds the
copy, and runs the oracle's own tests against it in a subprocess: at least one
of them must fail.  The unmutated copy must pass.  Only the copy is touched."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = [os.path.join(ROOT, "tests", f) for f in
         ("test_oracle_codecs.py", "test_oracle_attention.py", "test_oracle_sagebwd.py", "test_oracle_varlen.py",
          "test_oracle_sagebwd_backward.py")]

# (name, text in sage_oracle.c, replacement); each text occurs exactly once.  The
# packed-sequence composition lives in oracle.py: those entries name that file.
MUTATIONS = [
    ("dS dropped", "sv[c] = (s0 + ds) * sm_scale;", "sv[c] = (s0) * sm_scale;"),
    ("dS sign", "sv[c] = (s0 + ds) * sm_scale;", "sv[c] = (s0 - ds) * sm_scale;"),
    ("GQA map", "const int64_t hk = (int64_t)b * Hkv + h / (Hq / Hkv); /* kv head of this query head */",
     "const int64_t hk = (int64_t)b * Hkv + h % Hkv; /* kv head of this query head */"),
    ("causal offset", "return c <= r + (M - N);", "return c <= r;"),
    ("l not rescaled", "l = alpha * l + rs;", "l = l + rs;"),
    ("INT8 divisor", "float orc_int8_scale(float absmax) { return absmax / 127.0f; }",
     "float orc_int8_scale(float absmax) { return absmax / 128.0f; }"),
    ("INT8 clamp", "if (r > 127.0f) r = 127.0f;", "if (r > 126.0f) r = 126.0f;"),
    ("P~ scale 448", "orc_e4m3_encode(pv[c] * 448.0)", "orc_e4m3_encode(pv[c] * 256.0)"),
    ("output 448", "o = o / 448.0 * (double)qz->dv[hk * d + e];", "o = o / 256.0 * (double)qz->dv[hk * d + e];"),
    ("delta_V dropped", "o = o / 448.0 * (double)qz->dv[hk * d + e];", "o = o / 448.0;"),
    ("V_m dropped", "vrow[e] = o + (double)qz->vm[hk * d + e];", "vrow[e] = o;"),
    ("s_P1 constant", "exp(mt - m_new) / (448.0 * 6.0)", "exp(mt - m_new) / (448.0 * 4.0)"),
    ("s_P2 divisor", "s2c = orc_e4m3_encode(amax / 6.0);", "s2c = orc_e4m3_encode(amax / 4.0);"),
    ("ties away from zero", "r = nearbyint(ldexp(a, -ulp_exp));", "r = round(ldexp(a, -ulp_exp));"),
    ("mean divisor", "*mean = (n > 0) ? (float)(((double)acc * 0x1p-24) / (double)n) : 0.0f;",
     "*mean = (n > 0) ? (float)(((double)acc * 0x1p-24) / (double)(n + 1)) : 0.0f;"),
    ("K mean not subtracted (INT8/FP8)", "float x = bf16f(K[(int64_t)t * d + c]) - kbar[c];",
     "float x = bf16f(K[(int64_t)t * d + c]);"),
    ("Q mean not subtracted", "g[(int64_t)(r - r0) * d + c] = bf16f(Q[(int64_t)r * d + c]) - qbar[c];",
     "g[(int64_t)(r - r0) * d + c] = bf16f(Q[(int64_t)r * d + c]);"),
    ("NVFP4 scale divisor", "return orc_e4m3_encode((double)(absmax / 6.0f));",
     "return orc_e4m3_encode((double)(absmax / 4.0f));"),
    ("per-token Q dequantized per block",
     "const double sq = (flags & ORC_Q_PER_TOKEN) ? (double)qz->dqt[hb * N + r] : (double)qz->dq[hb * Tm + ib];",
     "const double sq = (double)qz->dq[hb * Tm + ib];"),
    # (a power-of-two level-1 scale commutes with the E4M3 / E2M1 roundings away from
    # the subnormal range, so the planted constant is not one)
    ("running max forgets the previous tiles", "m_new = (mt > m) ? mt : m;", "m_new = mt;"),
    ("alpha sign", "alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);",
     "alpha = (m == -INFINITY) ? 0.0 : exp(m_new - m);"),
    ("sm_scale before dS", "sv[c] = (s0 + ds) * sm_scale;", "sv[c] = s0 * sm_scale + ds;"),
    ("V mean not subtracted before quantizing",
     "g[(int64_t)t * d + c] = bf16f(V[(int64_t)t * d + c]) - vm[c];",
     "g[(int64_t)t * d + c] = bf16f(V[(int64_t)t * d + c]);"),
    ("delta_V doubled", "dv[c] = orc_fp8_scale(amax);", "dv[c] = orc_fp8_scale(amax * 2.0f);"),
    ("pad keys visible", "if (c >= M) return 0;", "if (c > M) return 0;"),
    ("INT8 rounds half away from zero", "r = rintf(t);", "r = roundf(t);"),
    ("INT8 truncates", "r = rintf(t);", "r = truncf(t);"),
    ("E4M3 code without the scale", "return orc_e4m3_encode((double)(x / scale));",
     "return orc_e4m3_encode((double)(x));"),
    ("NVFP4 V scale not stored", "out->vs[(hb * Mt16 + tb) * d + c] = sc;", "out->vs[(hb * Mt16 + tb) * d + c] = 0x38;"),
    ("NVFP4 Q scale not stored", "out->qs[(hb * N + r) * G16 + gi] = sc;", "out->qs[(hb * N + r) * G16 + gi] = 0x38;"),
    ("NVFP4 K code from the next element",
     "out->kc[(hb * M + t) * d + gi * 16 + e] = orc_nvfp4_code(gg[e], sc);",
     "out->kc[(hb * M + t) * d + gi * 16 + e] = orc_nvfp4_code(gg[(e + 1) & 15], sc);"),
    ("P2 not divided by s_P1", "p2[c] = (sP1 == 0.0) ? 0.0 : pv[u + c] / sP1;", "p2[c] = pv[u + c];"),
    ("P^ not multiplied back by s_P2", "ph = orc_e2m1_decode(orc_e2m1_encode(p2[c] / s2)) * s2;",
     "ph = orc_e2m1_decode(orc_e2m1_encode(p2[c] / s2));"),
    ("E2M1 code of the unscaled P2", "ph = orc_e2m1_decode(orc_e2m1_encode(p2[c] / s2)) * s2;",
     "ph = orc_e2m1_decode(orc_e2m1_encode(p2[c])) * s2;"),
    ("NVFP4 V block max from one token",
     "            for (t = t0; t < t1; ++t)\n              if (fabsf(g[(int64_t)t * d + c]) > amax) amax = "
     "fabsf(g[(int64_t)t * d + c]);\n            sc = orc_nvfp4_scale(amax);\n            out->vs[",
     "            for (t = t0; t < t0 + 1; ++t)\n              if (fabsf(g[(int64_t)t * d + c]) > amax) amax = "
     "fabsf(g[(int64_t)t * d + c]);\n            sc = orc_nvfp4_scale(amax);\n            out->vs["),
    ("NVFP4 V scale index", "orc_e4m3_decode(qz->vs[(hk * Mt16 + t / 16) * d + e]);",
     "orc_e4m3_decode(qz->vs[(hk * Mt16 + t / 32) * d + e]);"),
    ("l summed over quantized P^", "for (c = 0; c < bk; ++c) rs += pv[c];",
     "for (c = 0; c < bk; ++c) rs += orc_e4m3_decode(orc_e4m3_encode(pv[c] * 448.0)) / 448.0;"),
    ("direct P~ keeps a level-1 scale", "(flags & ORC_P_DIRECT) ? 1.0 :", "(flags & ORC_P_DIRECT) ? (1.0 / 3.0) :"),
    # SageBwd forward (per-block INT8 V, per-token INT8 P~) and the softmax statistics
    ("SageBwd s_P divisor", "sP = (mt == -INFINITY) ? 0.0 : exp(mt - m_new) / 127.0;",
     "sP = (mt == -INFINITY) ? 0.0 : exp(mt - m_new) / 128.0;"),
    ("SageBwd s_P from the running max, not the tile's", "sP = (mt == -INFINITY) ? 0.0 : exp(mt - m_new) / 127.0;",
     "sP = (mt == -INFINITY) ? 0.0 : exp(m_new - m_new) / 127.0;"),
    ("SageBwd P^ truncated", "ph = nearbyint(pv[c] / sP);", "ph = floor(pv[c] / sP);"),
    ("SageBwd s_P not multiplied back", "rsc = sP * (double)qz->dvb[hk * Tn + j];", "rsc = (double)qz->dvb[hk * Tn + j];"),
    ("SageBwd s_V of the first block", "rsc = sP * (double)qz->dvb[hk * Tn + j];", "rsc = sP * (double)qz->dvb[hk * Tn];"),
    ("SageBwd V block max over one channel",
     "            for (c = 0; c < d; ++c)\n              if (fabsf(g[(int64_t)t * d + c]) > amax) amax = "
     "fabsf(g[(int64_t)t * d + c]);\n          sc = orc_int8_scale(amax);\n          out->dvb",
     "            for (c = 0; c < 1; ++c)\n              if (fabsf(g[(int64_t)t * d + c]) > amax) amax = "
     "fabsf(g[(int64_t)t * d + c]);\n          sc = orc_int8_scale(amax);\n          out->dvb"),
    ("SageBwd V codes from the E4M3 quantizer",
     "out->vc[(hb * M + t) * d + c] = (uint8_t)(int8_t)orc_int8_code(g[(int64_t)t * d + c], sc);",
     "out->vc[(hb * M + t) * d + c] = orc_fp8_code(g[(int64_t)t * d + c], sc);"),
    ("SageBwd Q and K on the E4M3 quantizer", "return mode == ORC_Q8_PV8 || mode == ORC_SAGEBWD_I8;",
     "return mode == ORC_Q8_PV8;"),
    ("SageBwd output keeps the 448 / delta_V epilogue", "(mode == ORC_Q8_PV8 || mode == ORC_QF8_PV8))",
     "mode != ORC_NVFP4)"),
    ("lse without the log", "if (lse) lse[ri] = m + log(l);", "if (lse) lse[ri] = m + l;"),
    # SageBwd backward
    ("backward dS without D_i", "x = P[r * bk + c] * (dp - Dr[r0 + r]);", "x = P[r * bk + c] * dp;"),
    ("backward dS without P", "x = P[r * bk + c] * (dp - Dr[r0 + r]);", "x = (dp - Dr[r0 + r]);"),
    ("backward D_i from dO alone", "acc += orc_bf16_decode(dO[(int64_t)r * d + e]) * O[(int64_t)r * d + e];",
     "acc += orc_bf16_decode(dO[(int64_t)r * d + e]);"),
    ("backward dO block maximum of one row", "    for (r = r0; r < r1; ++r)\n      for (e = 0; e < d; ++e)\n        if (fabsf(bf16f(dO",
     "    for (r = r0; r < r0 + 1; ++r)\n      for (e = 0; e < d; ++e)\n        if (fabsf(bf16f(dO"),
    ("backward P not normalised by lse", "pv = exp((s0 + ds) * sm_scale - lse[bh * N + r0 + r]);",
     "pv = exp((s0 + ds) * sm_scale);"),
    ("backward s_P divisor", "sP = pmax / 127.0;", "sP = pmax / 128.0;"),
    ("backward s_dS divisor", "sdS = smax / 127.0;", "sdS = smax / 128.0;"),
    ("backward dO scale not multiplied back", "* (double)dos[i];", ";"),
    ("backward dK without sm_scale", "for (int64_t i = 0; i < n; ++i) dk[i] *= sm_scale;", ""),
    ("backward dQ without sm_scale", "for (int64_t i = 0; i < n; ++i) dq[i] *= sm_scale;", ""),
    ("backward k_bar correction dropped", "+ gx * (double)kbar[e];", ";"),
    ("backward k_bar correction from the INT8 dS", "+ gx * (double)kbar[e];", "+ g * (double)kbar[e];"),
    ("backward q_bar correction dropped", "+ gx * (double)qbar[e];", ";"),
    ("varlen keys sliced at the query offsets", "ks = np.ascontiguousarray(kb[ck[s]:ck[s + 1]]",
     "ks = np.ascontiguousarray(kb[cq[s]:cq[s] + Lk]", "oracle.py"),
    ("varlen output rows not transposed back", "o.reshape(Hq, Lq, d).transpose(1, 0, 2)",
     "o.reshape(Lq, Hq, d)", "oracle.py"),
    ("varlen causal offset of the packed matrix", "o, l = attn_rows_lse(shape, mode, flags, bq, bk, causal,",
     "o, l = attn_rows_lse(shape, mode, flags, bq, bk, causal and Lq == Lk,", "oracle.py"),
]


def _copy_oracle(dst, mutation=None):
    pkg = os.path.join(dst, "oracle")
    os.makedirs(pkg)
    for f in ("__init__.py", "oracle.py", "sage_oracle.c", "sage_oracle.h"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(pkg, f))
    if mutation is not None:
        old, new = mutation[:2]
        src = os.path.join(pkg, mutation[2] if len(mutation) > 2 else "sage_oracle.c")
        text = open(src).read()
        assert text.count(old) == 1, old
        open(src, "w").write(text.replace(old, new))
    # build the copy here, so that the subprocess only loads it
    out = subprocess.run([sys.executable, "-c", "import oracle; oracle.build(force=True)"], cwd=dst,
                         capture_output=True, text=True)
    assert out.returncode == 0, out.stderr[-2000:]


def _run_pins(dst):
    env = dict(os.environ, PYTHONPATH=dst + os.pathsep + ROOT)
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *TESTS],
                          cwd=dst, env=env, capture_output=True, text=True, timeout=600)


def _check(tmp, name, mutation):
    d = os.path.join(tmp, "m%02d" % name)
    os.makedirs(d)
    _copy_oracle(d, mutation)
    r = _run_pins(d)
    return r


def test_unmutated_copy_passes_and_every_planted_mistake_fails_a_pin(tmp_path):
    """All copies built and run in parallel (one subprocess each)."""
    from concurrent.futures import ThreadPoolExecutor
    jobs = [None] + [m[1:] for m in MUTATIONS]
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda a: _check(str(tmp_path), a[0], a[1]), enumerate(jobs)))
    clean = results[0]
    assert clean.returncode == 0, clean.stdout[-3000:]
    # 1: some test failed (not an import, collection or usage error)
    missed = [m[0] for m, r in zip(MUTATIONS, results[1:]) if not (r.returncode == 1 and " failed" in r.stdout)]
    assert not missed, missed
