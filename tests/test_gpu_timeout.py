"""The bounded-wait unwind path of both attention kernels, exercised without a
fault: a child process sets a short spin limit (SAGE_SPIN_LIMIT, clock
cycles) and the test hook SAGE_TEST_STALL=1, which makes each CTA's QK issuer
wait on a barrier that nothing arrives on.  The wait runs out, the kernel
records SAGE_ERR_TIMEOUT with the site of that wait (29), every warp leaves its
loop, the CTA waits for its own copies and MMAs, frees TMEM and returns.  The
same process then clears the hook and runs the same request again: the context
must still be usable and the output must match the oracle."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, %(root)r)
sys.path.insert(0, os.path.join(%(root)r, "tests"))
import numpy as np
import torch
import bit_quantized_attention_gb300 as sage
import oracle
from gpu_helpers import output_metrics
from workload import CONFIGS
from workload import make_inputs

out = {}
for name, cfg in (("int8", CONFIGS["tiny"]),
                  ("int8_smooth_q", CONFIGS["tiny"].with_(name="t_sq", flags=7, d=128, bk=128)),
                  ("nvfp4", CONFIGS["tiny"].with_(name="t_fp4", mode=2, bk=128, d=128))):
    q, k, v = make_inputs(cfg)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    os.environ["SAGE_TEST_STALL"] = "1"
    ws = sage.sage_quantize_qkv(qd, kd, vd, cfg.mode, cfg.flags, cfg.bq, cfg.bk)
    sage.sage_attn_fwd(ws, cfg.causal, cfg.sm_scale)
    torch.cuda.synchronize()
    stalled = sage.sage_read_status(ws)
    os.environ["SAGE_TEST_STALL"] = "0"
    ws = sage.sage_quantize_qkv(qd, kd, vd, cfg.mode, cfg.flags, cfg.bq, cfg.bk)
    o = sage.sage_attn_fwd(ws, cfg.causal, cfg.sm_scale)
    torch.cuda.synchronize()
    clean = sage.sage_read_status(ws)
    shape = (cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.M, cfg.d)
    qz = oracle.quantize(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, q, k, v)
    ref = oracle.attn_rows(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, cfg.causal, cfg.sm_scale, q, k, v, qz,
                           oracle.all_rows(shape))
    m = output_metrics(o.float().cpu().numpy().reshape(ref.shape), oracle.bf16_round(ref))
    out[name] = dict(stalled=list(stalled), clean=list(clean), max_rel=m["max_rel"], rel_l1=m["rel_l1"])
print("RESULT " + json.dumps(out))
"""


def test_bounded_wait_runs_out_and_unwinds():
    import __graft_entry__
    __graft_entry__.build_library()
    import oracle
    oracle.build()
    env = dict(os.environ, SAGE_SPIN_LIMIT="20000000")  # about 10 ms
    r = subprocess.run([sys.executable, "-c", CHILD % {"root": ROOT}], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    for name, x in res.items():
        assert x["stalled"] == [5, 29], (name, x)  # SAGE_ERR_TIMEOUT at the QK issuer's stall wait
        assert x["clean"] == [0, 0], (name, x)
        assert x["max_rel"] <= 1e-2 and x["rel_l1"] <= 2e-3, (name, x)
