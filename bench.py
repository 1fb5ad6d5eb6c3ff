"""Throughput of the quantized attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--bk BK] [--impl reference]

One step = the whole hot path over one batch: the smoothing + quantization
pre-pass (sage_quantize_qkv) and the fused attention (sage_attn_fwd), with
inputs resident in HBM.  Metric: TOPS = 4*B*H*N*M*d / t (halved when causal).
Timing: W warm-up steps, then K steps bracketed by a barrier and a device
synchronize, CUDA events on the launching stream, max over ranks.  Inputs
(Q, K, V in bf16) are larger than L2, so no flush is needed between steps.

Extra keys on the JSON line:
  e2e          the same metric through sage_attn_host (pinned host buffers, the
               host->device copies and the device->host copy of O in the timed region)
  roofline     the attention kernel against the measured tensor peak
  cpu_baseline the CPU oracle on a bounded sample of the same workload (all
               host cores, and one thread extrapolated)
  clocks       SM clocks and throttle reasons sampled during the timed region
  per_workload the other workloads (LLM prefill, chunked GQA prefill, NVFP4),
               each timed on its own with its roofline, pre-pass time and clocks
  ablation     the method's switches timed on the video and NVFP4 workloads
               (smoothing on/off, per-token Q, E4M3 Q/K, direct P~, SageBwd)
  backward     the SageBwd training step on the LLM prefill shape: forward,
               the backward's pre-pass and the backward, with its roofline
The headline workload is the video-diffusion one (B2 H48 N=M=17776 d64, Q/K/V
smoothing), the largest non-causal INT8 / FP8 case.
Under torchrun (N > 1) every rank runs its own batch of the workload on its
own GPU (independent problems, no collective on the data path): weak scaling.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 126 * 1024 * 1024
NOMINAL_FP8_OVER_BF16 = 2.0   # dense fp8 / dense bf16 tensor rate (4.5 / 2.25 PFLOP/s)
NOMINAL_FP4_OVER_BF16 = 6.0   # dense fp4 / dense bf16 tensor rate (13.5 / 2.25 PFLOP/s)
LAUNCHES_PER_STEP = 5         # init, statistics, finalize, quantize, attention
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["bf16_tflops"], d.get("bf16_tflops_sustained"), d["hbm_gbs"], "measured"
    return FALLBACK_BF16_TFLOPS, None, FALLBACK_HBM_GBS, "fallback"


def attention_peak(mode: int, bf16_tflops: float):
    """Dense tensor peak of the attention kernel's instruction mix, TFLOP/s.
    INT8 Q/K runs QK^T as kind::f16 (INT8 codes held as fp16) and P^V as
    kind::f8f6f4: equal op counts at the bf16 and fp8 rates."""
    fp8 = bf16_tflops * NOMINAL_FP8_OVER_BF16
    if mode == 0:
        return 2.0 / (1.0 / bf16_tflops + 1.0 / fp8), "kind::f16 (QK) + kind::f8f6f4 (PV)"
    if mode == 1:
        return fp8, "kind::f8f6f4"
    return bf16_tflops * NOMINAL_FP4_OVER_BF16, "kind::mxf4nvf4.block_scale (QK and PV)"


def peak_source(mode: int, src: str, bf16: float) -> str:
    ratio = {0: "nominal fp8/bf16 ratio %.0f (harmonic mean of bf16 and fp8)" % NOMINAL_FP8_OVER_BF16,
             1: "nominal fp8/bf16 ratio %.0f" % NOMINAL_FP8_OVER_BF16,
             2: "nominal fp4/bf16 ratio %.0f" % NOMINAL_FP4_OVER_BF16}[mode]
    return "%s bf16 burst %.1f TFLOP/s x %s" % (src, bf16, ratio)


ATTN_KERNEL = {0: "attn_q8_kernel", 1: "attn_q8_kernel", 2: "attn_fp4_kernel"}
# the files each attention kernel is compiled from (its DRAM traffic depends on
# nothing else in the library)
ATTN_SOURCES = {0: ("attn_q8.cu", "attn_q8.cuh", "attn_q8x2.cuh", "attn_q8x2_64.cu", "sm103.cuh", "layout.h",
                    "launch.h"),
                1: ("attn_q8.cu", "attn_q8.cuh", "attn_q8x2.cuh", "attn_q8x2_64.cu", "sm103.cuh", "layout.h",
                    "launch.h"),
                2: ("attn_fp4.cu", "sm103.cuh", "layout.h", "launch.h")}


def read_traffic(key: str, mode: int = 0):
    """DRAM bytes per attention launch recorded from an ncu capture, or None when
    the kernel's sources changed since (lines: key kernel_hash bytes)."""
    path = os.path.join(ROOT, "profiles", "attn_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) == 3 and not line.startswith("#") and parts[0] == key and \
                parts[1] == kernel_hash(ATTN_SOURCES[mode]):
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi sampled every PERIOD_MS in the background; summary() keeps
    only the samples whose timestamps fall inside the timed window (none inside:
    the clock is reported as null)."""
    PERIOD_MS = 20
    FIELDS = "timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active," \
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None
        self.window = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def mark(self, t0: float, t1: float):
        """wall-clock bounds of the timed region"""
        self.window = (t0, t1)

    def __exit__(self, *a):
        time.sleep(0.1)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        import datetime
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append(dict(ts=ts, sm=float(parts[2]), smax=float(parts[3]), power=float(parts[4]),
                                 hw=parts[6], hwt=parts[7], swt=parts[8], swp=parts[9]))
            except ValueError:
                continue
        os.unlink(self.path)
        inside = [r for r in rows if self.window and self.window[0] <= r["ts"] <= self.window[1]]
        use = inside
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": len(rows), "samples_in_timed_region": 0,
                    "reasons": ["no sample inside the timed region"]}
        sms = sorted(r["sm"] for r in use)
        reasons = set()
        for r in use:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(r["smax"] for r in use),
                "samples": len(use), "samples_in_timed_region": len(inside),
                "power_w_max": max(r["power"] for r in use), "reasons": sorted(reasons)}


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of per-rank timings over all ranks (the slowest rank
    sets the job's time); the values themselves with one rank."""
    values = [float(v) for v in values]
    if dist is None:
        return values
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_tops(ops_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return ops_per_rank * world / (ms * 1e-3) / 1e12


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------------- reference arm
class OracleSample:
    """The oracle (as it stands) on a bounded sample of the workload: the
    pre-pass of some (batch, kv-head) groups and the attention rows of a spread
    of query rows of their heads, on all host cores."""

    def __init__(self, cfg, threads: int | None = None, groups: int = 1):
        import oracle
        from workload import make_inputs
        self.oracle = oracle
        self.cfg = cfg
        self.threads = threads or os.cpu_count() or 1
        g = max(1, min(cfg.Hkv, groups))
        # g kv-heads of batch 0 and their query heads
        self.sub = cfg.with_(B=1, Hq=(cfg.Hq // cfg.Hkv) * g, Hkv=g)
        self.q, self.k, self.v = make_inputs(self.sub)
        s = self.sub
        self.shape = (s.B, s.Hq, s.Hkv, s.N, s.M, s.d)

    def run(self, nrows: int):
        """Time the pre-pass and nrows attention rows; returns (TOPS, seconds, rows)."""
        import numpy as np
        s, o = self.sub, self.oracle
        t0 = time.perf_counter()
        qz = o.quantize(self.shape, s.mode, s.flags, s.bq, s.bk, self.q, self.k, self.v)
        tq = time.perf_counter() - t0
        # rows spread evenly over all query rows of the sample (causal rows see
        # about M/2 keys on average)
        rows = np.linspace(0, s.Hq * s.N - 1, nrows).astype(np.int64)
        t1 = time.perf_counter()
        o.parallel_attn_rows(self.shape, s.mode, s.flags, s.bq, s.bk, s.causal, s.sm_scale, self.q, self.k,
                             self.v, qz, rows, threads=self.threads)
        ta = time.perf_counter() - t1
        off = s.M - s.N
        pairs = sum(min(s.M, int(r) % s.N + off + 1) if s.causal else s.M for r in rows)
        # the literal metric counts half the pairs when causal: scale to it so the
        # GPU and CPU values share one unit
        lit_over_exact = self.cfg.ops / (4.0 * self.cfg.d * self.cfg.B * self.cfg.Hq * self.cfg.visible_pairs)
        # pre-pass share: its time prorated to the fraction of query rows done
        t_total = ta + tq * (len(rows) / (s.Hq * s.N))
        return 4.0 * s.d * pairs * lit_over_exact / t_total / 1e12, t_total, len(rows)

    @classmethod
    def calibrated(cls, cfg, budget_s: float):
        """A sample sized to about budget_s seconds of oracle work."""
        smp = cls(cfg)
        # two probes: the cost of a row from their difference, so the fixed part
        # of a run (thread start-up, the prorated pre-pass) does not count per row
        _, s1, n1 = smp.run(32)
        _, s2, n2 = smp.run(min(512, smp.sub.Hq * smp.sub.N))
        per_row = max((s2 - s1) / max(n2 - n1, 1), s2 / max(n2, 1) / 4, 1e-6)
        fixed = max(s1 - n1 * per_row, 0.0)
        want = int(max(32, (budget_s - fixed) / per_row))
        per_group = smp.sub.Hq * smp.sub.N
        if want > per_group and cfg.Hkv > 1:
            smp = cls(cfg, groups=-(-want // per_group))
        return smp, int(min(want, smp.sub.Hq * smp.sub.N))

    def describe(self, nrows: int) -> str:
        return ("oracle pre-pass of %d kv-head(s) (%d query heads, time prorated) + attention of %d query rows "
                "spread over them" % (self.sub.Hkv, self.sub.Hq, nrows))


def run_reference(args, cfg):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    per_step = max(1.0, min(args.ref_budget, 150.0 / (args.steps + args.warmup)))
    smp, nrows = OracleSample.calibrated(cfg, per_step)
    vals = []
    for i in range(args.warmup + args.steps):
        tops, secs, _ = smp.run(nrows)
        if i >= args.warmup:
            vals.append((tops, secs))
    tops = sum(v[0] for v in vals) / len(vals)
    out = {
        "impl": "reference", "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * sum(v[1] for v in vals) / len(vals), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg),
        "cpu_baseline": {"value": tops, "unit": "TOPS", "cores": smp.threads, "kind": "oracle",
                         "sample": smp.describe(nrows)},
        "e2e": {"value": tops, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# --------------------------------------------------------------------------- GPU arm
METRIC = "quantized attention TOPS (4*B*H*N*M*d/s, causal halved) and % of tensor peak"


def workload_config(cfg):
    return {"workload": cfg.name, "B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "N": cfg.N, "M": cfg.M, "d": cfg.d,
            "causal": cfg.causal, "quant_mode": ["int8_qk_fp8_pv", "fp8_qk_fp8_pv", "nvfp4", "sagebwd_int8"][cfg.mode],
            "flags": {"smooth_k": bool(cfg.flags & 1), "smooth_q": bool(cfg.flags & 2),
                      "smooth_v": bool(cfg.flags & 4), "p_direct": bool(cfg.flags & 8),
                      "q_per_token": bool(cfg.flags & 0x10)},
            "bq": cfg.bq, "bk": cfg.bk,
            "l2": "inputs larger than L2 (%.0f MB of bf16 Q/K/V per step), no flush" % (
                2.0 * cfg.d * (cfg.B * cfg.Hq * cfg.N + 2 * cfg.B * cfg.Hkv * cfg.M) / 1e6),
            "parallelism": "independent batch per GPU"}


def time_steps(sage, cfg, q, k, v, dev, stream, steps, warmup, barrier=lambda: None, sampler=None):
    """W warm-up steps, then K timed steps (pre-pass + attention) on inputs
    resident in HBM: CUDA events on the launching stream around the whole
    region and around each attention launch.  Returns (total ms, mean attention
    ms, device status)."""
    import torch
    shape = sage.shape_of(q, k)
    ws = sage.new_workspace(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, dev)
    o = torch.empty_like(q)

    def step(ev=None):
        sage.sage_quantize_qkv(q, k, v, cfg.mode, cfg.flags, cfg.bq, cfg.bk, workspace=ws, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        sage.sage_attn_fwd(ws, cfg.causal, cfg.sm_scale, out=o, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    assert sage.sage_read_status(ws) == (0, 0), "device status after warm-up (%s)" % cfg.name
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    w0 = time.time()
    t_start.record(stream)
    for i in range(steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if sampler is not None:
        sampler.mark(w0, time.time())
    barrier()
    total_ms = t_start.elapsed_time(t_end)
    attn_ms = sum(a.elapsed_time(b) for a, b in evs) / steps
    st = sage.sage_read_status(ws)
    del ws, o
    return total_ms, attn_ms, st


def roofline_of(cfg, attn_ms):
    """The attention kernel against the dense peak of its instruction mix."""
    bf16, _, _, src = peaks()
    peak, kinds = attention_peak(cfg.mode, bf16)
    # algorithmic work of one launch: 4 d flops per visible (query, key) pair
    algo_flops = 4.0 * cfg.d * cfg.B * cfg.Hq * cfg.visible_pairs
    achieved = algo_flops / (attn_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": read_traffic(cfg.name + "_bk%d" % cfg.bk, cfg.mode),
            "kernel": ATTN_KERNEL[cfg.mode] + " (sage_attn_fwd)", "instructions": kinds,
            "peak_source": peak_source(cfg.mode, src, bf16), "attn_ms": attn_ms,
            "flops_per_launch": algo_flops}


def bench_workload(sage, cfg, dev, stream, steps, warmup, local):
    """One workload timed on its own (same steps and warm-up as the headline),
    with its roofline, pre-pass time and the clocks seen while it ran."""
    from workload import make_inputs
    qh, kh, vh = make_inputs(cfg)
    q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
    del qh, kh, vh
    with ClockSampler(local) as clk:
        total_ms, attn_ms, st = time_steps(sage, cfg, q, k, v, dev, stream, steps, warmup, sampler=clk)
    ms = total_ms / steps
    return {"config": workload_config(cfg), "value": cfg.ops / (ms * 1e-3) / 1e12, "unit": "TOPS",
            "ms_per_step": ms, "attn_only_tops": cfg.ops / (attn_ms * 1e-3) / 1e12,
            "prepass_ms": ms - attn_ms, "roofline": roofline_of(cfg, attn_ms), "clocks": clk.summary(),
            "device_status": list(st)}


def bench_backward(sage, cfg, dev, stream, steps, warmup, local):
    """The SageBwd training step on one workload: the forward in the SageBwd
    mode (pre-pass + attention with its log-sum-exp), the backward's pre-pass
    (dO codes, D = rowsum(dO o O)) and the backward (dQ, dK, dV), each timed
    with CUDA events; the backward against the bf16 dense peak (all of its
    products run as kind::f16)."""
    import torch
    from workload import make_inputs
    qh, kh, vh = make_inputs(cfg)
    q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
    del qh, kh, vh
    gen = torch.Generator(device=dev).manual_seed(5)
    dout = torch.randn(q.shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    shape = sage.shape_of(q, k)
    ws = sage.new_workspace(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, dev)
    o = torch.empty_like(q)
    dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
    dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
    dv = torch.empty(k.shape, dtype=torch.float32, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps + warmup)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize(dev)
        w0 = time.time()
        for i in range(steps + warmup):
            if i == warmup:
                torch.cuda.synchronize(dev)
                w0 = time.time()
            ev[i][0].record(stream)
            sage.sage_quantize_qkv(q, k, v, cfg.mode, cfg.flags, cfg.bq, cfg.bk, workspace=ws, stream=stream)
            sage.sage_attn_fwd(ws, cfg.causal, cfg.sm_scale, out=o, stream=stream)
            ev[i][1].record(stream)
            sage.sage_bwd_prepare(ws, o, dout, stream=stream)
            ev[i][2].record(stream)
            sage.sage_attn_bwd(ws, cfg.causal, cfg.sm_scale, v, dout, dq=dq, dk=dk, dv=dv, stream=stream)
            ev[i][3].record(stream)
        torch.cuda.synchronize(dev)
        clk.mark(w0, time.time())
    st = sage.sage_read_status(ws)
    t = ev[warmup:]
    fwd = sum(a.elapsed_time(b) for a, b, _, _ in t) / steps
    prep = sum(b.elapsed_time(c) for _, b, c, _ in t) / steps
    bwd = sum(c.elapsed_time(d) for _, _, c, d in t) / steps
    bf16, _, _, src = peaks()
    pairs = cfg.B * cfg.Hq * cfg.visible_pairs
    algo = 10.0 * cfg.d * pairs        # five products of 2 d flops per visible pair
    achieved = algo / (bwd * 1e-3) / 1e12
    return {"config": workload_config(cfg), "fwd_ms": fwd, "bwd_prepare_ms": prep, "bwd_ms": bwd,
            "step_ms": fwd + prep + bwd,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                         "frac": achieved / bf16, "traffic": None,
                         "kernel": "bwd_dkdv_kernel + bwd_dq_kernel (sage_attn_bwd)",
                         "instructions": "kind::f16 (INT8 codes as fp16, bf16 dO V^T)",
                         "peak_source": "%s bf16 burst %.1f TFLOP/s" % (src, bf16),
                         "flops_per_launch": algo,
                         "flops_executed_per_launch": 14.0 * cfg.d * pairs,
                         "note": "algorithmic: 5 products; the two kernels run 7 (S and dP are formed in both)"},
            "clocks": clk.summary(), "device_status": list(st)}


def ablation_variants(cfg):
    """The method's switches on one workload (the pages' technique-overhead and
    granularity tables): (name, config, SAGE_PINGPONG value)."""
    out = [("as configured", cfg, None),
           ("Q smoothing %s" % ("off" if cfg.flags & 2 else "on"), cfg.with_(flags=cfg.flags ^ 2), None),
           ("V smoothing %s" % ("off" if cfg.flags & 4 else "on"), cfg.with_(flags=cfg.flags ^ 4), None)]
    if cfg.mode in (0, 1):
        out.append(("per-token Q scales", cfg.with_(flags=cfg.flags | 0x10), None))
        out.append(("tiles in turn", cfg, "1"))
    if cfg.mode == 0:
        out.append(("E4M3 Q/K", cfg.with_(mode=1), None))
        out.append(("SageBwd forward (bk 64)", cfg.with_(mode=3, bk=64), None))
    if cfg.mode == 2:
        out.append(("direct P~", cfg.with_(flags=cfg.flags | 8), None))
        out.append(("tiles in turn", cfg, "1"))
    return out


def ablation_rows(sage, cfg, dev, stream, steps, warmup):
    """Each variant timed like the bench on the same inputs: step (pre-pass +
    attention) and attention alone, in ms."""
    from workload import make_inputs
    qh, kh, vh = make_inputs(cfg)
    q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
    del qh, kh, vh
    rows = []
    try:
        for name, c, ping in ablation_variants(cfg):
            if ping:
                os.environ["SAGE_PINGPONG"] = ping
            else:
                os.environ.pop("SAGE_PINGPONG", None)
            total_ms, attn_ms, st = time_steps(sage, c, q, k, v, dev, stream, steps, warmup)
            rows.append({"variant": name, "mode": c.mode, "flags": c.flags, "bk": c.bk,
                         "step_ms": total_ms / steps, "attn_ms": attn_ms, "device_status": list(st)})
    finally:
        os.environ.pop("SAGE_PINGPONG", None)
    base = rows[0]["attn_ms"]
    for r in rows:
        r["attn_vs_configured"] = r["attn_ms"] / base
    return rows


def run_gpu(args, cfg):
    import torch

    import bit_quantized_attention_gb300 as sage
    from workload import CONFIGS, make_inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    def barrier():
        if pg is not None:
            pg.barrier()

    qh, kh, vh = make_inputs(cfg)
    q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
    shape = sage.shape_of(q, k)
    stream = torch.cuda.current_stream(dev)
    with ClockSampler(local) as clk:
        total_ms, attn_ms, code = time_steps(sage, cfg, q, k, v, dev, stream, args.steps, args.warmup,
                                             barrier=barrier, sampler=clk)
    clocks = clk.summary()
    total_ms, attn_ms = max_over_ranks([total_ms, attn_ms], pg, dev)
    ms_per_step = total_ms / args.steps
    value = job_tops(cfg.ops, world, ms_per_step)
    del q, k, v

    # ---- e2e through the C ABI on host buffers (pinned), copies inside the timed region
    q_pin, k_pin, v_pin = qh.pin_memory(), kh.pin_memory(), vh.pin_memory()
    o_pin = torch.empty_like(qh).pin_memory()
    nbytes = sage.sage_host_buffer_bytes(shape, cfg.mode, cfg.bq, cfg.bk)
    raw = torch.empty(nbytes + 1024, dtype=torch.uint8, device=dev)
    dev_buf = raw[(-raw.data_ptr()) % 1024:][:nbytes]
    for _ in range(max(1, args.warmup // 2)):
        sage.sage_attn_host(shape, cfg.causal, cfg.sm_scale, cfg.mode, cfg.flags, cfg.bq, cfg.bk,
                            q_pin, k_pin, v_pin, o_pin, dev_buf, stream=stream)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        sage.sage_attn_host(shape, cfg.causal, cfg.sm_scale, cfg.mode, cfg.flags, cfg.bq, cfg.bk,
                            q_pin, k_pin, v_pin, o_pin, dev_buf, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / args.steps
    (e2e_ms,) = max_over_ranks([e2e_ms], pg, dev)
    e2e_val = job_tops(cfg.ops, world, e2e_ms)
    h2d = (qh.numel() + kh.numel() + vh.numel()) * 2
    d2h = qh.numel() * 2
    del raw, dev_buf, q_pin, k_pin, v_pin, o_pin

    out = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ["int8/e4m3", "e4m3", "e2m1", "int8"][cfg.mode], "data": "synthetic",
        "config": workload_config(cfg),
        "e2e": {"value": e2e_val, "unit": "TOPS", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "roofline": roofline_of(cfg, attn_ms),
        "attn_only_tops": cfg.ops / (attn_ms * 1e-3) / 1e12,
        "prepass_ms": ms_per_step - attn_ms,
        "clocks": clocks,
        "device_status": list(code),
    }
    # the other workloads, each timed on its own in this process (rank 0 at N = 1:
    # they describe the kernels, not the job)
    if rank == 0 and world == 1 and args.per_workload:
        per = {}
        for name in args.per_workload.split(","):
            if name and name != cfg.name:
                c = CONFIGS[name].with_(bk=args.bk) if args.bk else CONFIGS[name]
                per[name] = bench_workload(sage, c, dev, stream, args.steps, args.warmup, local)
        out["per_workload"] = per
    if rank == 0 and world == 1 and args.backward:
        c = CONFIGS[args.backward].with_(mode=3, bk=64)
        out["backward"] = bench_backward(sage, c, dev, stream, args.steps, args.warmup, local)
    if rank == 0 and world == 1 and args.ablations:
        abl = {}
        for name in args.ablations.split(","):
            if name:
                c = CONFIGS[name].with_(bk=args.bk) if args.bk else CONFIGS[name]
                abl[name] = ablation_rows(sage, c, dev, stream, args.steps, args.warmup)
        out["ablation"] = abl
    if rank == 0 and world == 1 and not args.no_cpu_baseline:  # the CPU baseline: rank 0 at N = 1 only
        smp, nrows = OracleSample.calibrated(cfg, args.ref_budget)
        tops, secs, _ = smp.run(nrows)
        out["cpu_baseline"] = {"value": tops, "unit": "TOPS", "cores": smp.threads, "kind": "oracle",
                               "sample": smp.describe(nrows), "seconds": secs,
                               "single_thread": single_thread_baseline(cfg, args.ref_budget / 3)}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def run_ablation(args, cfg):
    """The method's switches on one workload as a markdown table (no JSON line):
    Q / V smoothing on and off, per-token Q scales, E4M3 Q/K, direct P~
    (NVFP4), the tiles-in-turn softmax schedule, and the SageBwd forward's
    quantizers on the same inputs."""
    import torch

    import bit_quantized_attention_gb300 as sage

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rows = ablation_rows(sage, cfg, dev, torch.cuda.current_stream(dev), args.steps, args.warmup)
    print("| variant | mode | flags | bk | step ms | attention ms | attention vs as configured | status |")
    print("|---|---|---|---|---|---|---|---|")
    for r in rows:
        print("| %s | %d | 0x%x | %d | %.3f | %.3f | %.3f | %s |" % (
            r["variant"], r["mode"], r["flags"], r["bk"], r["step_ms"], r["attn_ms"], r["attn_vs_configured"],
            tuple(r["device_status"])))


def single_thread_baseline(cfg, budget_s: float):
    """The oracle on one host thread over a smaller sample of the same workload,
    extrapolated to the metric's unit (TOPS)."""
    smp = OracleSample(cfg, threads=1)
    _, s1, n1 = smp.run(8)
    n = int(max(8, min(smp.sub.Hq * smp.sub.N, n1 * budget_s / max(s1, 1e-6))))
    tops, secs, rows = smp.run(n)
    return {"value": tops, "unit": "TOPS", "cores": 1, "seconds": secs,
            "sample": smp.describe(rows) + " on one thread (extrapolated to the whole workload by its row count)"}


def kernel_hash(files=None) -> str:
    """Hash of CUDA/C++ sources' code (the given csrc files, else all of them):
    comments dropped and whitespace runs collapsed, so an edit to the
    documentation does not void a measurement while any change to the code does."""
    import hashlib
    import re
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "bit_quantized_attention_gb300", "csrc")
    for f in sorted(files if files is not None else os.listdir(csrc)):
        if not f.endswith((".cu", ".cuh", ".h")):
            continue
        text = open(os.path.join(ROOT, "bit_quantized_attention_gb300", "csrc", f), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(f.encode() + b"\0" + " ".join(text.split()).encode() + b"\0")
    return h.hexdigest()[:12]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="video",
                    help="the headline workload (video: the largest non-causal INT8 / FP8 one)")
    ap.add_argument("--per-workload", default="llm_prefill,chunked_gqa,nvfp4",
                    help="other workloads timed in the same run, each with its own roofline ('' for none)")
    ap.add_argument("--backward", default="llm_prefill",
                    help="workload whose SageBwd forward + backward is timed on the JSON line ('' for none)")
    ap.add_argument("--ablations", default="video,nvfp4",
                    help="workloads whose switch ablations go on the JSON line ('' for none)")
    ap.add_argument("--bk", type=int, default=128, help="key tile = K scale block (the workload leaves it open)")
    ap.add_argument("--impl", default="sage", choices=["sage", "reference"])
    ap.add_argument("--ref-budget", type=float, default=15.0, help="seconds of oracle work per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="override B (smaller cases for profiling)")
    ap.add_argument("--heads", type=int, default=0, help="override Hq (Hkv scaled to keep the group size)")
    ap.add_argument("--ablation", action="store_true",
                    help="time the method's switches on the workload and print a table (no JSON line)")
    ap.add_argument("--flags", type=lambda x: int(x, 0), default=None,
                    help="override the workload's flags (ablations: 1 smooth K, 2 smooth Q, 4 smooth V, "
                         "8 direct P~ in the NVFP4 mode, 0x10 per-token Q scales)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from workload import CONFIGS
    cfg = CONFIGS[args.workload]
    if args.bk:
        cfg = cfg.with_(bk=args.bk)
    if args.batch:
        cfg = cfg.with_(B=args.batch)
    if args.flags is not None:
        cfg = cfg.with_(flags=args.flags)
    if args.heads:
        g = cfg.Hq // cfg.Hkv
        if args.heads % g:
            ap.error("--heads must be a multiple of the workload's group size %d" % g)
        cfg = cfg.with_(Hq=args.heads, Hkv=args.heads // g)
    if args.ablation:
        import __graft_entry__
        __graft_entry__.build()
        run_ablation(args, cfg)
    elif args.impl == "reference":
        run_reference(args, cfg)
    else:
        import __graft_entry__
        __graft_entry__.build()
        run_gpu(args, cfg)


if __name__ == "__main__":
    main()
