"""Host logic of bench.py on the CPU: the work counts behind the metric and the
roofline, the source hash that keys recorded counters, the reference arm's JSON
line, and the multi-rank reduction (world size 2 over gloo)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workload import CONFIGS  # noqa: E402


def _brute_pairs(N, M, causal):
    off = M - N
    return sum(sum(1 for j in range(M) if (not causal) or j <= i + off) for i in range(N))


@pytest.mark.parametrize("N,M,causal", [(7, 7, True), (5, 13, True), (9, 9, False), (1, 1, True), (3, 300, True)])
def test_visible_pairs_match_brute_force(N, M, causal):
    cfg = CONFIGS["tiny"].with_(N=N, M=M, causal=causal)
    assert cfg.visible_pairs == _brute_pairs(N, M, causal)


def test_literal_ops_halved_only_when_causal():
    c = CONFIGS["llm_prefill"]
    full = 4.0 * c.B * c.Hq * c.N * c.M * c.d
    assert c.ops == full / 2
    assert c.with_(causal=False).ops == full


def _fake_tree(tmp_path, text):
    d = tmp_path / "bit_quantized_attention_gb300" / "csrc"
    d.mkdir(parents=True, exist_ok=True)
    (d / "k.cu").write_text(text)
    return str(tmp_path)


def test_kernel_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    code = "int f(int x) {\n  return x + 1;  // one more\n}\n/* block\n comment */\n"
    monkeypatch.setattr(bench, "ROOT", _fake_tree(tmp_path / "a", code))
    h0 = bench.kernel_hash()
    monkeypatch.setattr(bench, "ROOT", _fake_tree(tmp_path / "b", code.replace("one more", "plus one") + "// x\n"))
    assert bench.kernel_hash() == h0
    monkeypatch.setattr(bench, "ROOT", _fake_tree(tmp_path / "c", code.replace("x + 1", "x + 2")))
    assert bench.kernel_hash() != h0


def test_traffic_record_needs_the_kernels_current_sources(tmp_path, monkeypatch):
    d = tmp_path / "bit_quantized_attention_gb300" / "csrc"
    d.mkdir(parents=True)
    for f in set(bench.ATTN_SOURCES[0]) | set(bench.ATTN_SOURCES[2]) | {"api.cu"}:
        (d / f).write_text("int %s_x;\n" % f.replace(".", "_"))
    root = str(tmp_path)
    monkeypatch.setattr(bench, "ROOT", root)
    os.makedirs(os.path.join(root, "profiles"))
    with open(os.path.join(root, "profiles", "attn_traffic.txt"), "w") as f:
        f.write("# comment\nwl_bk128 %s 123\nwl_bk64 000000000000 456\n" % bench.kernel_hash(bench.ATTN_SOURCES[0]))
    assert bench.read_traffic("wl_bk128", 0) == 123.0
    assert bench.read_traffic("wl_bk64", 0) is None
    assert bench.read_traffic("other", 0) is None
    assert bench.read_traffic("wl_bk128", 2) is None          # the NVFP4 kernel's files differ
    (d / "api.cu").write_text("int changed;\n")             # not a file the kernel is built from
    assert bench.read_traffic("wl_bk128", 0) == 123.0
    (d / "attn_q8.cu").write_text("int changed;\n")
    assert bench.read_traffic("wl_bk128", 0) is None


def test_job_tops_is_all_ranks_over_the_slowest():
    assert bench.job_tops(1e12, 1, 1000.0) == pytest.approx(1.0)
    assert bench.job_tops(1e12, 4, 500.0) == pytest.approx(8.0)
    assert bench.max_over_ranks([1.5, 2.0]) == [1.5, 2.0]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as b
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 3.0 - rank]  # rank 1 slower on the first, faster on the second
        got = b.max_over_ranks(mine, dist, "cpu")
        assert got == [10.0 + world - 1, 3.0], got
        assert b.job_tops(2e12, world, got[0]) == pytest.approx(2e12 * world / (got[0] * 1e-3) / 1e12)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_world_size_two_gloo():
    import torch.multiprocessing as mp
    mp.start_processes(_rank_main, args=(2, _free_port()), nprocs=2, join=True, start_method="spawn")


def _run_bench(args, env_extra=None, timeout=300):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_json_line():
    r = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3",
                    "--ref-budget", "0.5"])
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 1 and line["warmup"] == 3
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"] and line["config"]["workload"] == "tiny"


def test_reference_arm_other_ranks_do_no_work():
    r = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_warmup_below_three_rejected():
    r = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "2"])
    assert r.returncode != 0
