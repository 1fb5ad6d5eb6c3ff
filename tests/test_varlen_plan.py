"""The packed-sequence plan (host code in csrc/layout.h), compiled with the
host C++ compiler alone and checked against its definition: one work item per
query block of every sequence and head, each exactly once, longest first (the
number of key tiles a block visits); the sequence table is the cu_seqlens
differences and offsets; the tables sit after the batched regions.  CPU only."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_quantized_attention_gb300", "csrc")

HARNESS = r"""
#include "layout.h"
#include <cstdio>
#include <vector>
int main() {
  int nseq, Hq, Hkv, d, mode, bq, bk, causal;
  if (scanf("%d %d %d %d %d %d %d %d", &nseq, &Hq, &Hkv, &d, &mode, &bq, &bk, &causal) != 8) return 2;
  std::vector<int> cq(nseq + 1), ck(nseq + 1);
  for (int i = 0; i <= nseq; ++i) scanf("%d", &cq[i]);
  for (int i = 0; i <= nseq; ++i) scanf("%d", &ck[i]);
  sage::VarlenPlan P;
  const sage_status st = sage::plan_varlen(nseq, cq.data(), ck.data(), Hq, Hkv, d, mode, bq, bk, causal, &P);
  printf("status %d\n", (int)st);
  if (st != SAGE_OK) return 0;
  printf("shape %d %d %d %d %d %d\n", P.shape.B, P.shape.Hq, P.shape.Hkv, P.shape.N, P.shape.M, P.shape.d);
  printf("layout %zu %d %zu %zu %zu\n", P.L.total, P.L.Tm, P.seq_off, P.item_off, P.total);
  for (const auto &s : P.seqs) printf("seq %d %d %d %d\n", s.N, s.M, s.q0, s.k0);
  for (int c : P.item_codes) printf("item %d\n", c);
  return 0;
}
"""


@pytest.fixture(scope="module")
def plan_bin(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("plan")
    src = d / "plan.cpp"
    src.write_text(HARNESS)
    exe = d / "plan"
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, "-o", str(exe), str(src)], check=True)
    return str(exe)


def run_plan(exe, cq, ck, Hq=4, Hkv=2, d=64, mode=0, bq=128, bk=64, causal=0):
    inp = " ".join(map(str, [len(cq) - 1, Hq, Hkv, d, mode, bq, bk, causal] + list(cq) + list(ck)))
    out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout.split("\n")
    res = {"seqs": [], "items": []}
    for line in out:
        f = line.split()
        if not f:
            continue
        if f[0] == "status":
            res["status"] = int(f[1])
        elif f[0] == "shape":
            res["shape"] = tuple(map(int, f[1:]))
        elif f[0] == "layout":
            res["layout"] = tuple(map(int, f[1:]))
        elif f[0] == "seq":
            res["seqs"].append(tuple(map(int, f[1:])))
        elif f[0] == "item":
            res["items"].append(int(f[1]))
    return res


def tiles(n, m, i, bk, causal):
    """key tiles query block i of a sequence with n queries, m keys visits"""
    tn = -(-m // bk)
    if not causal:
        return tn
    last_row = min(n, i * 128 + 128) - 1
    return min(tn, (last_row + m - n) // bk + 1)


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("bk", [64, 128])
def test_plan_matches_definition(plan_bin, causal, bk):
    cq = [0, 100, 100, 400, 401, 1000]
    ck = [0, 150, 160, 700, 702, 1600]
    Hq, Hkv = 4, 2
    r = run_plan(plan_bin, cq, ck, Hq=Hq, Hkv=Hkv, bk=bk, causal=causal)
    assert r["status"] == 0
    lq = [b - a for a, b in zip(cq, cq[1:])]
    lk = [b - a for a, b in zip(ck, ck[1:])]
    assert r["shape"] == (5, Hq, Hkv, max(lq), max(lk), 64)
    assert r["seqs"] == [(lq[s], lk[s], cq[s], ck[s]) for s in range(5)]
    total_ws, Tm, seq_off, item_off, total = r["layout"]
    assert Tm == -(-max(lq) // 128)
    assert seq_off == total_ws and item_off % 1024 == 0 and item_off >= seq_off + 16 * 5
    assert total % 1024 == 0 and total >= item_off + 4 * len(r["items"])
    want = {}
    for s in range(5):
        for h in range(Hq):
            for i in range(-(-lq[s] // 128)):
                want[(s * Hq + h) * Tm + i] = tiles(lq[s], lk[s], i, bk, causal)
    assert sorted(r["items"]) == sorted(want)                     # each block exactly once
    t = [want[c] for c in r["items"]]
    assert t == sorted(t, reverse=True)                             # longest first


@pytest.mark.parametrize("cq,ck,causal,status", [
    ([1, 5], [0, 5], 0, 1),            # must start at 0
    ([0, 5, 3], [0, 5, 9], 0, 1),      # decreasing
    ([0, 5], [0, 0], 0, 1),            # queries without keys
    ([0, 0, 0], [0, 3, 9], 0, 1),      # no queries anywhere
    ([0, 9], [0, 5], 1, 2),            # causal with more queries than keys
    ([0, 9], [0, 5], 0, 0),            # the same without the mask is fine
])
def test_plan_rejects(plan_bin, cq, ck, causal, status):
    assert run_plan(plan_bin, cq, ck, causal=causal)["status"] == status
