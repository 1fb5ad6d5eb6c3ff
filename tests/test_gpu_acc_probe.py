"""The accumulator-precision probe of the SageAttention2 summary, repeated on
sm_103a: does the E4M3 tensor-core MMA (kind::f8f6f4, the P~V product of the
INT8 / FP8 kernel) keep FP32 in its accumulator?  The probe kernel is test code
(tests/gpu_probes/acc_probe.cu), built here with nvcc for sm_103a."""
import ctypes as C
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_quantized_attention_gb300", "csrc")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("probe") / "acc_probe.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    "-I", CSRC, "-o", out, os.path.join(ROOT, "tests", "gpu_probes", "acc_probe.cu")], check=True)
    lib = C.CDLL(out)
    lib.acc_probe.argtypes = [C.c_void_p] * 5
    lib.acc_probe.restype = C.c_int
    return lib


def run(probe, a, b, d0):
    dev = torch.device("cuda")
    ta = torch.from_numpy(a).to(dev)
    tb = torch.from_numpy(b).to(dev)
    td = torch.from_numpy(d0).to(dev)
    out = torch.full((128, 64), float("nan"), dtype=torch.float32, device=dev)
    st = torch.zeros(2, dtype=torch.int32, device=dev)
    assert probe.acc_probe(ta.data_ptr(), tb.data_ptr(), td.data_ptr(), out.data_ptr(), st.data_ptr()) == 0
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, 0]
    return out.cpu().numpy()


def test_zero_products_return_d_unchanged(probe):
    rng = np.random.default_rng(0)
    mant = rng.integers(0, 1 << 23, size=(128, 64), dtype=np.uint32)
    expo = rng.integers(100, 150, size=(128, 64), dtype=np.uint32)
    sign = rng.integers(0, 2, size=(128, 64), dtype=np.uint32)
    d0 = ((sign << 31) | (expo << 23) | mant).view(np.float32)
    got = run(probe, np.zeros((128, 128), np.uint8), np.zeros((64, 128), np.uint8), d0)
    assert np.array_equal(got.view(np.uint32), d0.view(np.uint32))


def test_small_products_land_in_fp32(probe):
    """A[m][0] = 2^-9 (E4M3 code 0x01), B[n][0] = 2^-(k-9): D = 1 + 2^-k for k in
    10..18, exact in FP32 (FP22, 13 mantissa bits, would lose every k > 13)."""
    a = np.zeros((128, 128), np.uint8)
    a[:, 0] = 0x01                                   # 2^-9, the smallest E4M3 subnormal
    b = np.zeros((64, 128), np.uint8)
    ks = 10 + np.arange(64) % 9                      # k = 10 .. 18
    for n, k in enumerate(ks):
        j = int(k) - 9                               # B = 2^-j, j = 1 .. 9
        b[n, 0] = (7 - j) << 3 if j <= 6 else 1 << (9 - j)   # normal 2^(e-7), or subnormal m 2^-9
    d0 = np.ones((128, 64), np.float32)
    got = run(probe, a, b, d0)
    want = (1.0 + 2.0 ** -ks.astype(np.float64)).astype(np.float32)
    exact = [bool(np.all(got[:, n] == want[n])) for n in range(64)]
    kept = {int(k): all(e for e, kk in zip(exact, ks) if kk == k) for k in sorted(set(ks.tolist()))}
    assert all(kept.values()), kept
