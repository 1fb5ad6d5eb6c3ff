"""Operand layout of the backward's MMAs on sm_103a: a B operand read
MN-major out of a [K rows][N] tile stored in the 128-byte swizzled chunks of
a K-major load (the backward reduces over keys or queries of tiles loaded as
[tokens][d] rows).  The probe kernel is test code
(tests/gpu_probes/mn_major_probe.cu), built here with nvcc for sm_103a; small
integer operands make every product and sum exact in fp32."""
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
    out = str(tmp_path_factory.mktemp("mnprobe") / "mn_probe.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    "-I", CSRC, "-o", out, os.path.join(ROOT, "tests", "gpu_probes", "mn_major_probe.cu")],
                   check=True)
    lib = C.CDLL(out)
    lib.mn_probe.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p]
    lib.mn_probe.restype = C.c_int
    return lib


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_mn_major_b_operand(probe, mode):
    rng = np.random.default_rng(11 + mode)
    a = rng.integers(-8, 9, size=(128, 128)).astype(np.float16)
    b = rng.integers(-8, 9, size=(128, 128)).astype(np.float16)
    dev = torch.device("cuda")
    ta = torch.from_numpy(a.view(np.int16)).to(dev)
    tb = torch.from_numpy(b.view(np.int16)).to(dev)
    out = torch.full((128, 128), float("nan"), dtype=torch.float32, device=dev)
    st = torch.zeros(2, dtype=torch.int32, device=dev)
    assert probe.mn_probe(ta.data_ptr(), tb.data_ptr(), out.data_ptr(), mode, st.data_ptr()) == 0
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, 0]
    got = out.cpu().numpy()
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    if mode == 0:
        want = a64 @ b64
    elif mode == 1:
        want = a64[:, 64:] @ b64[64:, :]
    else:
        want = a64[:, :64] @ b64[:64, :64]
        got = got[:, :64]
    assert np.array_equal(got, want.astype(np.float32)), np.argwhere(got != want)[:5]
