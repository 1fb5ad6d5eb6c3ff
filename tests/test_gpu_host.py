"""The end-to-end call on host buffers (sage_attn_host): chunked by kv heads
and pipelined over three streams, it must give bit for bit what the device
calls give on the whole request (each chunk is an independent problem with
the same means, scales and tiles), for every mode, with GQA, causal masks and
ragged lengths; its status word must read clean."""
import numpy as np
import pytest
import torch

from test_gpu_quantize import _small
from workload import make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    _small("host_video_like", B=2, Hq=6, Hkv=6, N=300, M=300, flags=7, d=64, bk=128),
    _small("host_gqa_causal", B=1, Hq=8, Hkv=2, N=200, M=500, causal=True, flags=3, d=128, bk=128),
    _small("host_bk64_many_chunks", B=3, Hq=12, Hkv=4, N=130, M=257, flags=5, d=64, bk=64),
    _small("host_fp8", mode=1, B=2, Hq=4, Hkv=4, N=256, M=256, flags=1, d=128, bk=128),
    _small("host_nvfp4", mode=2, B=2, Hq=4, Hkv=4, N=256, M=384, flags=1, d=128, bk=128),
    # 96 heads x 128 query blocks = 12288 blocks: the largest chunk count (24 chunks of 4 kv heads)
    _small("host_24_chunks", B=1, Hq=96, Hkv=96, N=16384, M=16384, flags=7, d=64, bk=128),
]


@pytest.fixture(scope="module")
def sage():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_quantized_attention_gb300 as s
    return s


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_host_call_matches_device_calls(sage, cfg):
    q, k, v = make_inputs(cfg)
    dev = torch.device("cuda")
    want = sage.sage_attn_fwd(sage.sage_quantize_qkv(q.to(dev), k.to(dev), v.to(dev), cfg.mode, cfg.flags, cfg.bq,
                                                     cfg.bk), cfg.causal, cfg.sm_scale)
    shape = sage.shape_of(q, k)
    n = sage.sage_host_buffer_bytes(shape, cfg.mode, cfg.bq, cfg.bk)
    assert n > 0
    raw = torch.full((n + 1024,), 0xFF, dtype=torch.uint8, device=dev)
    buf = raw[(-raw.data_ptr()) % 1024:][:n]
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    op = torch.zeros_like(q).pin_memory()
    for _ in range(2):  # twice: the second call reuses the internal streams and the buffer
        op.zero_()
        sage.sage_attn_host(shape, cfg.causal, cfg.sm_scale, cfg.mode, cfg.flags, cfg.bq, cfg.bk, qp, kp, vp, op, buf)
        torch.cuda.synchronize()
        assert sage.sage_host_status(buf) == (0, 0)
        assert np.array_equal(op.view(torch.int16).numpy(), want.cpu().view(torch.int16).numpy())
