"""The two library calls of a step, captured into one CUDA graph and replayed:
every launch of the path must be capturable (no host synchronisation, no
allocation inside the calls), and the replays must give the eager result bit
for bit.  The first eager call runs before the capture: it performs the
one-time host-side look-ups (function attributes, the SM count)."""
import numpy as np
import pytest
import torch

from test_gpu_quantize import _small
from workload import make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    _small("graph_int8_smooth_causal", N=300, M=500, causal=True, flags=7, d=128, bk=128),
    _small("graph_fp8_d64", mode=1, N=256, M=256, flags=1, d=64, bk=64),
    _small("graph_nvfp4", mode=2, N=256, M=384, flags=3, d=128, bk=128),
]


@pytest.fixture(scope="module")
def sage():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_quantized_attention_gb300 as s
    return s


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_step_replays_from_a_cuda_graph(sage, cfg):
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_inputs(cfg))
    shape = sage.shape_of(q, k)
    ws = sage.new_workspace(shape, cfg.mode, cfg.flags, cfg.bq, cfg.bk, dev)
    o = torch.empty_like(q)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):  # eager, off the default stream (capture needs one)
        sage.sage_quantize_qkv(q, k, v, cfg.mode, cfg.flags, cfg.bq, cfg.bk, workspace=ws, stream=side)
        sage.sage_attn_fwd(ws, cfg.causal, cfg.sm_scale, out=o, stream=side)
    torch.cuda.synchronize(dev)
    eager = o.clone()
    assert sage.sage_read_status(ws) == (0, 0)
    o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        sage.sage_quantize_qkv(q, k, v, cfg.mode, cfg.flags, cfg.bq, cfg.bk, workspace=ws, stream=side)
        sage.sage_attn_fwd(ws, cfg.causal, cfg.sm_scale, out=o, stream=side)
    for _ in range(3):
        o.zero_()
        g.replay()
        torch.cuda.synchronize(dev)
        assert torch.equal(o, eager)
    assert sage.sage_read_status(ws) == (0, 0)
    assert np.isfinite(eager.float().cpu().numpy()).all()
