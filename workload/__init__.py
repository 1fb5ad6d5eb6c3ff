"""Seeded synthetic inputs for the quantized-attention hot path.

This package is shared by the tests, the oracle driver and ``bench.py``.  It
holds only shapes and random draws: none of the method's arithmetic (means,
scales, quantizers, softmax) lives here, so neither the oracle nor the CUDA
path can lean on the other through it.
"""
from .configs import CONFIGS, Config, config_by_name  # noqa: F401
from .gen import make_inputs, make_qkv_float  # noqa: F401
