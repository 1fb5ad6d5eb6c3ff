"""The five workloads the quantized-attention path is measured and checked on.

Shapes and value structure follow the pages' benchmark protocol (batch, heads,
Gaussian inputs, head dims 64/128; SageAttention2 summary §5 "Generation
budget"; SageAttention3 summary §5) and the LLM-prefill / video-diffusion /
chunked-prefill / NVFP4 cases named for this path.  Nothing here computes the
method: it only names sizes, modes and the recipe used by ``workload.gen``.

Mode numbers and flag bits are written out here as plain integers so this
module imports nothing from the product or from the oracle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

# quant_mode values (same meaning on both sides of the check)
MODE_Q8_PV8 = 0     # INT8 per-block Q/K, FP8 E4M3 P~ (scale 1/448) and per-channel FP8 V
MODE_QF8_PV8 = 1    # FP8 E4M3 per-block Q/K, FP8 P~ / V as above
MODE_NVFP4 = 2      # E2M1 in 1x16 blocks with E4M3 scales, two-level P~

# flag bits
SMOOTH_K = 1
SMOOTH_Q = 2
SMOOTH_V = 4


@dataclass(frozen=True)
class Config:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    M: int
    d: int
    causal: bool
    sm_scale: float
    mode: int
    flags: int
    bq: int = 128
    bk: int = 64
    seed: int = 0
    # value structure (see gen.py)
    k_fixed_channels: tuple = ()        # channels shifted by +k_fixed_shift for all tokens
    k_fixed_shift: float = 0.0
    k_offset_std: float = 0.0            # per-(b, head, channel) offset shared by all tokens
    k_outliers: int = 0                  # channels (drawn once from the seed) shifted by +k_outlier_shift
    k_outlier_shift: float = 0.0
    q_offset_std: float = 0.0            # per-(b, head, channel) offset shared by all tokens
    q_block_shift_std: float = 0.0       # per-(b, head, 64-token block, channel) shift
    q_block_len: int = 64
    v_bias_std: float = 0.0              # per-(b, head, channel) bias
    v_student_t: float = 0.0             # >0: V ~ Student-t with this many degrees of freedom
    v_clip: float = 0.0                  # >0: clip V to +-v_clip
    q_from_k_noise: float = 0.0          # >0: each query row is a random key row of its kv head
                                         # (before K's offsets) plus N(0, noise^2): peaked rows
    note: str = ""

    @property
    def ops(self) -> float:
        """The literal throughput numerator: 4*B*H*N*M*d, halved when causal."""
        v = 4.0 * self.B * self.Hq * self.N * self.M * self.d
        return v / 2 if self.causal else v

    @property
    def visible_pairs(self) -> int:
        """Exact number of (query, key) pairs the mask leaves visible, per (b, head)."""
        if not self.causal:
            return self.N * self.M
        off = self.M - self.N
        # query i sees keys 0 .. i + off (bottom-right alignment), capped at M
        tot = 0
        for i in range(self.N):
            tot += max(0, min(self.M, i + off + 1))
        return tot

    def with_(self, **kw) -> "Config":
        return replace(self, **kw)


CONFIGS = {
    "tiny": Config(
        name="tiny", B=1, Hq=2, Hkv=2, N=256, M=256, d=64, causal=False,
        sm_scale=1.0 / 8.0, mode=MODE_Q8_PV8, flags=SMOOTH_K, bq=128, bk=64, seed=0,
        k_fixed_channels=(3, 17), k_fixed_shift=10.0,
        note="tiny correctness case: N(0,1), K channels 3 and 17 shifted by +10"),
    "llm_prefill": Config(
        name="llm_prefill", B=4, Hq=32, Hkv=32, N=4096, M=4096, d=128, causal=True,
        sm_scale=1.0 / math.sqrt(128), mode=MODE_Q8_PV8, flags=SMOOTH_K, bq=128, bk=64,
        seed=1, k_offset_std=3.0, k_outliers=4, k_outlier_shift=20.0,
        note="LLM prefill: K offsets N(0,3^2) per channel + 4 outlier channels at +20"),
    "video": Config(
        name="video", B=2, Hq=48, Hkv=48, N=17776, M=17776, d=64, causal=False,
        sm_scale=1.0 / 8.0, mode=MODE_Q8_PV8, flags=SMOOTH_K | SMOOTH_Q | SMOOTH_V,
        bq=128, bk=64, seed=2, k_offset_std=2.0, q_offset_std=2.0, q_block_shift_std=1.0,
        q_block_len=64, v_bias_std=2.0,
        note="video-diffusion self-attention, N=17776 (ragged), Q/K/V smoothing"),
    "chunked_gqa": Config(
        name="chunked_gqa", B=1, Hq=32, Hkv=8, N=4096, M=65536, d=128, causal=True,
        sm_scale=1.0 / math.sqrt(128), mode=MODE_Q8_PV8, flags=SMOOTH_K, bq=128, bk=64,
        seed=3, k_offset_std=3.0, k_outliers=4, k_outlier_shift=20.0, v_student_t=3.0,
        v_clip=64.0,
        note="chunked prefill, GQA 32/8, bottom-right causal, Student-t(3) V clipped at 64"),
    "nvfp4": Config(
        name="nvfp4", B=2, Hq=24, Hkv=24, N=8192, M=8192, d=128, causal=False,
        sm_scale=1.0 / math.sqrt(128), mode=MODE_NVFP4, flags=SMOOTH_K, bq=128, bk=64,
        seed=4, k_offset_std=3.0,
        note="NVFP4 microscaling mode with two-level P~"),
}

ORDER = ["tiny", "llm_prefill", "video", "chunked_gqa", "nvfp4"]


def config_by_name(name: str) -> Config:
    return CONFIGS[name]
