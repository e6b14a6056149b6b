"""The five synthetic MoE-layer workloads (shapes, seeds, residency, split policy).

Each workload stands in for a layer shape of the models the FreeToken paper
serves (DeepSeek-V4-Flash routes 6 of 256 experts: FreeToken, Abstract and
section 1).  Nothing here computes any part of the layer; these are plain
records consumed by ``moe_inputs.gen``.

Field meanings
--------------
T, H, E, k, I   tokens per call, hidden size, experts per layer, top-k, SwiGLU
                intermediate size.
n_layers        layers stacked in one timed pass (each with its own seed).
steps           decode-trace length (number of successive calls per layer).
seed            base seed; layer l uses ``seed + l``.
cache_slots     slots in the cache pool (pool A).  ``None`` = identity table,
                every expert resident.
phi_q16         fetch fraction B_P/B_H in Q16 (FreeToken section 3.2, Eq. 4).
fill_policy     0 = lowest expert ids fill first, 1 = seeded random subset.
min_fill        1 = keep at least one fill when phi > 0 (section 3.2 text).
bias            'none' | 'zipf' (Zipf(1.1) expert bias) | 'hotset'
                (per-step temporal locality bias).
"""
from dataclasses import dataclass
from typing import Optional

FILL_LOWEST_ID = 0
FILL_RANDOM = 1
Q16 = 1 << 16


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    seed: int
    n_layers: int = 1
    steps: int = 1
    cache_slots: Optional[int] = None
    phi_q16: int = 0
    fill_policy: int = FILL_LOWEST_ID
    min_fill: int = 1
    bias: str = "none"
    zipf_s: float = 1.1
    hot_size: int = 0
    hot_keep: float = 0.0
    hot_beta: float = 0.0

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def expert_bytes(self) -> int:
        """S: bytes of one complete expert (gate, up, down banks, bf16)."""
        return 3 * self.H * self.I * 2


TINY = LayerConfig("tiny", T=64, H=256, E=8, k=2, I=512, seed=0)

# 37% of 256 experts resident (the paper's RTX 5090 serving capacity for
# Qwen3.6, section 5.3), pure on-demand fill (phi = 1, the B_P >= B_H end of Eq. 4).
DECODE = LayerConfig("decode", T=1, H=4096, E=256, k=6, I=2048, seed=1, steps=32,
                     cache_slots=95, phi_q16=Q16, fill_policy=FILL_LOWEST_ID,
                     min_fill=1, bias="zipf")

# B_P/B_H = 0.25, random F/C split, 37% of 128 experts resident.
BATCHED_DECODE = LayerConfig("batched_decode", T=32, H=2048, E=128, k=8, I=768, seed=2,
                             steps=32, cache_slots=47, phi_q16=Q16 // 4,
                             fill_policy=FILL_RANDOM, min_fill=1, bias="hotset",
                             hot_size=48, hot_keep=0.7, hot_beta=2.0)

PREFILL = LayerConfig("prefill", T=8192, H=4096, E=256, k=6, I=2048, seed=3)

# 11% of the 4x256 (layer, expert) pairs resident; the rest are served from the
# staging pool; no fills during prefill (phi = 0).
LONG_PREFILL = LayerConfig("long_prefill", T=16384, H=4096, E=256, k=6, I=2048, seed=500,
                           n_layers=4, cache_slots=113, phi_q16=0, min_fill=1, bias="zipf")

# Profiling case for ncu captures: the decode layer shape (one expert = 50 MB,
# six routed per token) with 32 experts so that the whole device footprint
# stays near 2 GB.  Not a benchmark workload.
DECODE_PROFILE = LayerConfig("decode_profile", T=1, H=4096, E=32, k=6, I=2048, seed=11, steps=32,
                             cache_slots=12, phi_q16=Q16, fill_policy=FILL_LOWEST_ID, min_fill=1,
                             bias="zipf")

# Profiling case for ncu captures of the prefill kernels: the prefill layer
# shape with 64 experts and 2048 tokens, so each expert gets ~192 rows as in
# the 8192-token block over 256 experts (about 3.5 GB on the device).  Not a
# benchmark workload.
PREFILL_PROFILE = LayerConfig("prefill_profile", T=2048, H=4096, E=64, k=6, I=2048, seed=12)

# Profiling case for ncu captures of the tensor-bound GEMM regime of long
# prefill: ~768 rows per expert (three 256-row chunks) over 16 experts, about
# 1.5 GB on the device.  Not a benchmark workload.
GEMM_PROFILE = LayerConfig("gemm_profile", T=2048, H=4096, E=16, k=6, I=2048, seed=13)

CONFIGS = {c.name: c for c in (TINY, DECODE, BATCHED_DECODE, PREFILL, LONG_PREFILL, DECODE_PROFILE,
                               PREFILL_PROFILE, GEMM_PROFILE)}
