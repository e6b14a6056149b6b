"""Seeded synthetic inputs shared by the oracle's tests and the GPU harness.

Holds workload records (``configs``), host-side numpy draws (``gen``) and the
upload of those draws into device tensors (``device``).  None of it computes
any step of the MoE layer.
"""
from .configs import CONFIGS, LayerConfig, Q16, FILL_LOWEST_ID, FILL_RANDOM  # noqa: F401
