"""Seeded synthetic inputs shared by the fp64 oracle and the CUDA path.

This package describes workloads (shapes, per-layer window sizes, which layers
carry value embeddings) and draws seeded random weights and token ids.  It
holds none of the forward pass's arithmetic: both sides receive exactly the
same tensors from here and compute independently.
"""
from .configs import ModelConfig, Workload, WORKLOADS, get_workload, sssl_windows, alternating_ve_layers
from .weights import make_weights, make_tokens, weight_names

__all__ = [
    "ModelConfig", "Workload", "WORKLOADS", "get_workload", "sssl_windows",
    "alternating_ve_layers", "make_weights", "make_tokens", "weight_names",
]
