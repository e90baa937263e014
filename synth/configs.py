"""Workload descriptions for the nanochat-style decoder-only GPT forward pass.

Architecture facts follow the web pages this project is built from:

* "NanoChat基础训练报告" (NanoChat base-training report), section "模型架构"
  (model architecture): the d12 model has 12 layers, 6 query heads with
  n_kv_head = 6, width 768, head dim 128, a 32,768-entry vocabulary, context
  2,048, and value embeddings with a learned gate on the odd layers 1..11.
* "Nanochat在nanoGPT之上的新增功能" (what nanochat adds over nanoGPT), section 1
  feature table and the notes under it: the sliding-window pattern repeats
  three short-window layers (a quarter of the context) and one full-context
  layer, and the final layer is always full; value embeddings sit on
  alternating layers and the last layer always has one.

The short window is expressed as ``window_left = W``: a query at position i
sees keys j with max(0, i - W) <= j <= i.  ``-1`` means plain causal.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Tuple


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layer: int
    n_embd: int
    n_head: int
    n_kv_head: int
    head_dim: int
    mlp_hidden: int
    vocab_size: int
    seq_len_ctx: int
    window_left: Tuple[int, ...]
    has_ve: Tuple[int, ...]
    use_smear: bool
    use_backout: bool
    embed_norm: bool = False
    smear_gate_channels: int = 0   # 0 means n_embd
    ve_gate_channels: int = 0      # 0 means n_embd
    ve_gate_scale: float = 1.0
    rms_eps: float = 1e-6
    rope_base: float = 10000.0
    softcap: float = 15.0

    @property
    def c_s(self) -> int:
        return self.smear_gate_channels or self.n_embd

    @property
    def c_g(self) -> int:
        return self.ve_gate_channels or self.n_embd

    @property
    def q_dim(self) -> int:
        return self.n_head * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_head * self.head_dim


@dataclass(frozen=True)
class Workload:
    name: str
    model: ModelConfig
    B: int
    T: int
    init: str = "dense"     # "dense": every matrix nonzero; "literal": zero output projections
    seed: int = 0           # weight seed
    token_seed: int = 1

    @property
    def M(self) -> int:
        return self.B * self.T


def sssl_windows(n_layer: int, short: int) -> Tuple[int, ...]:
    """Per-layer window sizes for the repeating short/short/short/long pattern.

    Layer i takes the character "SSSL"[i % 4]; the last layer is always long.
    """
    w = []
    for i in range(n_layer):
        long_layer = ("SSSL"[i % 4] == "L") or (i == n_layer - 1)
        w.append(-1 if long_layer else short)
    return tuple(w)


def alternating_ve_layers(n_layer: int) -> Tuple[int, ...]:
    """Value-embedding layers: every other layer, counted back from the last one."""
    return tuple(1 if (i % 2) == ((n_layer - 1) % 2) else 0 for i in range(n_layer))


def _d_model(name, depth, n_head, n_kv_head, T_ctx, short):
    C = n_head * 128
    return ModelConfig(
        name=name, n_layer=depth, n_embd=C, n_head=n_head, n_kv_head=n_kv_head,
        head_dim=128, mlp_hidden=4 * C, vocab_size=32768, seq_len_ctx=T_ctx,
        window_left=sssl_windows(depth, short), has_ve=alternating_ve_layers(depth),
        use_smear=True, use_backout=True)


_TINY = ModelConfig(
    name="tiny", n_layer=1, n_embd=128, n_head=2, n_kv_head=1, head_dim=64,
    mlp_hidden=512, vocab_size=512, seq_len_ctx=64, window_left=(-1,), has_ve=(1,),
    use_smear=False, use_backout=False)

_D12 = _d_model("d12", 12, 6, 6, 2048, 512)
_D20 = _d_model("d20", 20, 10, 5, 2048, 512)
_D12L = replace(_d_model("d12_long", 12, 6, 6, 8192, 2048))
_D24 = _d_model("d24", 24, 12, 12, 2048, 512)

WORKLOADS = {
    # tiny GPT exactly as listed: literal init (zero output projections), features off
    "tiny": Workload("tiny", _TINY, B=1, T=64, init="literal"),
    # same shapes with every matrix nonzero, so the block actually changes x
    "tiny_dense": Workload("tiny_dense", _TINY, B=1, T=64, init="dense"),
    # every optional feature switched on at tiny size, two batch rows
    "tiny_all": Workload("tiny_all", replace(_TINY, name="tiny_all", use_smear=True, use_backout=True),
                         B=2, T=64, init="dense"),
    "d12": Workload("d12", _D12, B=8, T=2048),
    "d20": Workload("d20", _D20, B=4, T=2048),
    "d12_long": Workload("d12_long", _D12L, B=2, T=8192),
    "d24": Workload("d24", _D24, B=16, T=2048),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]
