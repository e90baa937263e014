"""Seeded synthetic weights and token ids.

Every tensor is drawn by its own CPU ``torch.Generator`` seeded with
``1000 * seed + index``, where ``index`` is the tensor's place in a fixed
enumeration (embedding; per layer q, k, v, o, fc, proj, value-embedding table,
value-embedding gate; smear gate; lm_head; scalars).  Draws are fp32
N(0, 0.02) rounded to bf16 (round to nearest even), so the fp64 oracle sees
exactly the values the GPU sees.

``init="literal"``: attention and MLP output projections are zero and the
residual scalars are (1, 0).  ``init="dense"``: every matrix is nonzero and the
scalars are drawn from U(0.8, 1.2) (residual) and U(0, 0.3) (x0).

Matrices use the nn.Linear convention [out_features, in_features].
"""
from __future__ import annotations

from typing import Dict, List

import torch

from .configs import ModelConfig, Workload

STD = 0.02
_PER_LAYER = ("wq", "wk", "wv", "wo", "wfc", "wproj", "ve", "veg")


def weight_names(cfg: ModelConfig) -> List[str]:
    names = ["wte"]
    for i in range(cfg.n_layer):
        for n in _PER_LAYER:
            if n in ("ve", "veg") and not cfg.has_ve[i]:
                continue
            names.append(f"{n}.{i}")
    if cfg.use_smear:
        names.append("smear")
    names.append("lm_head")
    return names


def _shape(cfg: ModelConfig, name: str):
    C, F, V = cfg.n_embd, cfg.mlp_hidden, cfg.vocab_size
    base = name.split(".")[0]
    return {
        "wte": (V, C), "wq": (cfg.q_dim, C), "wk": (cfg.kv_dim, C), "wv": (cfg.kv_dim, C),
        "wo": (C, cfg.q_dim), "wfc": (F, C), "wproj": (C, F), "ve": (V, cfg.kv_dim),
        "veg": (cfg.n_kv_head, cfg.c_g), "smear": (cfg.c_s,), "lm_head": (V, C),
    }[base]


def _index(cfg: ModelConfig, name: str) -> int:
    if name == "wte":
        return 0
    if name == "smear":
        return 1 + 8 * cfg.n_layer
    if name == "lm_head":
        return 2 + 8 * cfg.n_layer
    base, layer = name.split(".")
    return 1 + 8 * int(layer) + _PER_LAYER.index(base)


def _draw(shape, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * STD).to(torch.bfloat16)


def make_weights(cfg: ModelConfig, seed: int = 0, init: str = "dense") -> Dict[str, object]:
    """Return a dict of bf16 CPU tensors plus the fp32 scalar lists.

    Keys: the names of ``weight_names(cfg)`` and ``resid_lambdas``,
    ``x0_lambdas`` (lists of n_layer floats) and ``backout_lambda`` (float).
    """
    if init not in ("dense", "literal"):
        raise ValueError(init)
    out: Dict[str, object] = {}
    for name in weight_names(cfg):
        shape = _shape(cfg, name)
        base = name.split(".")[0]
        if init == "literal" and base in ("wo", "wproj"):
            out[name] = torch.zeros(shape, dtype=torch.bfloat16)
        else:
            out[name] = _draw(shape, 1000 * seed + _index(cfg, name))
    L = cfg.n_layer
    if init == "dense":
        g = torch.Generator().manual_seed(1000 * seed + 3 + 8 * L)
        lr = 0.8 + 0.4 * torch.rand(L, generator=g, dtype=torch.float32)
        l0 = 0.3 * torch.rand(L, generator=g, dtype=torch.float32)
        out["resid_lambdas"] = [float(v) for v in lr]
        out["x0_lambdas"] = [float(v) for v in l0]
    else:
        out["resid_lambdas"] = [1.0] * L
        out["x0_lambdas"] = [0.0] * L
    out["backout_lambda"] = 0.5
    return out


def make_tokens(wl: Workload) -> torch.Tensor:
    """int32 [B, T] token ids, uniform in [0, vocab)."""
    g = torch.Generator().manual_seed(wl.token_seed)
    return torch.randint(0, wl.model.vocab_size, (wl.B, wl.T), generator=g, dtype=torch.int32)
