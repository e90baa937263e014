"""fp64 gradient of the mean next-token cross-entropy with respect to every weight of the
forward: the backward pass of a training step.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never imports this
module.

The forward is restated with torch fp64 CPU operations, step for step in the order and
notation of ``oracle/forward.py`` (which cites the pages for each step), so that reverse-mode
differentiation gives the exact gradient of the defined loss.  The differentiation itself is a
library step.  The loss is that of ``oracle/loss.py``: cross-entropy of the soft-capped logits
against the given targets, in nats, averaged over the positions whose target is >= 0.

Sources: [RPT] "NanoChat基础训练报告", loss progression table (the training loss); [ADD]
"Nanochat在nanoGPT之上的新增功能", section 1 table and notes (every step of the forward); the
per-layer residual and x0 scales and the backout scale are learned scalars ([ADD] residual-
scaling and backout rows), so they get gradients too.

Pinned by ``tests/test_oracle_backward.py``: the restated forward reproduces
``oracle.forward`` and the loss of ``oracle.loss``; the gradients equal central finite
differences of the fp64 loss on a small model, for sampled entries of every kind of weight.
"""
from __future__ import annotations

import math
from typing import Dict, Tuple

import numpy as np
import torch

from .forward import OracleWeights

f64 = torch.float64


def _rms(x: torch.Tensor, eps: float) -> torch.Tensor:
    return x / torch.sqrt((x * x).mean(-1, keepdim=True) + eps)


def _rope_tables(T: int, D: int, base: float):
    d = torch.arange(D // 2, dtype=f64)
    inv_freq = base ** (-2.0 * d / D)
    ang = torch.arange(T, dtype=f64)[:, None] * inv_freq[None, :]
    return torch.cos(ang), torch.sin(ang)


def _rope(x: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor) -> torch.Tensor:
    D = x.shape[-1]
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    c, s = cos[:, None, :], sin[:, None, :]
    return torch.cat([x1 * c + x2 * s, -x1 * s + x2 * c], -1)


def _attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window: int) -> torch.Tensor:
    """q [T, H, D], k, v [T, Hkv, D]; query head h reads kv head h // (H / Hkv); key j is visible
    to query i when j <= i and, with a window, j >= i - window."""
    T, H, D = q.shape
    group = H // k.shape[1]
    kk = k.repeat_interleave(group, dim=1)
    vv = v.repeat_interleave(group, dim=1)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    vis = j <= i
    if window >= 0:
        vis = vis & (j >= i - window)
    s = torch.einsum("thd,shd->hts", q, kk) / math.sqrt(D)
    p = torch.softmax(s.masked_fill(~vis, float("-inf")), dim=-1)
    return torch.einsum("hts,shd->thd", p, vv)


def forward_row(cfg, P: Dict[str, torch.Tensor], tok: torch.Tensor) -> torch.Tensor:
    """Soft-capped logits [T, V] of one batch row; P holds every weight and the scalars
    ``resid_lambdas`` [L], ``x0_lambdas`` [L], ``backout_lambda`` [] as fp64 tensors."""
    T = tok.shape[0]
    C, H, Hkv, D, L = cfg.n_embd, cfg.n_head, cfg.n_kv_head, cfg.head_dim, cfg.n_layer
    eps = cfg.rms_eps
    e = P["wte"][tok]
    if cfg.embed_norm:
        e = _rms(e, eps)
    x = e
    if cfg.use_smear and T > 1:
        cs = cfg.smear_gate_channels or C
        gate = torch.sigmoid(e[1:, :cs] @ P["smear"])
        x = torch.cat([e[:1], e[1:] + gate[:, None] * e[:-1]], 0)
    x0 = x
    cos, sin = _rope_tables(T, D, cfg.rope_base)
    mid = L // 2 - 1
    x_mid = x0 if mid < 0 else None
    for i in range(L):
        x = P["resid_lambdas"][i] * x + P["x0_lambdas"][i] * x0
        a = _rms(x, eps)
        q = (a @ P[f"wq.{i}"].T).reshape(T, H, D)
        k = (a @ P[f"wk.{i}"].T).reshape(T, Hkv, D)
        v = (a @ P[f"wv.{i}"].T).reshape(T, Hkv, D)
        q = _rms(_rope(q, cos, sin), eps)
        k = _rms(_rope(k, cos, sin), eps)
        if cfg.has_ve[i]:
            cg = cfg.ve_gate_channels or C
            gate = cfg.ve_gate_scale * torch.sigmoid(a[:, :cg] @ P[f"veg.{i}"].T)
            v = v + gate[:, :, None] * P[f"ve.{i}"][tok].reshape(T, Hkv, D)
        y = _attention(q, k, v, cfg.window_left[i])
        x = x + y.reshape(T, H * D) @ P[f"wo.{i}"].T
        m = _rms(x, eps)
        h = torch.relu(m @ P[f"wfc.{i}"].T)
        x = x + (h * h) @ P[f"wproj.{i}"].T
        if i == mid:
            x_mid = x
    if cfg.use_backout:
        x = x - P["backout_lambda"] * x_mid
    z = _rms(x, eps) @ P["lm_head"].T
    return cfg.softcap * torch.tanh(z / cfg.softcap)


def parameters(W: OracleWeights) -> Dict[str, torch.Tensor]:
    """Every trainable quantity of the forward as an fp64 leaf tensor (weights exactly as given)."""
    P = {k: torch.tensor(v, dtype=f64) for k, v in W.mats.items()}
    P["resid_lambdas"] = torch.tensor(W.resid_lambdas, dtype=f64)
    P["x0_lambdas"] = torch.tensor(W.x0_lambdas, dtype=f64)
    P["backout_lambda"] = torch.tensor(W.backout_lambda, dtype=f64)
    return P


def mean_loss(cfg, P: Dict[str, torch.Tensor], tokens: np.ndarray, targets: np.ndarray) -> torch.Tensor:
    """Mean over the positions with a target >= 0 of log(sum_v exp z) - z[target]."""
    total, count = torch.zeros((), dtype=f64), 0
    for b in range(tokens.shape[0]):
        z = forward_row(cfg, P, torch.as_tensor(tokens[b], dtype=torch.long))
        t = torch.as_tensor(targets[b], dtype=torch.long)
        keep = t >= 0
        if keep.any():
            zk = z[keep]
            total = total + (torch.logsumexp(zk, -1) - zk.gather(1, t[keep][:, None])[:, 0]).sum()
            count += int(keep.sum())
    return total / count


def loss_and_grads(cfg, W: OracleWeights, tokens: np.ndarray,
                   targets: np.ndarray) -> Tuple[float, Dict[str, np.ndarray]]:
    """(mean loss, gradient of it with respect to every entry of ``parameters(W)``), fp64."""
    P = parameters(W)
    for p in P.values():
        p.requires_grad_(True)
    loss = mean_loss(cfg, P, tokens, targets)
    loss.backward()
    return float(loss.item()), {k: p.grad.detach().numpy().copy() for k, p in P.items()}


# ---------------------------------------------------------------- step backwards (closed forms)
# The backward of single steps of the forward, written out from calculus, in fp64 NumPy: the
# references of the GPU's backward kernels, each pinned by ``tests/test_oracle_backward.py``
# against central finite differences of its own forward step and against a property of it.

def rms_norm_backward(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """dL/dx of the weightless RMSNorm xn = x / sqrt(mean(x^2) + eps) over the last axis, given
    g = dL/dxn ([ADD] RMSNorm row: no learned weight).  With r = (mean(x^2) + eps)^(-1/2) and
    dr/dx_j = -r^3 x_j / C:  dL/dx_j = r g_j - r^3 x_j mean_i(g_i x_i)."""
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    r = 1.0 / np.sqrt((x * x).mean(-1, keepdims=True) + eps)
    return r * g - r ** 3 * x * (g * x).mean(-1, keepdims=True)


def softcap_ce_grad(u: np.ndarray, targets: np.ndarray, cap: float) -> np.ndarray:
    """d/du of the mean over counted rows (target in [0, V)) of log sum_v exp z_v - z_target, with
    z = cap * tanh(u / cap) ([ADD] logit soft-cap row; the loss as in ``oracle/loss.py``):
    (softmax(z) - onehot(target)) * (1 - (z / cap)^2) / (rows counted); ignored rows are zero."""
    u = np.asarray(u, dtype=np.float64)
    t = np.asarray(targets).reshape(-1)
    M, V = u.shape
    z = cap * np.tanh(u / cap)
    keep = (t >= 0) & (t < V)
    n = int(keep.sum())
    out = np.zeros_like(z)
    if n == 0:
        return out
    zk = z[keep]
    p = np.exp(zk - zk.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    p[np.arange(n), t[keep]] -= 1.0
    out[keep] = p * (1.0 - (zk / cap) ** 2) / n
    return out


def relu2_backward(u: np.ndarray, g: np.ndarray) -> np.ndarray:
    """d/du of relu(u)^2 times the upstream gradient g ([ADD] ReLU^2 row): 2 relu(u) g."""
    u = np.asarray(u, dtype=np.float64)
    return 2.0 * np.maximum(u, 0.0) * np.asarray(g, dtype=np.float64)
