"""Plain fp64 NumPy statement of the nanochat-style GPT forward pass.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Every step is the textbook definition evaluated in float64; bf16 weights are
upcast exactly and nothing is rounded in between.  Batch rows are processed
one at a time (they are independent) and attention is evaluated in blocks of
queries, each query's softmax taken over exactly its visible keys.

Sources (web pages, cited by title and section):

* [ADD] "Nanochat在nanoGPT之上的新增功能" (what nanochat adds over nanoGPT),
  section 1 feature table and the explanatory notes under it.
* [RPT] "NanoChat基础训练报告" (NanoChat base-training report), section
  "模型架构" (model architecture).
* [ARC] "nanochat — 架构与原理" (nanochat architecture and principles),
  section 2 component table and section 4 (packing keeps plain causal
  attention over a packed row).

Readings of points the pages leave open are marked READING and listed with
their justification in the design notes.  All functions here are pinned by
the CPU tests in ``tests/test_oracle_pins.py`` (closed forms, hand-computed
cases, brute force, library routines on special cases, and the parameter
count the report prints).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np

f64 = np.float64


# ----------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------

def param_shapes(cfg) -> Dict[str, tuple]:
    """Shapes of every weight tensor the forward reads ([out, in] for matrices).

    [ADD] §1 table: q, k, v and the output projection are separate matrices
    without biases; the embedding and lm_head are not shared; value embeddings
    are a per-token table on the value-embedding layers.  [RPT] model
    architecture: the value embeddings carry a learned gate.
    """
    C, F, V, D = cfg.n_embd, cfg.mlp_hidden, cfg.vocab_size, cfg.head_dim
    H, Hkv = cfg.n_head, cfg.n_kv_head
    s = {"wte": (V, C)}
    for i in range(cfg.n_layer):
        s[f"wq.{i}"] = (H * D, C)
        s[f"wk.{i}"] = (Hkv * D, C)
        s[f"wv.{i}"] = (Hkv * D, C)
        s[f"wo.{i}"] = (C, H * D)
        s[f"wfc.{i}"] = (F, C)
        s[f"wproj.{i}"] = (C, F)
        if cfg.has_ve[i]:
            s[f"ve.{i}"] = (V, Hkv * D)
            s[f"veg.{i}"] = (Hkv, cfg.ve_gate_channels or C)
    if cfg.use_smear:
        s["smear"] = (cfg.smear_gate_channels or C,)
    s["lm_head"] = (V, C)
    return s


def param_count(cfg, include_gates: bool = True, include_wte: bool = True) -> int:
    n = 0
    for k, shp in param_shapes(cfg).items():
        base = k.split(".")[0]
        if not include_gates and base in ("veg", "smear"):
            continue
        if not include_wte and base == "wte":
            continue
        n += int(np.prod(shp))
    return n


@dataclass
class OracleWeights:
    """Weights as float32 NumPy arrays (exact copies of the bf16 values)."""
    mats: Dict[str, np.ndarray]
    resid_lambdas: List[float]
    x0_lambdas: List[float]
    backout_lambda: float

    @classmethod
    def from_synth(cls, cfg, w: dict) -> "OracleWeights":
        mats = {}
        shapes = param_shapes(cfg)
        for k, shp in shapes.items():
            t = w[k]
            a = t.float().numpy() if hasattr(t, "float") else np.asarray(t, dtype=np.float32)
            if tuple(a.shape) != tuple(shp):
                raise ValueError(f"{k}: shape {a.shape} != {shp}")
            mats[k] = a
        return cls(mats, list(map(float, w["resid_lambdas"])), list(map(float, w["x0_lambdas"])),
                   float(w["backout_lambda"]))

    def m(self, k: str) -> np.ndarray:
        return self.mats[k].astype(f64)


# ----------------------------------------------------------------------------
# elementwise / row operations
# ----------------------------------------------------------------------------

def rms_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """Parameter-free RMSNorm over the last axis ([ADD] §1 table, normalisation row).

    READING: x / sqrt(mean(x^2) + eps); the pages give no epsilon.
    """
    x = np.asarray(x, dtype=f64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def sigmoid(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=f64)
    return 1.0 / (1.0 + np.exp(-z))


def relu2(z: np.ndarray) -> np.ndarray:
    """Squared ReLU ([ADD] §1 table, activation row, and the ReLU² note)."""
    z = np.asarray(z, dtype=f64)
    r = np.maximum(z, 0.0)
    return r * r


def softcap(z: np.ndarray, cap: float) -> np.ndarray:
    """tanh soft cap that keeps logits inside (-cap, cap) ([ADD] §1 table, logit soft-cap row)."""
    z = np.asarray(z, dtype=f64)
    return cap * np.tanh(z / cap)


# ----------------------------------------------------------------------------
# rotary embedding
# ----------------------------------------------------------------------------

def rope_tables(T: int, D: int, base: float):
    """cos/sin of the rotation angles, shape [T, D/2].

    [ADD] RoPE note: relative positions are encoded by rotations in the complex
    plane, with no learned position table.  READING: pair channel d with
    d + D/2; pair d turns by pos * base^(-2d/D); positions restart at 0 in every
    batch row.
    """
    d = np.arange(D // 2, dtype=f64)
    inv_freq = base ** (-2.0 * d / D)
    ang = np.arange(T, dtype=f64)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def apply_rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate [T, n_heads, D] by position.  READING: y1 = x1 cos + x2 sin, y2 = -x1 sin + x2 cos."""
    D = x.shape[-1]
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([x1 * c + x2 * s, -x1 * s + x2 * c], axis=-1)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, window: int, block: int = 256) -> np.ndarray:
    """Causal grouped-query softmax attention with an optional left window.

    q: [T, H, D]; k, v: [T, Hkv, D] -> y: [T, H, D].
    [ADD] §1 table: grouped-query attention (n_kv_head may be below n_head) and
    per-layer sliding windows.  READING: query head h reads kv head
    h // (H / Hkv); scores are scaled by 1/sqrt(D).  Queries are processed in
    blocks; each query's softmax runs over exactly its visible keys.
    """
    T, H, D = q.shape
    Hkv = k.shape[1]
    group = H // Hkv
    scale = 1.0 / math.sqrt(D)
    y = np.empty((T, H, D), dtype=f64)
    for h in range(H):
        g = h // group
        for t0 in range(0, T, block):
            t1 = min(T, t0 + block)
            lo = 0 if window < 0 else max(0, t0 - window)
            s = (q[t0:t1, h, :] @ k[lo:t1, g, :].T) * scale
            ii = np.arange(t0, t1)[:, None]
            jj = np.arange(lo, t1)[None, :]
            vis = jj <= ii
            if window >= 0:
                vis &= jj >= ii - window
            s = np.where(vis, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            y[t0:t1, h, :] = p @ v[lo:t1, g, :]
    return y


# ----------------------------------------------------------------------------
# model
# ----------------------------------------------------------------------------

def embed_smear(cfg, W: OracleWeights, tok: np.ndarray) -> np.ndarray:
    """Token embedding followed by smear; returns x0 = [T, C].

    [ADD] smear note: the previous token's embedding is mixed into the current
    one through a learned sigmoid gate, x + sigmoid(gate(x)) * x_prev.
    READING: the gate is one scalar per token, a linear map of the first c_s
    channels of the current token's embedding; x_prev is the previous token's
    embedding before smearing; the first token of a row is unchanged; the
    result is also the x0 that the per-layer x0 scaling mixes back in.
    """
    e = W.m("wte")[tok]
    if cfg.embed_norm:
        e = rms_norm(e, cfg.rms_eps)
    x = e.copy()
    if cfg.use_smear and len(tok) > 1:
        cs = cfg.smear_gate_channels or cfg.n_embd
        gate = sigmoid(e[1:, :cs] @ W.m("smear"))
        x[1:] = e[1:] + gate[:, None] * e[:-1]
    return x


def block(cfg, W: OracleWeights, i: int, x: np.ndarray, x0: np.ndarray, tok: np.ndarray,
          cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """One transformer block, including the per-layer residual / x0 scaling.

    Order: x <- resid_lambda*x + x0_lambda*x0 ([ADD] residual-scaling row;
    READING: applied at the start of every block); pre-norm attention with
    separate bias-free q/k/v projections, RoPE, then RMSNorm of q and k per
    head ([ADD] QK-norm row: normalised after RoPE); on value-embedding layers
    v <- v + gate * ve[token] ([ADD] value-residual note; [RPT] learned gate;
    READING: gate = ve_gate_scale * sigmoid(a[:, :c_g] . W_g[kv head]) with a the
    block's normed input); windowed causal GQA; output projection added to
    the residual; then the pre-norm ReLU² MLP added to the residual.
    """
    T = x.shape[0]
    H, Hkv, D = cfg.n_head, cfg.n_kv_head, cfg.head_dim
    eps = cfg.rms_eps
    x = W.resid_lambdas[i] * x + W.x0_lambdas[i] * x0
    a = rms_norm(x, eps)
    q = (a @ W.m(f"wq.{i}").T).reshape(T, H, D)
    k = (a @ W.m(f"wk.{i}").T).reshape(T, Hkv, D)
    v = (a @ W.m(f"wv.{i}").T).reshape(T, Hkv, D)
    q = rms_norm(apply_rope(q, cos, sin), eps)
    k = rms_norm(apply_rope(k, cos, sin), eps)
    if cfg.has_ve[i]:
        cg = cfg.ve_gate_channels or cfg.n_embd
        gate = cfg.ve_gate_scale * sigmoid(a[:, :cg] @ W.m(f"veg.{i}").T)        # [T, Hkv]
        ve = W.m(f"ve.{i}")[tok].reshape(T, Hkv, D)
        v = v + gate[:, :, None] * ve
    y = attention(q, k, v, cfg.window_left[i])
    x = x + y.reshape(T, H * D) @ W.m(f"wo.{i}").T
    m = rms_norm(x, eps)
    x = x + relu2(m @ W.m(f"wfc.{i}").T) @ W.m(f"wproj.{i}").T
    return x


def final_hidden(cfg, W: OracleWeights, tok: np.ndarray) -> np.ndarray:
    """Residual stream after backout and the final RMSNorm, [T, C].

    [ADD] backout note: the residual stream is cached at the middle of the
    stack and lambda * x_backout is subtracted before the final norm.
    READING: the cache is taken after block L//2 - 1 (x0 when L == 1).
    """
    tok = np.asarray(tok, dtype=np.int64)
    T = len(tok)
    x0 = embed_smear(cfg, W, tok)
    cos, sin = rope_tables(T, cfg.head_dim, cfg.rope_base)
    x = x0
    L = cfg.n_layer
    mid = L // 2 - 1
    x_mid = x0 if mid < 0 else None
    for i in range(L):
        x = block(cfg, W, i, x, x0, tok, cos, sin)
        if i == mid:
            x_mid = x
    if cfg.use_backout:
        x = x - W.backout_lambda * x_mid
    return rms_norm(x, cfg.rms_eps)


def forward_row(cfg, W: OracleWeights, tok: np.ndarray,
                positions: Optional[Sequence[int]] = None) -> np.ndarray:
    """Soft-capped logits [T, V] for one batch row (or [len(positions), V])."""
    xf = final_hidden(cfg, W, tok)
    if positions is not None:
        xf = xf[np.asarray(positions)]
    z = xf @ W.m("lm_head").T
    return softcap(z, cfg.softcap)


def forward(cfg, W: OracleWeights, tokens: np.ndarray) -> np.ndarray:
    """Soft-capped logits [B, T, V]; rows are independent."""
    tokens = np.asarray(tokens)
    return np.stack([forward_row(cfg, W, tokens[b]) for b in range(tokens.shape[0])])
