"""fp64 statement of the forward with FP8 (e4m3) tensorwise-scaled linear layers.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never imports this
module.

Sources: [ADD] "Nanochat在nanoGPT之上的新增功能", section 1 feature table (FP8 training row:
dynamic tensor-level FP8, e4m3 / e5m2); [ARC] "nanochat — 架构与原理", section 4 (one function
wraps a scaled matrix product, with the quantisation and dequantisation inside it).

READING (the pages give no formula): in the forward, every linear layer of the block and the
lm_head (q, k, v, output projection, MLP up and down projections, lm_head) quantises its input
activation and its weight, each as a whole tensor: scale = 448 / max|tensor| (448 is the largest
finite e4m3 value), round the scaled values to e4m3 (round to nearest even, saturating at
+-448), multiply the two quantised tensors exactly and divide by the product of the scales.  The
activation tensor is the layer input over the whole batch ([B*T, in]).  The small gate vectors
(smear, value-embedding gate) stay in high precision.  e5m2 is the gradient format and does not
enter the forward.

Pinned by ``tests/test_oracle_fp8.py``: e4m3 rounding equals torch's float8_e4m3fn conversion;
a product of tensors already on the e4m3 grid at unit scale is exact; the scaling commutes
with powers of two; the error obeys the e4m3 rounding bound; and the batched forward used here
equals ``oracle.forward`` when the linear map is exact.
"""
from __future__ import annotations

from typing import Callable

import numpy as np

from .forward import (OracleWeights, apply_rope, attention, embed_smear, relu2, rms_norm, rope_tables, sigmoid,
                      softcap)

f64 = np.float64
E4M3_MAX = 448.0


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 value (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
    infinities), ties to even, saturating at +-448.  In the binade [2^e, 2^(e+1)) the spacing is
    2^(e-3); below 2^-6 (the subnormals) it stays 2^-9."""
    x = np.asarray(x, dtype=f64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    step = 2.0 ** (np.maximum(e, -6.0) - 3.0)
    r = np.minimum(np.round(a / step) * step, E4M3_MAX)   # np.round rounds halves to even
    return np.sign(x) * r


def tensor_scale(t: np.ndarray) -> float:
    amax = float(np.max(np.abs(t))) if t.size else 0.0
    return E4M3_MAX / amax if amax > 0 else 1.0


def fp8_linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """x [N, in] . w[out, in]^T with both operands quantised to e4m3 at their tensorwise scales."""
    sx, sw = tensor_scale(x), tensor_scale(w)
    return (round_e4m3(x * sx) @ round_e4m3(w * sw).T) / (sx * sw)


def exact_linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    return x @ w.T


def forward_batched(cfg, W: OracleWeights, tokens: np.ndarray,
                    linear: Callable[[np.ndarray, np.ndarray], np.ndarray] = exact_linear) -> np.ndarray:
    """Soft-capped logits [B, T, V], every linear layer applied to the whole batch's rows through
    `linear` (the step order is that of oracle/forward.py; with exact_linear both agree)."""
    tokens = np.asarray(tokens, dtype=np.int64)
    B, T = tokens.shape
    C, H, Hkv, D, L = cfg.n_embd, cfg.n_head, cfg.n_kv_head, cfg.head_dim, cfg.n_layer
    eps = cfg.rms_eps
    lin = lambda x, name: linear(x.reshape(-1, x.shape[-1]), W.m(name)).reshape(x.shape[:-1] + (-1,))
    x0 = np.stack([embed_smear(cfg, W, tokens[b]) for b in range(B)])
    cos, sin = rope_tables(T, D, cfg.rope_base)
    x = x0
    mid = L // 2 - 1
    x_mid = x0 if mid < 0 else None
    for i in range(L):
        x = W.resid_lambdas[i] * x + W.x0_lambdas[i] * x0
        a = rms_norm(x, eps)
        q = lin(a, f"wq.{i}").reshape(B, T, H, D)
        k = lin(a, f"wk.{i}").reshape(B, T, Hkv, D)
        v = lin(a, f"wv.{i}").reshape(B, T, Hkv, D)
        y = np.empty((B, T, H, D), dtype=f64)
        for b in range(B):
            qb = rms_norm(apply_rope(q[b], cos, sin), eps)
            kb = rms_norm(apply_rope(k[b], cos, sin), eps)
            vb = v[b]
            if cfg.has_ve[i]:
                cg = cfg.ve_gate_channels or C
                gate = cfg.ve_gate_scale * sigmoid(a[b, :, :cg] @ W.m(f"veg.{i}").T)
                vb = vb + gate[:, :, None] * W.m(f"ve.{i}")[tokens[b]].reshape(T, Hkv, D)
            y[b] = attention(qb, kb, vb, cfg.window_left[i])
        x = x + lin(y.reshape(B, T, H * D), f"wo.{i}")
        m = rms_norm(x, eps)
        x = x + lin(relu2(lin(m, f"wfc.{i}")), f"wproj.{i}")
        if i == mid:
            x_mid = x
    if cfg.use_backout:
        x = x - W.backout_lambda * x_mid
    return softcap(lin(rms_norm(x, eps), "lm_head"), cfg.softcap)


def forward_fp8(cfg, W: OracleWeights, tokens: np.ndarray) -> np.ndarray:
    """The forward with every linear layer in e4m3 at tensorwise scales (READING above)."""
    return forward_batched(cfg, W, tokens, fp8_linear)
