"""Pins for the fp64 oracle against facts fixed outside the oracle itself.

Each test checks one oracle function against a closed form, a hand-computed
value, a brute-force loop on a tiny input, a library routine on a special
case, or a number printed on the source pages (``tests/golden``).  Each is
chosen so that a plausible slip (a dropped term, a flipped sign, a wrong
index or grouping, a transposed operand, an off-by-one window) fails.
"""
import json
import math
import os
from dataclasses import replace

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
from synth import get_workload, make_tokens, make_weights
from synth.configs import ModelConfig

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _tiny_cfg(**kw):
    base = get_workload("tiny_all").model
    return replace(base, **kw)


def _weights(cfg, init="dense", seed=0):
    return O.OracleWeights.from_synth(cfg, make_weights(cfg, seed=seed, init=init))


# ---------------------------------------------------------------- parameter count

def test_param_count_matches_report():
    """The report prints 286.3M total and 261.1M non-embedding parameters for d12."""
    g = json.load(open(os.path.join(GOLDEN, "d12_report.json")))
    cfg = get_workload("d12").model
    assert (cfg.n_layer, cfg.n_head, cfg.n_kv_head, cfg.n_embd, cfg.head_dim, cfg.vocab_size,
            cfg.seq_len_ctx) == (g["n_layer"], g["n_head"], g["n_kv_head"], g["n_embd"],
                                 g["head_dim"], g["vocab_size"], g["context"])
    assert [i for i, h in enumerate(cfg.has_ve) if h] == g["value_embedding_layers"]
    total = O.param_count(cfg, include_gates=False)
    assert total == 286_261_248          # closed form: 2VC + 6 V Hkv D + 12 (4C^2 + 8C^2)
    assert round(total / 1e6, 1) == g["params_total_millions"]
    assert round(O.param_count(cfg, include_gates=True) / 1e6, 1) == g["params_total_millions"]
    non_emb = O.param_count(cfg, include_gates=False, include_wte=False)
    assert non_emb == 261_095_424
    assert round(non_emb / 1e6, 1) == g["params_non_embedding_millions"]


def test_weight_shapes_nn_linear_convention():
    cfg = get_workload("d20").model
    s = O.param_shapes(cfg)
    assert s["wq.0"] == (1280, 1280) and s["wk.0"] == (640, 1280) and s["wv.0"] == (640, 1280)
    assert s["wo.0"] == (1280, 1280) and s["wfc.0"] == (5120, 1280) and s["wproj.0"] == (1280, 5120)
    assert "ve.0" not in s and s["ve.19"] == (32768, 640)
    assert s["lm_head"] == (32768, 1280)


# ---------------------------------------------------------------- rms norm

def test_rms_norm_unit_rms_and_scale_invariance():
    x = rng.standard_normal((7, 96)) * 3.0
    y = O.rms_norm(x, 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(O.rms_norm(5.0 * x, 0.0), y, rtol=1e-12)
    # hand value: [3, 4] has rms sqrt(12.5)
    np.testing.assert_allclose(O.rms_norm(np.array([3.0, 4.0]), 0.0), [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)])
    # epsilon enters under the square root
    np.testing.assert_allclose(O.rms_norm(np.array([1.0, 1.0]), 1.0), [1 / math.sqrt(2.0)] * 2)


def test_rms_norm_matches_torch():
    x = rng.standard_normal((5, 64))
    ref = F.rms_norm(torch.from_numpy(x), (64,), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(x, 1e-6), ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- rope

def test_rope_d2_hand_rotation():
    # D = 2: one pair, angle = pos * base^0 = pos.  (1, 0) at pos 1 -> (cos 1, -sin 1)
    cos, sin = O.rope_tables(3, 2, 10000.0)
    x = np.zeros((3, 1, 2)); x[:, 0, 0] = 1.0
    y = O.apply_rope(x, cos, sin)
    np.testing.assert_allclose(y[1, 0], [0.5403023058681398, -0.8414709848078965], rtol=1e-14)
    np.testing.assert_allclose(y[0, 0], [1.0, 0.0])
    x2 = np.zeros((3, 1, 2)); x2[:, 0, 1] = 1.0   # (0, 1) at pos 2 -> (sin 2, cos 2)
    np.testing.assert_allclose(O.apply_rope(x2, cos, sin)[2, 0], [0.9092974268256817, -0.4161468365471424], rtol=1e-14)


def test_rope_frequencies_half_split():
    # D = 4, base 10000: pair (0, 2) turns by pos * 1, pair (1, 3) by pos * 0.01
    cos, sin = O.rope_tables(101, 4, 10000.0)
    np.testing.assert_allclose(cos[100], [math.cos(100.0), math.cos(1.0)], rtol=1e-12)
    np.testing.assert_allclose(sin[100], [math.sin(100.0), math.sin(1.0)], rtol=1e-12)
    x = np.zeros((101, 1, 4)); x[:, 0, 1] = 1.0      # channel 1 pairs with channel 3
    y = O.apply_rope(x, cos, sin)[100, 0]
    np.testing.assert_allclose(y, [0.0, math.cos(1.0), 0.0, -math.sin(1.0)], atol=1e-14)


def test_rope_matches_complex_rotation():
    T, H, D = 9, 3, 16
    x = rng.standard_normal((T, H, D))
    cos, sin = O.rope_tables(T, D, 500.0)
    z = x[..., : D // 2] + 1j * x[..., D // 2:]
    theta = np.arange(T)[:, None] * 500.0 ** (-2.0 * np.arange(D // 2) / D)
    zr = z * np.exp(-1j * theta)[:, None, :]
    np.testing.assert_allclose(O.apply_rope(x, cos, sin), np.concatenate([zr.real, zr.imag], -1), atol=1e-13)


def test_rope_norm_preserving_and_relative():
    T, D = 40, 32
    cos, sin = O.rope_tables(T, D, 10000.0)
    q = rng.standard_normal((1, 1, D)); k = rng.standard_normal((1, 1, D))
    Q = O.apply_rope(np.repeat(q, T, 0), cos, sin)[:, 0]
    K = O.apply_rope(np.repeat(k, T, 0), cos, sin)[:, 0]
    np.testing.assert_allclose(np.linalg.norm(Q, axis=-1), np.linalg.norm(q), rtol=1e-12)
    d1 = Q[10] @ K[3]; d2 = Q[30] @ K[23]; d3 = Q[7] @ K[0]
    np.testing.assert_allclose([d2, d3], [d1, d1], rtol=1e-10)


def test_qk_norm_unit_rms_after_rope():
    cfg = get_workload("tiny_all").model
    x = rng.standard_normal((16, 2, 64)) * 0.3
    cos, sin = O.rope_tables(16, 64, 10000.0)
    y = O.rms_norm(O.apply_rope(x, cos, sin), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, -1)), 1.0, rtol=1e-12)


# ---------------------------------------------------------------- attention

def _brute_attention(q, k, v, window):
    T, H, D = q.shape
    Hkv = k.shape[1]
    y = np.zeros_like(q)
    for h in range(H):
        g = h * Hkv // H
        for i in range(T):
            keys = [j for j in range(T) if j <= i and (window < 0 or i - j <= window)]
            s = [sum(q[i, h, d] * k[j, g, d] for d in range(D)) / math.sqrt(D) for j in keys]
            m = max(s)
            w = [math.exp(a - m) for a in s]
            z = sum(w)
            for d in range(D):
                y[i, h, d] = sum(w[n] * v[keys[n], g, d] for n in range(len(keys))) / z
    return y


@pytest.mark.parametrize("window", [-1, 0, 1, 3, 20])
def test_attention_brute_force_tiny(window):
    T, H, Hkv, D = 11, 4, 2, 4
    q = rng.standard_normal((T, H, D)); k = rng.standard_normal((T, Hkv, D)); v = rng.standard_normal((T, Hkv, D))
    np.testing.assert_allclose(O.attention(q, k, v, window, block=4), _brute_attention(q, k, v, window), atol=1e-12)


def test_attention_window_counts_keys():
    # window W: query i sees exactly min(i+1, W+1) keys -> with v one-hot over positions the
    # output support is exactly those keys
    T, W = 12, 3
    q = np.zeros((T, 1, 4)); k = np.zeros((T, 1, 4))
    v = np.eye(T)[:, None, :4].copy()  # placeholder shape fix below
    v = np.zeros((T, 1, T)); v[np.arange(T), 0, np.arange(T)] = 1.0
    q = np.zeros((T, 1, T)); k = np.zeros((T, 1, T))
    y = O.attention(q, k, v, W)[:, 0]
    for i in range(T):
        expect = np.zeros(T); lo = max(0, i - W); expect[lo:i + 1] = 1.0 / (i + 1 - lo)
        np.testing.assert_allclose(y[i], expect, atol=1e-15)


def test_attention_window_ge_T_is_causal_and_matches_sdpa():
    T, H, D = 33, 2, 8
    q = rng.standard_normal((T, H, D)); k = rng.standard_normal((T, H, D)); v = rng.standard_normal((T, H, D))
    full = O.attention(q, k, v, -1, block=8)
    np.testing.assert_allclose(O.attention(q, k, v, T, block=8), full, atol=1e-13)
    np.testing.assert_allclose(O.attention(q, k, v, 10 * T, block=8), full, atol=1e-13)
    tq = torch.from_numpy(q).permute(1, 0, 2)
    ref = F.scaled_dot_product_attention(tq, torch.from_numpy(k).permute(1, 0, 2),
                                         torch.from_numpy(v).permute(1, 0, 2), is_causal=True)
    np.testing.assert_allclose(full, ref.permute(1, 0, 2).numpy(), atol=1e-12)


def test_attention_gqa_matches_sdpa_enable_gqa_and_duplicated_mha():
    T, H, Hkv, D = 21, 6, 2, 8
    q = rng.standard_normal((T, H, D)); k = rng.standard_normal((T, Hkv, D)); v = rng.standard_normal((T, Hkv, D))
    y = O.attention(q, k, v, -1, block=5)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q).permute(1, 0, 2), torch.from_numpy(k).permute(1, 0, 2),
                                         torch.from_numpy(v).permute(1, 0, 2), is_causal=True, enable_gqa=True)
    np.testing.assert_allclose(y, ref.permute(1, 0, 2).numpy(), atol=1e-12)
    kd = np.repeat(k, H // Hkv, axis=1); vd = np.repeat(v, H // Hkv, axis=1)
    np.testing.assert_allclose(O.attention(q, kd, vd, -1), y, atol=1e-13)


def test_attention_window_matches_sdpa_mask_and_row0():
    T, H, D, W = 40, 2, 8, 7
    q = rng.standard_normal((T, H, D)); k = rng.standard_normal((T, H, D)); v = rng.standard_normal((T, H, D))
    y = O.attention(q, k, v, W, block=16)
    i = torch.arange(T)[:, None]; j = torch.arange(T)[None, :]
    mask = (j <= i) & (i - j <= W)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q).permute(1, 0, 2), torch.from_numpy(k).permute(1, 0, 2),
                                         torch.from_numpy(v).permute(1, 0, 2), attn_mask=mask)
    np.testing.assert_allclose(y, ref.permute(1, 0, 2).numpy(), atol=1e-12)
    np.testing.assert_array_equal(y[0], v[0])


# ---------------------------------------------------------------- elementwise

def test_relu2_softcap_sigmoid_closed_forms():
    z = np.array([-2.0, -0.0, 0.0, 0.5, 3.0])
    np.testing.assert_array_equal(O.relu2(z), [0.0, 0.0, 0.0, 0.25, 9.0])
    assert O.softcap(np.array([15.0]), 15.0)[0] == pytest.approx(15 * math.tanh(1.0))
    big = O.softcap(np.array([-1e6, 1e6, 100.0]), 15.0)
    assert np.all(np.abs(big) <= 15.0)
    small = np.array([1e-4, -3e-3])
    np.testing.assert_allclose(O.softcap(small, 15.0), small, rtol=1e-5)
    np.testing.assert_allclose(O.sigmoid(np.array([0.0])), [0.5])
    x = rng.standard_normal(10)
    np.testing.assert_allclose(O.sigmoid(x) + O.sigmoid(-x), 1.0, rtol=1e-14)


# ---------------------------------------------------------------- smear / value embeddings / scalars

def test_smear_zero_gate_is_half_previous():
    cfg = _tiny_cfg()
    W = _weights(cfg)
    W.mats["smear"] = np.zeros_like(W.mats["smear"])
    tok = np.array([3, 7, 7, 100, 5])
    x = O.embed_smear(cfg, W, tok)
    e = W.m("wte")[tok]
    np.testing.assert_array_equal(x[0], e[0])
    np.testing.assert_allclose(x[1:], e[1:] + 0.5 * e[:-1], rtol=0, atol=0)


def test_smear_hand_example():
    cfg = replace(_tiny_cfg(), n_embd=128, smear_gate_channels=2)
    W = _weights(cfg)
    W.mats["smear"] = np.array([1.0, -2.0], dtype=np.float32)
    tok = np.array([0, 1])
    W.mats["wte"][:2] = 0.0
    W.mats["wte"][0, :3] = [1.0, 0.0, 4.0]
    W.mats["wte"][1, :3] = [0.5, 0.25, 8.0]
    x = O.embed_smear(cfg, W, tok)
    g = 1.0 / (1.0 + math.exp(-(0.5 * 1.0 + 0.25 * -2.0)))   # = sigmoid(0) = 0.5
    np.testing.assert_allclose(x[1, :3], [0.5 + g * 1.0, 0.25 + g * 0.0, 8.0 + g * 4.0])


def test_ve_gate_special_cases():
    cfg = get_workload("tiny_dense").model
    tok = make_tokens(get_workload("tiny_dense")).numpy()[0][:20]
    W = _weights(cfg)
    cos, sin = O.rope_tables(20, cfg.head_dim, cfg.rope_base)
    x0 = O.embed_smear(cfg, W, tok)
    # zero VE table -> identical to a layer without value embeddings
    Wz = _weights(cfg); Wz.mats["ve.0"] = np.zeros_like(Wz.mats["ve.0"])
    no_ve = replace(cfg, has_ve=(0,))
    np.testing.assert_allclose(O.block(cfg, Wz, 0, x0, x0, tok, cos, sin),
                               O.block(no_ve, W, 0, x0, x0, tok, cos, sin), atol=1e-14)
    # zero gate weights -> gate 0.5: equal to adding 0.5*ve to the V projection's output, i.e. to a
    # value weight whose rows are unchanged but a value table halved with full gate
    Wg = _weights(cfg); Wg.mats["veg.0"] = np.zeros_like(Wg.mats["veg.0"])
    Wh = _weights(cfg); Wh.mats["veg.0"] = np.zeros_like(Wh.mats["veg.0"])
    Wh.mats["ve.0"] = Wh.mats["ve.0"] * np.float32(0.5)
    c2 = replace(cfg, ve_gate_scale=2.0)   # 2 * sigmoid(0) = 1
    np.testing.assert_allclose(O.block(cfg, Wg, 0, x0, x0, tok, cos, sin),
                               O.block(c2, Wh, 0, x0, x0, tok, cos, sin), atol=1e-13)


def _gate_pin_case(cfg, T, seed):
    """Inputs for the value-embedding gate pins: one VE layer, block input x with an RMS far from
    1 (so a gate taken from un-normed x differs from one taken from a = rms(x)), and the normed
    input a computed by torch's rms_norm (a library routine, not the oracle)."""
    W = _weights(cfg, seed=seed)
    g = np.random.default_rng(seed)
    x = g.standard_normal((T, cfg.n_embd)) * 0.05
    x0 = g.standard_normal((T, cfg.n_embd)) * 0.02
    tok = g.integers(0, cfg.vocab_size, T)
    mixed = W.resid_lambdas[0] * x + W.x0_lambdas[0] * x0
    a = F.rms_norm(torch.from_numpy(mixed), (cfg.n_embd,), eps=cfg.rms_eps).numpy()
    assert np.all(np.abs(np.sqrt(np.mean(mixed ** 2, -1)) - 1.0) > 0.5)
    return W, x, x0, tok, a


def _fold_gated_ve_into_wv(cfg, W, a, tok, Z):
    """Value weights W_v' with a W_v'^T = a W_v^T + gate * ve[tok] on every kv head, where
    gate[t, g] = sigmoid(Z[t, g]) (ve_gate_scale = 1): with T <= C and the rows of a independent,
    the least-squares solution reproduces the gated table rows exactly (up to rounding)."""
    T, Hkv, D = len(tok), cfg.n_kv_head, cfg.head_dim
    ve = W.m("ve.0")[tok].reshape(T, Hkv, D)
    target = (1.0 / (1.0 + np.exp(-Z)))[:, :, None] * ve          # [T, Hkv, D]
    dWv_t, *_ = np.linalg.lstsq(a, target.reshape(T, Hkv * D), rcond=None)
    return W.m("wv.0") + dWv_t.T


@pytest.mark.parametrize("shape", ["gqa_h4_kv2", "d20_width"])
def test_ve_gate_per_head_from_normed_input(shape):
    """The gate of kv head g is sigmoid(a . W_g[g]) with a the block's RMS-normed input, and it
    scales kv head g's slice of the value-embedding row of the token.  Gate weights are solved so
    that a . W_g[g] equals chosen pre-activations Z[:, g] (some saturating at +-40, some not);
    the value-embedding layer must then equal a layer without value embeddings whose value
    projection is shifted to add exactly sigmoid(Z) * ve[tok] per head.  Fails if the gate is
    taken from the un-normed x, if gate rows are paired with the wrong kv head, or if the table
    row is split into heads in another order."""
    if shape == "gqa_h4_kv2":
        cfg = replace(get_workload("tiny_all").model, n_head=4, n_kv_head=2, head_dim=32, has_ve=(1,),
                      use_smear=False, use_backout=False)
        T = 12
    else:   # the d20 attention shape (10 heads of 128, 5 kv heads) on one layer, small vocabulary
        cfg = replace(get_workload("d20").model, n_layer=1, vocab_size=512, seq_len_ctx=16,
                      window_left=(-1,), has_ve=(1,))
        T = 16
    W, x, x0, tok, a = _gate_pin_case(cfg, T, seed=7)
    g = np.random.default_rng(11)
    Z = g.standard_normal((T, cfg.n_kv_head)) * 1.5
    Z[:, 0] = 40.0                      # kv head 0: gate 1 (saturated)
    Z[:, 1] = -40.0                     # kv head 1: gate 0 (saturated)
    Z[: T // 2, -1] = g.uniform(-2, 2, T // 2) if cfg.n_kv_head > 2 else Z[: T // 2, -1]
    Wg, *_ = np.linalg.lstsq(a, Z, rcond=None)                  # a @ Wg = Z
    np.testing.assert_allclose(a @ Wg, Z, atol=1e-9)
    W.mats["veg.0"] = Wg.T.copy()
    cos, sin = O.rope_tables(T, cfg.head_dim, cfg.rope_base)
    got = O.block(cfg, W, 0, x, x0, tok, cos, sin)
    Wf = _weights(cfg, seed=7)
    Wf.mats["wv.0"] = _fold_gated_ve_into_wv(cfg, W, a, tok, Z)
    expect = O.block(replace(cfg, has_ve=(0,)), Wf, 0, x, x0, tok, cos, sin)
    np.testing.assert_allclose(got, expect, atol=1e-9, rtol=1e-9)


def test_ve_gate_hand_element():
    """T = 2, two kv heads: gate pre-activations 0 and ln 3 give gates 1/2 and 3/4, so the value
    of kv head 1 at token t gains exactly 3/4 of columns D..2D of that token's table row."""
    cfg = replace(get_workload("tiny_all").model, n_head=2, n_kv_head=2, head_dim=64, has_ve=(1,),
                  use_smear=False, use_backout=False)
    T = 2
    W, x, x0, tok, a = _gate_pin_case(cfg, T, seed=3)
    Z = np.array([[0.0, math.log(3.0)], [0.0, math.log(3.0)]])
    Wg, *_ = np.linalg.lstsq(a, Z, rcond=None)
    W.mats["veg.0"] = Wg.T.copy()
    gates = 1.0 / (1.0 + np.exp(-Z))
    np.testing.assert_allclose(gates[0], [0.5, 0.75], rtol=1e-15)
    # with a zero value projection the values are the gated table rows; with every query and key
    # zero (zero q/k projections: after QK-norm they stay 0, eps > 0) attention averages the values
    # uniformly over the visible keys: y[1, head 1] = (v[0, 1] + v[1, 1]) / 2
    for k in ("wq.0", "wk.0", "wv.0"):
        W.mats[k] = np.zeros_like(W.mats[k])
    W.mats["wo.0"] = np.eye(cfg.n_embd, dtype=np.float64)       # y lands in the residual unchanged
    W.mats["wproj.0"] = np.zeros_like(W.mats["wproj.0"])        # no MLP contribution
    cos, sin = O.rope_tables(T, cfg.head_dim, cfg.rope_base)
    out = O.block(cfg, W, 0, x, x0, tok, cos, sin)
    mixed = W.resid_lambdas[0] * x + W.x0_lambdas[0] * x0
    D = cfg.head_dim
    ve = W.m("ve.0")
    y1_head1 = 0.75 * (ve[tok[0], D:2 * D] + ve[tok[1], D:2 * D]) / 2.0
    y1_head0 = 0.5 * (ve[tok[0], :D] + ve[tok[1], :D]) / 2.0
    np.testing.assert_allclose(out[1, D:2 * D] - mixed[1, D:2 * D], y1_head1, atol=1e-14)
    np.testing.assert_allclose(out[1, :D] - mixed[1, :D], y1_head0, atol=1e-14)
    np.testing.assert_allclose(out[0, :D] - mixed[0, :D], 0.5 * ve[tok[0], :D], atol=1e-14)


def test_ve_gate_kv_head_permutation_equivariance():
    """Relabelling the kv heads (their q-head groups, key and value rows, gate rows and table
    column blocks together, and the output projection's columns to match) leaves the block's
    output unchanged."""
    cfg = replace(get_workload("tiny_all").model, n_head=6, n_kv_head=3, head_dim=32, n_embd=192,
                  mlp_hidden=256, has_ve=(1,), use_smear=False, use_backout=False)
    T = 10
    W, x, x0, tok, a = _gate_pin_case(cfg, T, seed=5)
    W.mats["veg.0"] = np.random.default_rng(2).standard_normal(W.mats["veg.0"].shape) * 3.0
    H, Hkv, D = cfg.n_head, cfg.n_kv_head, cfg.head_dim
    grp = H // Hkv
    perm = [2, 0, 1]                                    # new kv head g is old kv head perm[g]
    qperm = [perm[h // grp] * grp + h % grp for h in range(H)]

    def rows(m, order):
        return np.concatenate([m[o * D:(o + 1) * D] for o in order], 0)

    P = _weights(cfg, seed=5)
    P.mats = dict(W.mats)
    P.mats["wq.0"] = rows(W.m("wq.0"), qperm)
    P.mats["wk.0"] = rows(W.m("wk.0"), perm)
    P.mats["wv.0"] = rows(W.m("wv.0"), perm)
    P.mats["wo.0"] = rows(W.m("wo.0").T, qperm).T
    P.mats["veg.0"] = W.m("veg.0")[perm]
    P.mats["ve.0"] = rows(W.m("ve.0").T, perm).T
    cos, sin = O.rope_tables(T, D, cfg.rope_base)
    np.testing.assert_allclose(O.block(cfg, P, 0, x, x0, tok, cos, sin), O.block(cfg, W, 0, x, x0, tok, cos, sin),
                               atol=1e-13)


def _plain_gpt_torch(cfg, W, tok):
    """Pre-norm GPT from library routines: rms_norm, linear, complex-rotation RoPE, causal SDPA."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    T = len(tok)
    H, Hkv, D, eps = cfg.n_head, cfg.n_kv_head, cfg.head_dim, cfg.rms_eps
    x = t(W.m("wte"))[torch.from_numpy(tok)]
    theta = torch.arange(T, dtype=torch.float64)[:, None] * cfg.rope_base ** (
        -2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
    rot = torch.polar(torch.ones_like(theta), -theta)[:, None, :]

    def rope(u):
        z = torch.complex(u[..., : D // 2], u[..., D // 2:]) * rot
        return torch.cat([z.real, z.imag], -1)

    for i in range(cfg.n_layer):
        a = F.rms_norm(x, (cfg.n_embd,), eps=eps)
        q = F.linear(a, t(W.m(f"wq.{i}"))).view(T, H, D)
        k = F.linear(a, t(W.m(f"wk.{i}"))).view(T, Hkv, D)
        v = F.linear(a, t(W.m(f"wv.{i}"))).view(T, Hkv, D)
        q = F.rms_norm(rope(q), (D,), eps=eps); k = F.rms_norm(rope(k), (D,), eps=eps)
        y = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                           is_causal=True, enable_gqa=True).transpose(0, 1)
        x = x + F.linear(y.reshape(T, H * D), t(W.m(f"wo.{i}")))
        m = F.rms_norm(x, (cfg.n_embd,), eps=eps)
        x = x + F.linear(torch.relu(F.linear(m, t(W.m(f"wfc.{i}")))) ** 2, t(W.m(f"wproj.{i}")))
    z = F.linear(F.rms_norm(x, (cfg.n_embd,), eps=eps), t(W.m("lm_head")))
    return (cfg.softcap * torch.tanh(z / cfg.softcap)).numpy()


def test_features_off_reduces_to_plain_pre_norm_gpt():
    cfg = replace(get_workload("tiny_all").model, n_layer=2, window_left=(-1, -1), has_ve=(0, 0),
                  use_smear=False, use_backout=False)
    wts = make_weights(cfg, init="dense")
    wts["resid_lambdas"] = [1.0, 1.0]; wts["x0_lambdas"] = [0.0, 0.0]
    W = O.OracleWeights.from_synth(cfg, wts)
    tok = np.array([5, 9, 400, 2, 2, 77, 310, 1, 0, 511, 64, 3])
    np.testing.assert_allclose(O.forward_row(cfg, W, tok), _plain_gpt_torch(cfg, W, tok), atol=1e-12)


def test_resid_lambdas_x0_mix():
    # with zero projections every block is the identity on its mixed input:
    # x_L = prod(lr) x0 + (sum of l0 terms) x0; the final norm removes the scale entirely
    cfg = replace(get_workload("tiny_all").model, n_layer=3, window_left=(-1,) * 3, has_ve=(0, 0, 0),
                  use_smear=False, use_backout=True)
    wts = make_weights(cfg, init="literal")
    wts["resid_lambdas"] = [2.0, 0.5, 3.0]; wts["x0_lambdas"] = [1.0, 0.25, -1.0]; wts["backout_lambda"] = 1.0
    W = O.OracleWeights.from_synth(cfg, wts)
    tok = np.array([4, 8, 15, 16, 23, 42])
    # x after block 0 = 3 x0 (mid, since L//2 - 1 = 0); block 1: 0.5*3+0.25 = 1.75; block 2: 3*1.75-1 = 4.25
    # backout: 4.25 - 1.0 * 3 = 1.25 -> rms_norm(1.25 x0)
    x0 = O.embed_smear(cfg, W, tok)
    expect = O.softcap(O.rms_norm(1.25 * x0, cfg.rms_eps) @ W.m("lm_head").T, 15.0)
    np.testing.assert_allclose(O.forward_row(cfg, W, tok), expect, atol=1e-13)


def test_backout_single_layer_subtracts_x0():
    cfg = replace(get_workload("tiny").model, use_backout=True)
    wts = make_weights(cfg, init="literal")    # zero projections: block output = x0
    wts["backout_lambda"] = 0.25
    W = O.OracleWeights.from_synth(cfg, wts)
    tok = np.arange(10)
    x0 = O.embed_smear(cfg, W, tok)
    expect = O.softcap(O.rms_norm(0.75 * x0, cfg.rms_eps) @ W.m("lm_head").T, 15.0)
    np.testing.assert_allclose(O.forward_row(cfg, W, tok), expect, atol=1e-13)


# ---------------------------------------------------------------- whole model properties

def test_causality_and_window_locality():
    cfg = get_workload("tiny_all").model
    W = _weights(cfg)
    tok = make_tokens(get_workload("tiny_all")).numpy()[0][:24]
    base = O.forward_row(cfg, W, tok)
    t = 13
    tok2 = tok.copy(); tok2[t] = (tok2[t] + 1) % cfg.vocab_size
    pert = O.forward_row(cfg, W, tok2)
    np.testing.assert_array_equal(pert[:t], base[:t])
    assert np.abs(pert[t:] - base[t:]).max() > 1e-6
    # one short-window layer (W=2) plus smear: token j reaches positions j .. j+W+1 only
    c1 = replace(cfg, window_left=(2,), use_backout=False)
    b1 = O.forward_row(c1, W, tok); p1 = O.forward_row(c1, W, tok2)
    diff = np.abs(p1 - b1).max(axis=1)
    assert np.all(diff[:t] == 0) and np.all(diff[t + 4:] < 1e-15) and diff[t + 3] > 0


def test_batch_rows_independent():
    wl = get_workload("tiny_all")
    cfg = wl.model
    W = _weights(cfg)
    tok = make_tokens(wl).numpy()
    y = O.forward(cfg, W, tok)
    y_perm = O.forward(cfg, W, tok[::-1])
    np.testing.assert_array_equal(y_perm, y[::-1])


def test_logits_bounded_and_near_uniform():
    wl = get_workload("tiny_all")
    cfg = wl.model
    W = _weights(cfg)
    tok = make_tokens(wl).numpy()
    y = O.forward(cfg, W, tok)
    assert np.all(np.abs(y) < cfg.softcap)
    # N(0, 0.02) weights: near-uniform predictions, mean cross-entropy close to ln V
    tgt = np.random.default_rng(0).integers(0, cfg.vocab_size, tok.shape)
    lse = np.log(np.exp(y).sum(-1))
    ce = np.mean(lse - np.take_along_axis(y, tgt[..., None], -1)[..., 0])
    assert abs(ce - math.log(cfg.vocab_size)) < 0.5


def test_positions_subset_matches_full():
    wl = get_workload("tiny_all")
    W = _weights(wl.model)
    tok = make_tokens(wl).numpy()[1]
    full = O.forward_row(wl.model, W, tok)
    np.testing.assert_array_equal(O.forward_row(wl.model, W, tok, positions=[0, 5, 63]), full[[0, 5, 63]])


# ---------------------------------------------------------------- cross-entropy / bits per byte

def test_cross_entropy_equal_logits_is_ln_v():
    for V in (2, 7, 512):
        z = np.full((3, V), 1.25)
        np.testing.assert_allclose(O.cross_entropy(z, np.array([0, V - 1, V // 2])), math.log(V), rtol=0, atol=1e-12)


def test_cross_entropy_two_class_closed_form():
    # z = (a, b): loss(target 0) = log(1 + e^(b - a)), loss(target 1) = log(1 + e^(a - b))
    a, b = 0.7, -2.3
    z = np.array([[a, b], [a, b]])
    got = O.cross_entropy(z, np.array([0, 1]))
    np.testing.assert_allclose(got, [math.log1p(math.exp(b - a)), math.log1p(math.exp(a - b))], rtol=1e-14)


def test_cross_entropy_dominant_target_and_shift_invariance():
    z = np.zeros((1, 4))
    z[0, 2] = 30.0
    assert O.cross_entropy(z, np.array([2]))[0] < 1e-12          # log(1 + 3 e^-30)
    assert abs(O.cross_entropy(z, np.array([1]))[0] - 30.0) < 1e-9
    zr = rng.normal(size=(5, 33)) * 4
    t = rng.integers(0, 33, 5)
    np.testing.assert_allclose(O.cross_entropy(zr + 17.5, t), O.cross_entropy(zr, t), rtol=1e-12)


def test_cross_entropy_matches_torch_and_ignores_negative_targets():
    z = rng.normal(size=(40, 97)) * 5
    t = rng.integers(0, 97, 40)
    t[[3, 11]] = -1
    ref = F.cross_entropy(torch.from_numpy(z), torch.from_numpy(t), ignore_index=-1, reduction="none").numpy()
    got = O.cross_entropy(z, t)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    assert got[3] == 0.0 and got[11] == 0.0
    mean, bpb = O.loss_stats(got, t)
    np.testing.assert_allclose(mean, got[t >= 0].mean(), rtol=1e-14)
    assert math.isnan(bpb)


def test_loss_stats_bits_per_byte_hand_case():
    # losses ln2, 2 ln2, 3 ln2, 5; targets of byte lengths 1, 0 (special token), 2 and an ignored
    # position: bpb = (ln2 + 3 ln2) / (ln 2 * (1 + 2)) = 4/3; the mean counts the first three
    ln2 = math.log(2.0)
    losses = np.array([ln2, 2 * ln2, 3 * ln2, 5.0])
    targets = np.array([4, 0, 2, -1])
    token_bytes = np.array([0, 3, 2, 9, 1])
    mean, bpb = O.loss_stats(losses, targets, token_bytes)
    np.testing.assert_allclose(mean, 2 * ln2, rtol=1e-15)
    np.testing.assert_allclose(bpb, 4.0 / 3.0, rtol=1e-15)
    assert math.isnan(O.loss_stats(losses, np.array([-1, -1, -1, -1]), token_bytes)[0])
    assert math.isnan(O.loss_stats(losses, np.array([0, 0, -1, -1]), token_bytes)[1])   # no bytes


def test_model_cross_entropy_near_ln_v():
    # N(0, 0.02) weights: near-uniform predictions; the oracle's loss agrees with the direct formula
    wl = get_workload("tiny_all")
    cfg = wl.model
    y = O.forward(cfg, _weights(cfg), make_tokens(wl).numpy())
    tgt = np.random.default_rng(3).integers(0, cfg.vocab_size, y.shape[:2])
    losses = O.cross_entropy(y.reshape(-1, cfg.vocab_size), tgt.reshape(-1))
    assert abs(O.loss_stats(losses, tgt.reshape(-1))[0] - math.log(cfg.vocab_size)) < 0.5
