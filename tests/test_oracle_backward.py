"""Pins of the backward oracle (oracle/backward.py) on CPU: its restated forward reproduces
the forward oracle and the loss oracle, and every kind of gradient equals central finite
differences of the fp64 loss."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from oracle import backward as OB
from synth import get_workload, make_tokens, make_weights

VARIANTS = [dict(), dict(n_layer=3, window_left=(5, 5, -1), has_ve=(1, 0, 1), seq_len_ctx=64)]


def _case(variant, T=24):
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, **variant)
    W = O.OracleWeights.from_synth(cfg, make_weights(cfg, init="dense"))
    tok = make_tokens(wl).numpy()[:, :T]
    tgt = np.full_like(tok, -1)
    tgt[:, :-1] = tok[:, 1:]
    tgt[0, 3] = -1   # an ignored position inside a row
    return cfg, W, tok, tgt


@pytest.mark.parametrize("variant", VARIANTS)
def test_restated_forward_and_loss_match_the_oracles(variant):
    cfg, W, tok, tgt = _case(variant)
    P = OB.parameters(W)
    logits = []
    for b in range(tok.shape[0]):
        got = OB.forward_row(cfg, P, torch.as_tensor(tok[b], dtype=torch.long)).numpy()
        ref = O.forward_row(cfg, W, tok[b])
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
        logits.append(ref)
    ref_losses = O.cross_entropy(np.concatenate(logits), tgt.reshape(-1))
    ref_mean, _ = O.loss_stats(ref_losses, tgt.reshape(-1))
    np.testing.assert_allclose(float(OB.mean_loss(cfg, P, tok, tgt)), ref_mean, rtol=1e-13)


@pytest.mark.parametrize("variant", VARIANTS)
def test_gradients_match_central_differences(variant):
    cfg, W, tok, tgt = _case(variant)
    loss, grads = OB.loss_and_grads(cfg, W, tok, tgt)
    rng = np.random.default_rng(5)
    h = 1e-6
    checked = 0
    for name, g in grads.items():
        flat = np.abs(g).reshape(-1)
        picks = {int(flat.argmax()), int(rng.integers(0, flat.size))}
        for idx in picks:
            def loss_at(delta):
                P = OB.parameters(W)
                P[name].view(-1)[idx] += delta
                return float(OB.mean_loss(cfg, P, tok, tgt))
            fd = (loss_at(h) - loss_at(-h)) / (2 * h)
            an = float(g.reshape(-1)[idx])
            assert abs(fd - an) <= 1e-7 + 1e-5 * abs(an), (name, idx, fd, an)
            checked += 1
    assert checked >= 2 * len(grads) - 3   # every tensor, its largest entry and a random one
    assert np.isfinite(loss)


def test_gradient_is_zero_on_embedding_rows_of_absent_tokens():
    cfg, W, tok, tgt = _case(VARIANTS[1])
    _, grads = OB.loss_and_grads(cfg, W, tok, tgt)
    absent = np.setdiff1d(np.arange(cfg.vocab_size), tok.reshape(-1))
    assert absent.size > 0
    assert np.all(grads["wte"][absent] == 0.0)
    assert np.all(grads["ve.0"][absent] == 0.0)
    # a token seen before a row's last position feeds later counted positions (causality); one seen
    # only at a row's last position feeds nothing but that position's ignored logits
    present = np.unique(tok[:, :-1].reshape(-1))
    assert np.all(np.abs(grads["wte"][present]).sum(1) > 0)
    last_only = np.setdiff1d(np.unique(tok[:, -1]), present)
    assert np.all(grads["wte"][last_only] == 0.0)
    assert np.all(np.abs(grads["lm_head"]).sum(1) > 0)   # every vocabulary row enters the softmax


# ---------------------------------------------------------------- step backwards

def _central(f, x, h=1e-6):
    """Central differences of the scalar f at every entry of x (fp64)."""
    g = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        e = np.zeros_like(x)
        e[idx] = h
        g[idx] = (f(x + e) - f(x - e)) / (2 * h)
    return g


@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.5])
def test_rms_norm_backward_matches_central_differences(eps):
    rng = np.random.default_rng(11)
    x = rng.normal(size=(3, 16)) * np.array([[0.1], [1.0], [7.0]])   # RMS far from 1 in every row
    w = rng.normal(size=(3, 16))                                      # L = sum(w * rms(x)): g = w
    loss = lambda xx: float((w * (xx / np.sqrt((xx * xx).mean(-1, keepdims=True) + eps))).sum())
    got = OB.rms_norm_backward(x, w, eps)
    np.testing.assert_allclose(got, _central(loss, x), rtol=1e-6, atol=1e-8)


def test_rms_norm_backward_is_orthogonal_to_x_without_eps():
    """At eps = 0 the norm is invariant to scaling x, so its gradient has no component along x."""
    rng = np.random.default_rng(12)
    x, g = rng.normal(size=(5, 64)) * 3.0, rng.normal(size=(5, 64))
    dx = OB.rms_norm_backward(x, g, 0.0)
    np.testing.assert_allclose((dx * x).sum(-1), 0.0, atol=1e-12)
    assert np.abs(dx).max() > 0.1


def test_softcap_ce_grad_matches_central_differences_and_ignores_rows():
    rng = np.random.default_rng(13)
    M, V, cap = 5, 9, 15.0
    u = rng.normal(size=(M, V)) * 8.0          # some logits well into the cap's curve
    t = np.array([2, -1, 8, 0, 9])             # one ignored (negative), one out of range
    def loss(uu):
        z = cap * np.tanh(uu / cap)
        keep = (t >= 0) & (t < V)
        lse = np.log(np.exp(z[keep]).sum(-1))
        return float((lse - z[keep, t[keep]]).mean())
    got = OB.softcap_ce_grad(u, t, cap)
    # the differences' rounding floor: 2 * 2^-52 * |loss| (about 3) / h (1e-6), about 1.3e-9
    np.testing.assert_allclose(got, _central(loss, u), rtol=1e-6, atol=3e-9)
    assert np.all(got[1] == 0) and np.all(got[4] == 0)


def test_softcap_ce_grad_rows_balance_and_large_cap_limit():
    """Each counted row of (grad / (1 - (z/cap)^2)) sums to zero (softmax minus one-hot); with the
    cap far above the logits the factor is 1 and the gradient is (softmax - onehot) / n."""
    rng = np.random.default_rng(14)
    u = rng.normal(size=(4, 7))
    t = np.array([1, 3, 0, 6])
    g = OB.softcap_ce_grad(u, t, 15.0)
    z = 15.0 * np.tanh(u / 15.0)
    np.testing.assert_allclose((g / (1 - (z / 15.0) ** 2)).sum(-1), 0.0, atol=1e-15)
    big = OB.softcap_ce_grad(u, t, 1e8)
    p = np.exp(u) / np.exp(u).sum(-1, keepdims=True)
    p[np.arange(4), t] -= 1
    np.testing.assert_allclose(big, p / 4, rtol=1e-9, atol=1e-12)


def test_relu2_backward_matches_central_differences():
    rng = np.random.default_rng(15)
    u = rng.normal(size=(4, 6))
    u[u.__abs__() < 1e-3] = 0.5   # keep away from the kink at 0
    w = rng.normal(size=(4, 6))
    got = OB.relu2_backward(u, w)
    np.testing.assert_allclose(got, _central(lambda v: float((w * np.maximum(v, 0) ** 2).sum()), u), rtol=1e-6,
                               atol=1e-9)
    assert np.all(got[u < 0] == 0)
