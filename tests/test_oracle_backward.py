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
