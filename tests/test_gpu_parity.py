"""Whole-forward parity: nc_forward (C ABI, CUDA kernels) against the fp64 oracle on the same
seeded weights and tokens, for all five workloads.  Small workloads are compared on every
logit; the full-size ones (the configuration bench.py times) on whole batch rows or on sampled
positions of a row, which the oracle computes independently (rows are independent)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from synth import get_workload, make_tokens, make_weights
from tests.helpers import assert_parity, binding, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(wl_or_cfg, wts, tok):
    cfg = wl_or_cfg.model if hasattr(wl_or_cfg, "model") else wl_or_cfg
    B = binding()
    m = B.Model(cfg, to_device(wts))
    out = m.forward(tok.to(DEV))
    assert m.status() == 0
    return m, out


@pytest.mark.parametrize("name", ["tiny", "tiny_dense", "tiny_all"])
def test_tiny_workloads_every_logit(name):
    wl = get_workload(name)
    wts = make_weights(wl.model, init=wl.init)
    tok = make_tokens(wl)
    _, out = _run(wl, wts, tok)
    ref = O.forward(wl.model, O.OracleWeights.from_synth(wl.model, wts), tok.numpy())
    assert_parity(out.cpu().numpy(), ref, name)


@pytest.mark.parametrize("variant", [
    dict(embed_norm=True),
    dict(window_left=(5,)),
    dict(smear_gate_channels=32, ve_gate_channels=64, ve_gate_scale=2.0),
    dict(n_layer=3, window_left=(16, 16, -1), has_ve=(1, 0, 1)),
])
def test_tiny_all_variants(variant):
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, **variant)
    wts = make_weights(cfg, init="dense")
    tok = make_tokens(wl)
    _, out = _run(cfg, wts, tok)
    ref = O.forward(cfg, O.OracleWeights.from_synth(cfg, wts), tok.numpy())
    assert_parity(out.cpu().numpy(), ref, str(variant))


def test_ragged_sequence_and_batch():
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, seq_len_ctx=200, window_left=(37,))
    wts = make_weights(cfg, init="dense")
    tok = torch.randint(0, cfg.vocab_size, (3, 157), generator=torch.Generator().manual_seed(5), dtype=torch.int32)
    _, out = _run(cfg, wts, tok)
    ref = O.forward(cfg, O.OracleWeights.from_synth(cfg, wts), tok.numpy())
    assert_parity(out.cpu().numpy(), ref, "ragged")


def test_single_token_sequence():
    wl = get_workload("tiny_all")
    wts = make_weights(wl.model, init="dense")
    tok = torch.tensor([[7], [500]], dtype=torch.int32)
    _, out = _run(wl, wts, tok)
    ref = O.forward(wl.model, O.OracleWeights.from_synth(wl.model, wts), tok.numpy())
    assert_parity(out.cpu().numpy(), ref, "T=1")


@pytest.mark.parametrize("name,rows,stride", [("d12", (0, 7), 1), ("d20", (3,), 1), ("d12_long", (1,), 8),
                                              ("d24", (15,), 4)])
def test_full_size_workloads_sampled(name, rows, stride):
    """Full-size batch through nc_forward; the oracle recomputes whole batch rows (stride 1) or
    every stride-th position of a row (its final hidden state is computed for all positions)."""
    wl = get_workload(name)
    wts = make_weights(wl.model, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)
    _, out = _run(wl, wts, tok)
    W = O.OracleWeights.from_synth(wl.model, wts)
    for r in rows:
        pos = np.arange(0, wl.T, stride)
        if stride > 1:
            pos = np.unique(np.r_[pos, wl.T - 1])
        ref = O.forward_row(wl.model, W, tok[r].numpy(), positions=pos)
        got = out[r, torch.from_numpy(pos).to(DEV)].cpu().numpy()
        assert_parity(got, ref, f"{name} row {r}")


def test_bitwise_repeatable_and_row_independent():
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, seq_len_ctx=256, window_left=(64,))
    wts = make_weights(cfg, init="dense")
    tok = torch.randint(0, cfg.vocab_size, (4, 256), generator=torch.Generator().manual_seed(9), dtype=torch.int32)
    m, a = _run(cfg, wts, tok)
    b = m.forward(tok.to(DEV))
    assert torch.equal(a, b)
    perm = torch.tensor([2, 0, 3, 1])
    c = m.forward(tok[perm].contiguous().to(DEV))
    assert torch.equal(c, a[perm.to(DEV)])


def test_causality_bitwise():
    wl = get_workload("tiny_all")
    wts = make_weights(wl.model, init="dense")
    tok = make_tokens(wl)
    m, a = _run(wl, wts, tok)
    t = 40
    tok2 = tok.clone()
    tok2[:, t] = (tok2[:, t] + 1) % wl.model.vocab_size
    b = m.forward(tok2.to(DEV))
    assert torch.equal(a[:, :t], b[:, :t])
    assert not torch.equal(a[:, t:], b[:, t:])
