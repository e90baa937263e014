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


def test_d24_error_growth_with_depth():
    """How the logit error grows through the bf16 stack: the d24 weights cut to their first 6, 12,
    18 and 24 blocks (the same windows and value-embedding layers; backout at the cut model's
    middle), one row of 1,024 tokens, every logit against the oracle.  The margins table printed
    at the end of the run shows the headroom at each depth."""
    wl = get_workload("d24")
    cfg = wl.model
    wts = make_weights(cfg, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)[15:16, :1024].contiguous()
    for depth in (6, 12, 18, 24):
        c = replace(cfg, n_layer=depth, window_left=cfg.window_left[:depth], has_ve=cfg.has_ve[:depth])
        w = {k: v for k, v in wts.items() if "." not in k or int(k.split(".")[1]) < depth}
        w["resid_lambdas"] = wts["resid_lambdas"][:depth]
        w["x0_lambdas"] = wts["x0_lambdas"][:depth]
        _, out = _run(c, w, tok)
        ref = O.forward(c, O.OracleWeights.from_synth(c, w), tok.numpy())
        assert_parity(out.cpu().numpy(), ref, f"d24 first {depth} blocks, T=1024")
        del out


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


# ------------------------------------------------------------------------ loss path (fused lm_head + CE)

def _targets_and_bytes(tok, V, seed=11):
    """Next-token targets (the last position of each row ignored) and byte lengths of the
    vocabulary (some zero, as for special tokens)."""
    tgt = torch.full_like(tok, -1)
    tgt[:, :-1] = tok[:, 1:]
    tb = torch.randint(0, 9, (V,), generator=torch.Generator().manual_seed(seed), dtype=torch.int32)
    tb[:5] = 0
    return tgt, tb


def _loss_bound():
    # each loss errs by at most twice the largest logit error (log-sum-exp is 1-Lipschitz)
    from tests.helpers import MAX_ABS
    return 2 * MAX_ABS


@pytest.mark.parametrize("name", ["tiny", "tiny_all"])
def test_loss_path_tiny(name):
    wl = get_workload(name)
    cfg = wl.model
    wts = make_weights(cfg, init="dense")
    tok = make_tokens(wl)
    tgt, tb = _targets_and_bytes(tok, cfg.vocab_size)
    m, logits = _run(wl, wts, tok)
    loss, stats = m.forward_loss(tok.to(DEV), tgt.to(DEV), token_bytes=tb.to(DEV))
    assert m.status() == 0
    got = loss.cpu().double().numpy().reshape(-1)
    t = tgt.numpy().reshape(-1)
    ref_logits = O.forward(cfg, O.OracleWeights.from_synth(cfg, wts), tok.numpy())
    ref = O.cross_entropy(ref_logits.reshape(-1, cfg.vocab_size), t)
    np.testing.assert_allclose(got, ref, rtol=0, atol=_loss_bound())
    mean, bpb = O.loss_stats(ref, t, tb.numpy())
    np.testing.assert_allclose(stats.cpu().double().numpy(), [mean, bpb], rtol=0, atol=_loss_bound())
    # the logits path on this GPU gives the same losses up to exp2 rounding and summation order
    own = O.cross_entropy(logits.cpu().double().numpy().reshape(-1, cfg.vocab_size), t)
    np.testing.assert_allclose(got, own, rtol=0, atol=2e-4)


def test_loss_path_d12_sampled_rows_and_batch_mean():
    wl = get_workload("d12")
    cfg = wl.model
    wts = make_weights(cfg, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)
    tgt, tb = _targets_and_bytes(tok, cfg.vocab_size)
    m, logits = _run(wl, wts, tok)
    loss, stats = m.forward_loss(tok.to(DEV), tgt.to(DEV), token_bytes=tb.to(DEV))
    assert m.status() == 0
    W = O.OracleWeights.from_synth(cfg, wts)
    for r in (0, 7):
        ref_logits = O.forward_row(cfg, W, tok[r].numpy())
        ref = O.cross_entropy(ref_logits, tgt[r].numpy())
        np.testing.assert_allclose(loss[r].cpu().double().numpy(), ref, rtol=0, atol=_loss_bound())
    # whole batch: the statistics agree with fp64 cross-entropy of the logits path
    t = tgt.reshape(-1).numpy()
    own = np.concatenate([O.cross_entropy(logits[b].cpu().double().numpy(), tgt[b].numpy())
                          for b in range(tok.shape[0])])
    np.testing.assert_allclose(loss.cpu().double().numpy().reshape(-1), own, rtol=0, atol=2e-4)
    mean, bpb = O.loss_stats(own, t, tb.numpy())
    np.testing.assert_allclose(stats.cpu().double().numpy(), [mean, bpb], rtol=1e-5)


def test_loss_path_repeatable_and_launch_count():
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, seq_len_ctx=256, window_left=(64,))
    wts = make_weights(cfg, init="dense")
    tok = torch.randint(0, cfg.vocab_size, (4, 256), generator=torch.Generator().manual_seed(9), dtype=torch.int32)
    tgt, tb = _targets_and_bytes(tok, cfg.vocab_size)
    m, _ = _run(cfg, wts, tok)
    a = m.forward_loss(tok.to(DEV), tgt.to(DEV), token_bytes=tb.to(DEV))
    b = m.forward_loss(tok.to(DEV), tgt.to(DEV), token_bytes=tb.to(DEV))
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert m.launch_count(loss=True) == m.launch_count() + 2


# ------------------------------------------------------------------------ bf16 logits (opt-in output)

# bf16 keeps 8 significant bits: rounding to nearest moves a value by at most half an ulp, 2^-8 of its
# binade's lower end; a logit |z| < cap = 15 lies below 16, whose binade [8, 16) has half-ulp 2^-5
BF16_LOGIT_ULP = 2.0 ** -5


@pytest.mark.parametrize("name,B,T", [("tiny_all", 2, 64), ("d12", 1, 512)])
def test_logits_bf16_is_the_rounded_fp32_forward(name, B, T):
    """With logits_bf16 the forward writes the same soft-capped values rounded to nearest even:
    bit for bit the rounding of the fp32 forward's logits (same kernels, same accumulation), and
    within the oracle bound plus the rounding bound."""
    wl = get_workload(name)
    cfg = wl.model
    wts = make_weights(cfg, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)[:B, :T].contiguous()
    Bn = binding()
    w = to_device(wts)
    m32 = Bn.Model(cfg, w)
    m16 = Bn.Model(cfg, w, logits_bf16=True)
    z32 = m32.forward(tok.to(DEV))
    z16 = m16.forward(tok.to(DEV))
    assert m16.status() == 0 and z16.dtype == torch.bfloat16
    assert torch.equal(z16, z32.to(torch.bfloat16))
    ref = O.forward(cfg, O.OracleWeights.from_synth(cfg, wts), tok.numpy())
    g = z16.float().cpu().numpy()
    d = np.abs(g - ref)
    assert d.max() <= 5e-2 + BF16_LOGIT_ULP and d.sum() / np.abs(ref).sum() <= 1e-2 + 2 ** -8
    # the host entry point copies half the bytes out
    out_h = torch.empty((B, T, cfg.vocab_size), dtype=torch.bfloat16).pin_memory()
    m16.forward_host(tok.pin_memory(), out_h)
    assert torch.equal(out_h, z16.cpu())


@pytest.mark.parametrize("name,rows,T0", [("tiny_all", None, 40), ("d12", 2, 2040)])
def test_logits_bf16_prefill_and_decode(name, rows, T0):
    """bf16 logits of the prefill and of a decode step are the rounded fp32 ones.  At d12 the
    decode step's lm_head (4,096 blocks of 8 vocabulary rows) runs on persistent CTAs."""
    wl = get_workload(name)
    cfg = wl.model
    w = to_device(make_weights(cfg, seed=wl.seed, init=wl.init))
    tok = make_tokens(wl)[:rows].to(DEV)
    T_max = 64 if name == "tiny_all" else wl.T
    Bn = binding()
    outs = {}
    for bf in (False, True):
        m = Bn.Model(cfg, w, logits_bf16=bf)
        cache = m.kv_cache(tok.shape[0], T_max)
        pre = m.prefill(tok[:, :T0].contiguous(), cache, T_max)
        dec = m.decode_step(tok[:, T0 - 1].contiguous(), tok[:, T0].contiguous(), T0, cache, T_max)
        assert m.status() == 0
        outs[bf] = (pre, dec)
    assert outs[True][0].dtype == torch.bfloat16 and outs[True][1].dtype == torch.bfloat16
    assert torch.equal(outs[True][0], outs[False][0].to(torch.bfloat16))
    assert torch.equal(outs[True][1], outs[False][1].to(torch.bfloat16))
