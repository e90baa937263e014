"""GPU tests of the backward's first part (nc_forward_loss_grad_tail and its kernels) against the
oracle: the step backwards of oracle/backward.py for each kernel, and the fp64 reverse-mode
gradient of the whole model (oracle.backward.loss_and_grads) for the four weights the call
returns.  The loss is the mean next-token cross-entropy ("NanoChat基础训练报告", loss
progression table)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from oracle import backward as OB
from synth import get_workload, make_tokens, make_weights

from tests.helpers import GRAD_MARGINS, bf16_np, binding, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"
TANH_REL = 2.0 ** -10   # hardware tanh.approx: relative error below 2^-10
BF16 = 2.0 ** -8        # round-to-nearest-even to bf16 (8 significant bits): relative error at most 2^-8


def _ops():
    return binding().ops


def _rand_bf16(shape, scale=1.0, seed=0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _mm64(a, b):
    return bf16_np(a) @ bf16_np(b)


# ---------------------------------------------------------------- operand layouts of the GEMM

@pytest.mark.parametrize("M,N,K", [(520, 384, 200), (256, 256, 64), (136, 768, 1000), (1024, 32, 8)])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_gemm_operand_layouts(M, N, K, a_mn, b_mn):
    """acc = A . B^T with A read as [M][K] or [K][M] and B as [N][K] or [K][N], fp32 out, against the
    fp64 product of the same bf16 values.  Shapes: several pair tiles with ragged M, N and K (the
    last k-block zero-filled), a single tile, a long K, and K of one 8-element step."""
    A = _rand_bf16((K, M) if a_mn else (M, K), seed=1)
    B = _rand_bf16((K, N) if b_mn else (N, K), seed=2)
    a = bf16_np(A).T if a_mn else bf16_np(A)   # [M, K]
    b = bf16_np(B).T if b_mn else bf16_np(B)   # [N, K]
    ref = a @ b.T
    got = _ops().gemm_t(A.to(DEV), B.to(DEV), a_mn=bool(a_mn), b_mn=bool(b_mn), epi="f32")
    torch.cuda.synchronize()
    # fp32 accumulation of K products of exact bf16 x bf16 values: at most K * 2^-24 of sum |a||b|
    bound = (K * 2.0 ** -24 + 2.0 ** -22) * (np.abs(a) @ np.abs(b).T) + 1e-30
    err = np.abs(got.cpu().double().numpy() - ref)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3f}"


@pytest.mark.parametrize("M,N,K", [(256, 256, 4096), (520, 384, 200), (768, 768, 16384), (64, 32, 1000)])
def test_gemm_split_k(M, N, K):
    """A weight-gradient shape (few output tiles, long K over tokens, both operands token-major)
    split over K: the ranges' fp32 slabs added in a fixed order match the fp64 product, and
    repeated calls are bit-identical."""
    ops = _ops()
    n = binding().lib().nc_op_gemm_split_ws_bytes(M, N, K, N)
    assert n > 0   # these shapes are split
    A = _rand_bf16((K, M), seed=3)
    B = _rand_bf16((K, N), seed=4)
    a, b = bf16_np(A).T, bf16_np(B).T
    got = ops.gemm_t(A.to(DEV), B.to(DEV), a_mn=True, b_mn=True, epi="f32", split=True)
    got2 = ops.gemm_t(A.to(DEV), B.to(DEV), a_mn=True, b_mn=True, epi="f32", split=True)
    torch.cuda.synchronize()
    assert torch.equal(got, got2)
    # fp32 accumulation within each range and across the (at most 16) ranges
    bound = ((K + 16) * 2.0 ** -24 + 2.0 ** -22) * (np.abs(a) @ np.abs(b).T) + 1e-30
    err = np.abs(got.cpu().double().numpy() - a @ b.T)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3f}"


def test_gemm_layout_rejects_unaligned_extent():
    A = torch.zeros((64, 60), dtype=torch.bfloat16, device=DEV)   # [K][M] with M = 60: rows not 16-byte multiples
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(RuntimeError):
        _ops().gemm_t(A, B, a_mn=True, b_mn=True)


# ---------------------------------------------------------------- cross-entropy gradient pass

@pytest.mark.parametrize("M,V,C,use_ssp", [(300, 512, 128, True), (64, 32768, 768, True), (200, 256, 256, False)])
def test_lmhead_ce_grad(M, V, C, use_ssp):
    """The recomputed lm_head's gradient epilogue against oracle.backward.softcap_ce_grad times the
    row scale, with the log-sum-exp and 1/count from the GPU's own loss pass (its inputs)."""
    A = _rand_bf16((M, C), seed=41)
    Wl = _rand_bf16((V, C), scale=0.08, seed=42)
    ssp = torch.rand((M, C // 128), generator=torch.Generator().manual_seed(43)) * 200.0 if use_ssp else None
    rs = 1.0 / np.sqrt(ssp.double().numpy().sum(1) / C + 1e-6) if use_ssp else np.ones(M)
    g = torch.Generator().manual_seed(44)
    tgt = torch.randint(0, V, (M,), generator=g, dtype=torch.int32)
    tgt[:5] = torch.tensor([0, 127, -1, V - 1, V + 5], dtype=torch.int32)   # group edges, ignored, out of range
    ops = _ops()
    sspd = ssp.to(DEV) if use_ssp else None
    part, zt = ops.lmhead_ce(A.to(DEV), Wl.to(DEV), tgt.to(DEV), ssp=sspd, C=C, cap=15.0)
    _, _, lse, invc = ops.ce_finalize(part, zt, tgt.to(DEV), V, with_lse=True)
    got = ops.lmhead_ce_grad(A.to(DEV), Wl.to(DEV), tgt.to(DEV), lse, invc, ssp=sspd, C=C, cap=15.0)
    torch.cuda.synchronize()
    t = tgt.numpy()
    n = int(((t >= 0) & (t < V)).sum())
    assert abs(float(invc.item()) - 1.0 / n) <= 1e-7 / n
    u = rs[:, None] * _mm64(A, Wl.T)
    ref = rs[:, None] * OB.softcap_ce_grad(u, t, 15.0)
    gotn = got.cpu().double().numpy()
    assert np.all(gotn[2] == 0) and np.all(gotn[4] == 0)   # ignored and out-of-range rows
    # Bound per element: each z errs by at most cap * 2^-10 (hardware tanh) and so does the row's
    # log-sum-exp, so p = exp(z - lse) errs by a factor of at most e^(2 cap 2^-10); 1 - th^2 by at most
    # 2 * 2^-10 (absolute); the bf16 output by 2^-8 of itself.
    z = 15.0 * np.tanh(u / 15.0)
    p = np.exp(z - np.log(np.exp(z).sum(-1, keepdims=True)))
    oh = np.zeros_like(p)
    keep = (t >= 0) & (t < V)
    oh[np.where(keep)[0], t[keep]] = 1.0
    scale = (rs / n * keep)[:, None]
    d = 1.0 - (z / 15.0) ** 2
    bound = scale * (p * (np.exp(2 * 15.0 * TANH_REL) - 1) * d + np.abs(p - oh) * (2 * TANH_REL)) \
        + np.abs(ref) * BF16 * 1.01 + 1e-30
    err = np.abs(gotn - ref)
    GRAD_MARGINS.append((f"ce_grad M{M} V{V}: max err / per-element bound", float(np.max(err / bound)), 1.0))
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3f}"


# ---------------------------------------------------------------- squared ReLU backward

@pytest.mark.parametrize("M,F,C", [(300, 512, 128), (1000, 3072, 768)])
def test_mlp_hidden_grad(M, F, C):
    """rs * (dy . W_proj) * 2 sqrt(h) against oracle.backward.relu2_backward(u, rs * (dy . W_proj)),
    h = relu(u)^2 rounded to bf16 as the forward stores it."""
    dy = _rand_bf16((M, C), seed=51)
    w = _rand_bf16((C, F), scale=0.05, seed=52)        # the down projection's weight [C][F]
    u = torch.randn((M, F), generator=torch.Generator().manual_seed(53), dtype=torch.float64)
    u[:, :7] = 0.0                                     # exact zeros of the hidden layer
    h = (torch.relu(u) ** 2).to(torch.bfloat16)
    ssp = torch.rand((M, C // 128), generator=torch.Generator().manual_seed(54)) * 50.0
    rs = 1.0 / np.sqrt(ssp.double().numpy().sum(1) / C + 1e-6)
    got = _ops().mlp_hidden_grad(dy.to(DEV), w.to(DEV), h.to(DEV), ssp=ssp.to(DEV))
    torch.cuda.synchronize()
    gsrc = rs[:, None] * _mm64(dy, w)
    ref = OB.relu2_backward(u.numpy(), gsrc)
    # h = relu(u)^2 rounded to bf16 errs by 2^-8 of itself, so sqrt(h) by 2^-9 of relu(u); the bf16
    # output by 2^-8; the fp32 product by C 2^-24 of sum |dy||w|
    bound = np.abs(ref) * (2 ** -9 + BF16) * 1.01 + 2 * np.maximum(u.numpy(), 0) * rs[:, None] * \
        (C * 2.0 ** -24) * (np.abs(bf16_np(dy)) @ np.abs(bf16_np(w))) + 1e-30
    err = np.abs(got.cpu().double().numpy() - ref)
    GRAD_MARGINS.append((f"relu2 backward M{M} F{F}: max err / per-element bound", float(np.max(err / bound)), 1.0))
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3f}"
    assert bool(torch.all(got.cpu()[:, :7] == 0))


# ---------------------------------------------------------------- RMSNorm backward

@pytest.mark.parametrize("M,C,with_add", [(37, 128, False), (1000, 768, True), (64, 2048, True)])
def test_rms_backward(M, C, with_add):
    gen = torch.Generator().manual_seed(61)
    x = (torch.randn((M, C), generator=gen) * torch.linspace(0.1, 5.0, M)[:, None]).float()
    g = torch.randn((M, C), generator=gen, dtype=torch.float64)
    xd = x.double().numpy()
    ssp = torch.tensor((xd.reshape(M, C // 128, 128) ** 2).sum(-1), dtype=torch.float32)   # the forward's partials
    eps = 1e-6
    rs = 1.0 / np.sqrt(ssp.double().numpy().sum(1) / C + eps)
    G = torch.tensor(rs[:, None] * g.numpy(), dtype=torch.float32)    # the GEMMs hand over rs * dL/dxn
    add = torch.randn((M, C), generator=gen).float() if with_add else None
    dxf, dxb = _ops().rms_backward(G.to(DEV), x.to(DEV), ssp.to(DEV), eps=eps,
                                   add=add.to(DEV) if with_add else None)
    torch.cuda.synchronize()
    ref = OB.rms_norm_backward(xd, G.double().numpy() / rs[:, None], eps)
    if with_add:
        ref = ref + add.double().numpy()
    scale = np.abs(G.double().numpy()) + np.abs(xd) * rs[:, None] ** 2 * np.abs(G.double().numpy() * xd).mean(
        -1, keepdims=True) + (np.abs(add.double().numpy()) if with_add else 0)
    np.testing.assert_array_less(np.abs(dxf.cpu().double().numpy() - ref), 1e-5 * scale + 1e-30)
    np.testing.assert_array_less(np.abs(dxb.cpu().double().numpy() - ref), (BF16 * 1.01 + 1e-5) * scale + 1e-30)


# ---------------------------------------------------------------- the whole tail against the fp64 gradient

def _tail_case(name, B, T, variant=None):
    wl = get_workload(name)
    cfg = replace(wl.model, **(variant or {}))
    wts = make_weights(cfg, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)[:B, :T].contiguous()
    tgt = torch.full_like(tok, -1)
    tgt[:, :-1] = tok[:, 1:]
    tgt[0, 3] = -1   # an ignored position inside a row
    return cfg, wts, tok, tgt


# Bound on the relative (Frobenius) error of each gradient.  The four gradients are sums over tokens
# of products of the backward's bf16 operands (each rounded once: 2^-8) and of the forward's
# activations, which differ from the oracle's by the forward's own error.  Where that error enters
# the softmax, an error dz in the logits changes p by a factor e^(dz - E_p dz); at the forward's
# bound (|dz| <= 5e-2) that is at most e^0.1 - 1 = 0.105 per element, which bounds the relative error
# of the lm_head's output gradient, and through it of every product downstream, plus a few 2^-8
# roundings: 0.12.
GRAD_REL = 0.12


@pytest.mark.parametrize("name,B,T,variant", [
    ("tiny_all", 2, 64, None),
    ("tiny_all", 1, 50, None),                                                   # ragged token count
    ("tiny_all", 2, 40, dict(n_layer=3, window_left=(5, 5, -1), has_ve=(1, 0, 1))),
    ("d12", 1, 256, None),
])
def test_grad_tail_matches_oracle(name, B, T, variant):
    cfg, wts, tok, tgt = _tail_case(name, B, T, variant)
    Bn = binding()
    model = Bn.Model(cfg, to_device(wts), device=DEV)
    stats, g = model.loss_grad_tail(tok.to(DEV).int().contiguous(), tgt.to(DEV).int().contiguous())
    stats2, g2 = model.loss_grad_tail(tok.to(DEV).int().contiguous(), tgt.to(DEV).int().contiguous())
    torch.cuda.synchronize()
    assert model.status() == 0
    for k in g:   # fixed-order reductions throughout: repeated calls are bit-identical
        assert torch.equal(g[k], g2[k]), k
    assert torch.equal(stats[:1], stats2[:1]) and bool(torch.isnan(stats[1]))   # no token byte lengths: no bpb
    W = O.OracleWeights.from_synth(cfg, wts)
    loss, grads = OB.loss_and_grads(cfg, W, tok.numpy(), tgt.numpy())
    assert abs(float(stats[0]) - loss) <= 2 * 5e-2   # the loss errs by at most twice the logit bound
    last = cfg.n_layer - 1
    for k, ok in (("lm_head", "lm_head"), ("wproj", f"wproj.{last}"), ("wfc", f"wfc.{last}"), ("wo", f"wo.{last}")):
        got = g[k].cpu().double().numpy()
        ref = grads[ok]
        assert got.shape == ref.shape, k
        assert np.all(np.isfinite(got)), k
        rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
        mx = float(np.abs(got - ref).max() / np.abs(ref).max())
        GRAD_MARGINS.append((f"grad {name} B{B} T{T} L{cfg.n_layer} {k}: |g-o|_F / |o|_F", rel, GRAD_REL))
        GRAD_MARGINS.append((f"grad {name} B{B} T{T} L{cfg.n_layer} {k}: max|g-o| / max|o|", mx, GRAD_REL))
        assert rel <= GRAD_REL and mx <= GRAD_REL, (k, rel, mx)


def test_grad_tail_launch_count_and_timing_classes():
    cfg, wts, tok, tgt = _tail_case("tiny_all", 2, 64)
    Bn = binding()
    model = Bn.Model(cfg, to_device(wts), device=DEV)
    assert model.grad_tail_launch_count() == 5 * cfg.n_layer + 14
    model.timing(True)
    model.loss_grad_tail(tok.to(DEV).int().contiguous(), tgt.to(DEV).int().contiguous())
    t = model.timing_read()
    model.timing(False)
    assert t["lmhead_grad"][1] == 3 and t["mlp_grad"][1] == 4 and t["oproj_grad"][1] == 1
    assert t["rmsnorm_grad"][1] == 2
    # every launch is timed on its own except the loss reduction's two kernels, timed as one
    assert sum(n for _, n in t.values()) == model.grad_tail_launch_count() - 1
