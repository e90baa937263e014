"""GPU tests of the 8-bit (e4m3, tensorwise-scaled) path against the oracle (oracle/fp8.py):
the quantiser's codes, the kind::f8f6f4 product, and the whole forward with every linear layer in
e4m3 ("Nanochat在nanoGPT之上的新增功能", section 1 feature table, FP8 row; "nanochat — 架构与原理",
section 4)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from oracle import fp8 as OF
from synth import get_workload, make_tokens, make_weights

from tests.helpers import GRAD_MARGINS, binding, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ops():
    return binding().ops


def _f32(x):
    return np.asarray(x, dtype=np.float32)


# ---------------------------------------------------------------- quantiser

@pytest.mark.parametrize("src_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,C", [(300, 768), (64, 128), (1000, 3072)])
def test_fp8_quantize_codes_are_the_oracles(src_dtype, M, C):
    """Without a row scale the kernel's code decision is round_e4m3(float32(float32(v * 448) / amax))
    (a correctly rounded division): the oracle's rounding of that float32 value gives every code
    exactly.  For bf16 v it is also the exact-arithmetic decision (v * 448 is exact and a tie stays a
    tie), so the codes equal oracle.fp8's rounding of v * (448 / amax) in fp64 as well."""
    g = torch.Generator().manual_seed(7)
    src = torch.randn((M, C), generator=g) * torch.logspace(-3, 1, C)[None, :]
    src[3, 5] = 37.0   # an outlier sets the scale
    src = src.to(src_dtype)
    q, inv = _ops().fp8_quantize(src.to(DEV))
    torch.cuda.synchronize()
    v = _f32(src.float().numpy())
    amax = np.float32(np.max(np.abs(v)))
    assert float(inv.item()) == float(amax / np.float32(448.0))
    want = OF.round_e4m3(((v * np.float32(448.0)) / amax).astype(np.float32).astype(np.float64))
    got = q.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got, want)
    assert np.max(np.abs(got)) == 448.0
    if src_dtype == torch.bfloat16:   # the fp64 decision of the oracle itself
        assert np.array_equal(got, OF.round_e4m3(v.astype(np.float64) * OF.tensor_scale(v.astype(np.float64))))


def test_fp8_quantize_zero_tensor_and_saturation():
    src = torch.zeros((40, 256), device=DEV)
    q, inv = _ops().fp8_quantize(src)
    torch.cuda.synchronize()
    assert float(inv.item()) == 1.0 and bool(torch.all(q.float() == 0))


def test_fp8_quantize_row_scaled():
    """The normed residual stream: v = x * rs, rs = 1 / sqrt(mean x^2 + eps) from the partial sums.
    rs is computed with the hardware reciprocal square root (within 2 ulp of the oracle's), so a
    code may differ from the oracle's by one step where v * s lies that close to a rounding
    boundary: at most one e4m3 step (2^-3 of the binade's lower end) anywhere, on a small fraction."""
    g = torch.Generator().manual_seed(8)
    M, C = 512, 768
    x = torch.randn((M, C), generator=g) * torch.linspace(0.05, 8.0, M)[:, None]
    xd = x.double().numpy()
    ssp = torch.tensor((xd.reshape(M, C // 128, 128) ** 2).sum(-1), dtype=torch.float32)
    q, inv = _ops().fp8_quantize(x.to(DEV), ssp=ssp.to(DEV), eps=1e-6)
    torch.cuda.synchronize()
    a = O.rms_norm(xd, 1e-6)
    s = OF.tensor_scale(a)
    want = OF.round_e4m3(a * s)
    got = q.float().cpu().numpy().astype(np.float64)
    assert abs(float(inv.item()) * s - 1.0) < 1e-6
    step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(want), 2.0 ** -6))) - 3)
    assert np.all(np.abs(got - want) <= step * 1.0001)
    frac = float(np.mean(got != want))
    GRAD_MARGINS.append(("fp8 quantise, row-scaled: fraction of codes one step off", frac, 0.01))
    assert frac <= 0.01


# ---------------------------------------------------------------- product

@pytest.mark.parametrize("M,N,K", [(520, 384, 256), (256, 768, 768), (300, 3072, 768), (1000, 768, 3072)])
def test_gemm_fp8(M, N, K):
    """kind::f8f6f4 product of e4m3 operands, dequantised by the two scales: products of e4m3 values
    are exact in fp32, so the error is the fp32 accumulation's, K 2^-24 of sum |a||b| (times the scales)."""
    g = torch.Generator().manual_seed(9)
    A8 = (torch.randn((M, K), generator=g) * 30).to(torch.float8_e4m3fn)
    B8 = (torch.randn((N, K), generator=g) * 30).to(torch.float8_e4m3fn)
    sa = torch.tensor([0.0123], dtype=torch.float32)
    sb = torch.tensor([0.5], dtype=torch.float32)
    got = _ops().gemm_fp8(A8.to(DEV), B8.to(DEV), sa.to(DEV), sb.to(DEV), epi="f32")
    torch.cuda.synchronize()
    a = A8.float().numpy().astype(np.float64)
    b = B8.float().numpy().astype(np.float64)
    k = float(sa[0]) * float(sb[0])
    ref = (a @ b.T) * k
    bound = ((K + 2) * 2.0 ** -24) * (np.abs(a) @ np.abs(b).T) * k + 1e-30
    err = np.abs(got.cpu().double().numpy() - ref)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3f}"


# ---------------------------------------------------------------- one 8-bit linear layer

@pytest.mark.parametrize("M,N,K", [(300, 768, 768), (1024, 3072, 768), (256, 768, 3072)])
def test_fp8_linear_matches_oracle(M, N, K):
    """An 8-bit linear layer as the 8-bit forward runs it: the input (fp32) and the weight (bf16) each
    quantised at their tensorwise scale by the GPU, then the e4m3 product dequantised.  Both sides
    decide each code on the same float32 product v * s (the quantiser test pins that the GPU's
    codes are the oracle's rounding of it), so the result equals oracle.fp8's definition,
    round(x s_x) . round(w s_w)^T / (s_x s_w), to the fp32 accumulation (K 2^-24 of sum |a||b|)."""
    g = torch.Generator().manual_seed(10)
    x = torch.randn((M, K), generator=g) * torch.linspace(0.2, 3.0, K)[None, :]
    w = (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16)
    ops = _ops()
    x8, ix = ops.fp8_quantize(x.to(DEV))
    w8, iw = ops.fp8_quantize(w.to(DEV))
    got = ops.gemm_fp8(x8, w8, ix, iw, epi="f32")
    torch.cuda.synchronize()
    xv, wv = _f32(x.numpy()), _f32(w.float().numpy())
    ax, aw = np.float32(np.max(np.abs(xv))), np.float32(np.max(np.abs(wv)))
    qa = OF.round_e4m3(((xv * np.float32(448.0)) / ax).astype(np.float32).astype(np.float64))
    qb = OF.round_e4m3(((wv * np.float32(448.0)) / aw).astype(np.float32).astype(np.float64))
    k = float(ax / np.float32(448.0)) * float(aw / np.float32(448.0))
    ref = (qa @ qb.T) * k
    bound = ((K + 2) * 2.0 ** -24) * (np.abs(qa) @ np.abs(qb).T) * k + 1e-30
    err = np.abs(got.cpu().double().numpy() - ref)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3f}"
    # and against oracle.fp8.fp8_linear itself (fp64 scaling): the codes differ only where a float32
    # quotient lies within an ulp of a rounding tie (about 2^-24 / 2^-4 of the elements)
    full = OF.fp8_linear(x.numpy().astype(np.float64), w.float().numpy().astype(np.float64))
    rel = float(np.abs(got.cpu().double().numpy() - full).sum() / np.abs(full).sum())
    GRAD_MARGINS.append((f"fp8 linear {M}x{N}x{K} vs oracle.fp8.fp8_linear: sum|g - o| / sum|o|", rel, 1e-3))
    assert rel <= 1e-3


# ---------------------------------------------------------------- the 8-bit forward

# Bound of the whole 8-bit forward against the oracle's.  The two quantise the same tensors, but the
# GPU keeps q, k, v, y and h in bf16 and accumulates in fp32 as the bf16 path does, so after the
# first layer the quantisers' inputs differ by more than half an e4m3 step in many places and the
# two runs' rounding errors are no longer the same: each is the exact forward plus a quantisation
# error of its own.  By the triangle inequality |gpu - ref8| <= |gpu - exact| + |exact - ref8|, and
# the GPU's quantisation error is of the size of the oracle's (same scales, same e4m3 grid), so the
# bound is twice the oracle's own 8-bit error (ref8 against the exact oracle forward, computed here)
# plus the bf16 path's bound (max 5e-2, mean relative 1e-2).  Below: the GPU's output must also sit a
# quantisation error (not just a bf16 error) away from the exact forward, or it is not quantising.


@pytest.mark.parametrize("name,B,T,variant", [
    ("tiny_all", 2, 64, None),
    ("tiny_all", 1, 50, dict(n_layer=3, window_left=(5, 5, -1), has_ve=(1, 0, 1))),
    ("d12", 1, 256, None),
])
def test_fp8_forward_matches_oracle(name, B, T, variant):
    wl = get_workload(name)
    cfg = replace(wl.model, **(variant or {}))
    wts = make_weights(cfg, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)[:B, :T].contiguous()
    Bn = binding()
    m = Bn.Model(cfg, to_device(wts), fp8=True)
    z = m.forward(tok.to(DEV))
    z2 = m.forward(tok.to(DEV))
    torch.cuda.synchronize()
    assert m.status() == 0
    assert torch.equal(z, z2)   # scales and codes are the same on every run
    W = O.OracleWeights.from_synth(cfg, wts)
    ref = OF.forward_fp8(cfg, W, tok.numpy())
    exact = O.forward(cfg, W, tok.numpy())
    g = z.cpu().double().numpy()
    assert np.all(np.isfinite(g))

    def err(a, b):
        d = np.abs(a - b)
        return float(d.max()), float(d.sum() / np.abs(b).sum())

    q_max, q_rel = err(ref, exact)        # the oracle's own 8-bit error
    g_max, g_rel = err(g, ref)
    x_max, x_rel = err(g, exact)
    b_max, b_rel = 2 * q_max + 5e-2, 2 * q_rel + 1e-2
    tag = f"fp8 forward {name} B{B} T{T} L{cfg.n_layer}"
    GRAD_MARGINS.append((f"{tag}: max |g - o8|", g_max, b_max))
    GRAD_MARGINS.append((f"{tag}: sum|g - o8| / sum|o8|", g_rel, b_rel))
    GRAD_MARGINS.append((f"{tag}: oracle 8-bit vs exact, sum|o8 - o| / sum|o|", q_rel, 1.0))
    assert g_max <= b_max and g_rel <= b_rel, (g_max, g_rel, q_max, q_rel)
    # quantising for real: about the oracle's 8-bit error away from the exact forward, far above the
    # bf16 path's (which stays under 1e-2 mean relative)
    assert 0.25 * q_rel <= x_rel <= 2 * q_rel + 1e-2, (x_rel, q_rel)


def test_fp8_loss_path_and_rejections():
    wl = get_workload("tiny_all")
    cfg = wl.model
    wts = make_weights(cfg, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)
    tgt = torch.full_like(tok, -1)
    tgt[:, :-1] = tok[:, 1:]
    Bn = binding()
    m = Bn.Model(cfg, to_device(wts), fp8=True)
    z = m.forward(tok.to(DEV))
    loss, stats = m.forward_loss(tok.to(DEV), tgt.to(DEV))
    torch.cuda.synchronize()
    own = O.cross_entropy(z.cpu().double().numpy().reshape(-1, cfg.vocab_size), tgt.numpy().reshape(-1))
    np.testing.assert_allclose(loss.cpu().double().numpy().reshape(-1), own, rtol=0, atol=2e-4)
    with pytest.raises(RuntimeError):
        m.kv_cache(2, 64)
    with pytest.raises(RuntimeError):
        m.loss_grad_tail(tok.to(DEV), tgt.to(DEV))
    ve = sum(1 for v in cfg.has_ve if v)
    assert m.launch_count() == 2 + 12 * cfg.n_layer + ve + 2
    m.timing(True)
    m.forward(tok.to(DEV))
    t = m.timing_read()
    m.timing(False)
    assert t["fp8_quantize"][1] == 7 * cfg.n_layer + 2   # the fc output's maximum comes from its epilogue
    assert sum(n for _, n in t.values()) == m.launch_count()
