"""Kernel-level parity: each CUDA kernel (through the C ABI of nc_ops.h) against the oracle
step it implements, on seeded inputs, at sizes that span several tiles and a ragged tail."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from tests.helpers import bf16_np, binding

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rand_bf16(shape, scale=1.0, seed=0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _ops():
    return binding().ops


# ------------------------------------------------------------------------ GEMM mainloop

@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 96, 128), (1000, 768, 768), (64, 512, 128),
                                   (129, 2304, 768), (384, 3072, 192), (130, 32, 3072)])
def test_gemm_bf16(M, N, K):
    A = _rand_bf16((M, K), seed=1)
    Bm = _rand_bf16((N, K), seed=2)
    out = _ops().gemm(A.to(DEV), Bm.to(DEV), "bf16")
    torch.cuda.synchronize()
    ref = bf16_np(A) @ bf16_np(Bm).T
    got = bf16_np(out)
    np.testing.assert_allclose(got, ref, rtol=2 ** -7, atol=2e-3 * math.sqrt(K))


def test_gemm_large_sampled_rows():
    # d12 q|k|v shape: 128 row tiles x 9 column tiles on a persistent grid
    M, N, K = 16384, 2304, 768
    A = _rand_bf16((M, K), seed=3)
    Bm = _rand_bf16((N, K), scale=0.05, seed=4)
    out = _ops().gemm(A.to(DEV), Bm.to(DEV), "bf16")
    torch.cuda.synchronize()
    rows = np.r_[0:3, 127:131, 8191, 16255:16260, 16383, np.random.default_rng(0).integers(0, M, 64)]
    ref = bf16_np(A[rows]) @ bf16_np(Bm).T
    np.testing.assert_allclose(bf16_np(out[rows]), ref, rtol=2 ** -7, atol=2e-3 * math.sqrt(K) * 0.05)


def _groups(x, n=128):
    """Per-128-column partial sums along the last axis: [..., C] -> [..., C/128]."""
    return x.reshape(*x.shape[:-1], x.shape[-1] // n, n).sum(-1)


def _ssp_of(x64):
    return _groups(x64 * x64)


@pytest.mark.parametrize("M,N,K,a,b,use_y,use_xm,x_out", [
    (300, 768, 768, 1.0, 0.0, False, False, True),        # attention out-proj form (in place)
    (257, 768, 3072, 0.9, 0.2, True, True, True),         # MLP down-proj + backout cache + next block's mix
    (130, 1280, 512, 1.0, -0.5, True, False, False),      # last block: backout, no stream written
    (64, 128, 512, 1.1, 0.3, True, False, True),          # tiny width: the pair's second CTA idle
    (16, 768, 768, 1.0, 0.0, False, False, True),         # decode-sized: 16 rows, one 32-token tile
    (1000, 1536, 768, 0.95, 0.1, True, False, True),      # d24 width, ragged rows
    (5000, 1280, 5120, 0.9, 0.25, True, False, True),     # d20 shapes: 192-token tiles, ragged last tile
])
def test_gemm_residual_epilogue(M, N, K, a, b, use_y, use_xm, x_out):
    g = torch.Generator().manual_seed(M + N + K)
    A = _rand_bf16((M, K), seed=5)
    Bm = _rand_bf16((N, K), scale=0.02, seed=6)
    x = torch.randn((M, N), generator=g)
    Y = torch.randn((M, N), generator=g) if use_y else None
    xd = x.to(DEV)
    xm = torch.full((M, N), float("nan"), device=DEV) if use_xm else None
    xb, ssp = _ops().gemm_residual(A.to(DEV), Bm.to(DEV), xd, a, b, Y.to(DEV) if use_y else None,
                                   xd if x_out else None, xm)
    torch.cuda.synchronize()
    xr = x.double().numpy() + bf16_np(A) @ bf16_np(Bm).T
    xp = a * xr + (b * Y.double().numpy() if use_y else 0.0)
    if use_xm:
        np.testing.assert_allclose(xm.cpu().double().numpy(), xr, rtol=1e-5, atol=1e-4)
    if x_out:
        np.testing.assert_allclose(xd.cpu().double().numpy(), xp, rtol=1e-5, atol=1e-4)
    else:
        np.testing.assert_array_equal(xd.cpu().numpy(), x.numpy())
    np.testing.assert_allclose(bf16_np(xb), xp, rtol=2 ** -8, atol=1e-4)
    np.testing.assert_allclose(ssp.cpu().double().numpy(), _ssp_of(xp), rtol=1e-5, atol=1e-4)


def test_gemm_residual_full_size_sampled_rows():
    """The d12 MLP down projection with the next block's mix at full size (M = 16384: 224-token
    tiles, the last one ragged), checked on sampled rows."""
    M, N, K, a, b = 16384, 768, 3072, 0.9, 0.2
    g = torch.Generator().manual_seed(21)
    A = _rand_bf16((M, K), seed=22)
    Bm = _rand_bf16((N, K), scale=0.02, seed=23)
    x = torch.randn((M, N), generator=g)
    Y = torch.randn((M, N), generator=g)
    xd = x.to(DEV)
    xb, ssp = _ops().gemm_residual(A.to(DEV), Bm.to(DEV), xd, a, b, Y.to(DEV), xd, None)
    torch.cuda.synchronize()
    rows = np.unique(np.r_[0:3, 223:226, 8191, 16351:16353, 16383, np.random.default_rng(1).integers(0, M, 48)])
    xp = a * (x[rows].double().numpy() + bf16_np(A[rows]) @ bf16_np(Bm).T) + b * Y[rows].double().numpy()
    np.testing.assert_allclose(xd[rows].cpu().double().numpy(), xp, rtol=1e-5, atol=1e-4)
    np.testing.assert_allclose(bf16_np(xb[rows]), xp, rtol=2 ** -8, atol=1e-4)
    np.testing.assert_allclose(ssp[rows].cpu().double().numpy(), _ssp_of(xp), rtol=1e-5, atol=1e-4)


def test_gemm_relu2_and_softcap_row_scaled():
    M, N, K = 257, 1024, 768
    A = _rand_bf16((M, K), seed=8)
    Bm = _rand_bf16((N, K), scale=0.05, seed=9)
    acc = bf16_np(A) @ bf16_np(Bm).T
    ssp = torch.rand((M, K // 128), generator=torch.Generator().manual_seed(3)) * 200.0
    rs = 1.0 / np.sqrt(ssp.double().numpy().sum(1) / K + 1e-6)
    h = _ops().gemm(A.to(DEV), Bm.to(DEV), "relu2_bf16", ssp=ssp.to(DEV), C=K)
    z = _ops().gemm(A.to(DEV), Bm.to(DEV), "softcap_f32", ssp=ssp.to(DEV), C=K, cap=15.0)
    z1 = _ops().gemm(A.to(DEV), Bm.to(DEV), "softcap_f32", cap=15.0)
    torch.cuda.synchronize()
    np.testing.assert_allclose(bf16_np(h), O.relu2(rs[:, None] * acc), rtol=2 ** -7, atol=1e-3)
    # the soft-cap uses the hardware tanh (tanh.approx.f32, relative error below 2^-10 by its
    # documentation), so |cap * tanh| may err by up to cap * 2^-10 on top of the fp32 accumulation
    np.testing.assert_allclose(z.cpu().double().numpy(), O.softcap(rs[:, None] * acc, 15.0), rtol=0,
                               atol=15.0 * 2 ** -10)
    np.testing.assert_allclose(z1.cpu().double().numpy(), O.softcap(acc, 15.0), rtol=0, atol=15.0 * 2 ** -10)
    # bf16 logits: the same values rounded to nearest even, bit for bit
    zb = _ops().gemm(A.to(DEV), Bm.to(DEV), "softcap_bf16", ssp=ssp.to(DEV), C=K, cap=15.0)
    torch.cuda.synchronize()
    assert torch.equal(zb, z.to(torch.bfloat16))
    assert float(z1.abs().max()) < 15.0


# ------------------------------------------------------------------------ fused lm_head + cross-entropy

@pytest.mark.parametrize("M,V,C,use_ssp", [(257, 1024, 768, True), (130, 992, 128, False)])
def test_lmhead_cross_entropy(M, V, C, use_ssp):
    A = _rand_bf16((M, C), seed=21)
    Wl = _rand_bf16((V, C), scale=0.08, seed=22)
    acc = bf16_np(A) @ bf16_np(Wl).T
    ssp = torch.rand((M, C // 128), generator=torch.Generator().manual_seed(23)) * 200.0 if use_ssp else None
    rs = 1.0 / np.sqrt(ssp.double().numpy().sum(1) / C + 1e-6) if use_ssp else np.ones(M)
    g = torch.Generator().manual_seed(24)
    tgt = torch.randint(0, V, (M,), generator=g, dtype=torch.int32)
    tgt[:6] = torch.tensor([0, 127, 128, V - 1, -1, V - 97], dtype=torch.int32)   # group edges, ignored, last group
    tb = torch.randint(0, 9, (V,), generator=g, dtype=torch.int32)
    tb[:3] = 0
    ops = _ops()
    sspd = ssp.to(DEV) if use_ssp else None
    part, zt = ops.lmhead_ce(A.to(DEV), Wl.to(DEV), tgt.to(DEV), ssp=sspd, C=C, cap=15.0)
    loss, stats = ops.ce_finalize(part, zt, tgt.to(DEV), V, token_bytes=tb.to(DEV))
    z_gpu = ops.gemm(A.to(DEV), Wl.to(DEV), "softcap_f32", ssp=sspd, C=C if use_ssp else 0, cap=15.0)
    torch.cuda.synchronize()
    got = loss.cpu().double().numpy()
    t = tgt.numpy()
    # against the oracle: each logit errs by at most cap * 2^-10 (hardware tanh, documented relative
    # error below 2^-10), and the log-sum-exp is 1-Lipschitz in the largest logit error, so a loss
    # errs by at most twice that
    ref = O.cross_entropy(O.softcap(rs[:, None] * acc, 15.0), t)
    np.testing.assert_allclose(got, ref, rtol=0, atol=2 * 15.0 * 2 ** -10)
    # against fp64 cross-entropy of this GPU's own soft-capped logits (same tanh values): only the
    # hardware exp2 (relative error near 2^-22) and fp32 sums differ
    own = O.cross_entropy(z_gpu.cpu().double().numpy(), t)
    np.testing.assert_allclose(got, own, rtol=0, atol=2e-4)
    assert got[4] == 0.0
    mean, bpb = O.loss_stats(own, t, tb.numpy())
    st = stats.cpu().double().numpy()
    np.testing.assert_allclose(st, [mean, bpb], rtol=1e-5)


def test_cross_entropy_target_out_of_range_sets_status():
    M, V, C = 64, 256, 128
    A, Wl = _rand_bf16((M, C), seed=31), _rand_bf16((V, C), scale=0.05, seed=32)
    tgt = torch.randint(0, V, (M,), generator=torch.Generator().manual_seed(33), dtype=torch.int32)
    tgt[5] = V + 3
    status = torch.zeros((1,), dtype=torch.int32, device=DEV)
    part, zt = _ops().lmhead_ce(A.to(DEV), Wl.to(DEV), tgt.to(DEV), cap=15.0, status=status)
    loss, stats = _ops().ce_finalize(part, zt, tgt.to(DEV), V, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6   # NC_ERR_TOKEN_RANGE
    assert float(loss[5]) == 0.0
    own = O.cross_entropy(_ops().gemm(A.to(DEV), Wl.to(DEV), "softcap_f32", cap=15.0).cpu().double().numpy(),
                          np.where(tgt.numpy() >= V, -1, tgt.numpy()))
    np.testing.assert_allclose(float(stats[0]), own[np.arange(M) != 5].mean(), rtol=1e-5)


# ------------------------------------------------------------------------ embedding

@pytest.mark.parametrize("embed_norm,a", [(False, 1.0), (True, 1.3)])
def test_embed_smear(embed_norm, a):
    from dataclasses import replace
    from synth import get_workload, make_weights
    cfg = replace(get_workload("tiny_all").model, embed_norm=embed_norm, smear_gate_channels=64)
    wts = make_weights(cfg)
    B_, T = 3, 50
    tok = torch.randint(0, cfg.vocab_size, (B_, T), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    x0, x, xb, ssp = _ops().embed_smear(tok.to(DEV), wts["wte"].to(DEV), wts["smear"].to(DEV), 64, embed_norm,
                                        cfg.rms_eps, a)
    torch.cuda.synchronize()
    W = O.OracleWeights.from_synth(cfg, wts)
    ref = np.concatenate([O.embed_smear(cfg, W, tok[b].numpy()) for b in range(B_)])
    np.testing.assert_allclose(x0.cpu().double().numpy(), ref, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(x.cpu().double().numpy(), a * ref, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(bf16_np(xb), a * ref, rtol=2 ** -8, atol=1e-6)
    np.testing.assert_allclose(ssp.cpu().double().numpy(), _ssp_of(a * ref), rtol=1e-5, atol=1e-7)


def test_embed_token_out_of_range_sets_status():
    V, C = 512, 128
    wte = _rand_bf16((V, C), 0.02, seed=1).to(DEV)
    tok = torch.tensor([[1, 2, V + 5, 3]], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    x0, x, xb, ssp = _ops().embed_smear(tok, wte, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6
    assert torch.all(x0[2] == 0) and torch.isfinite(x0).all()


# ------------------------------------------------------------------------ q|k|v epilogue

@pytest.mark.parametrize("H,Hkv,D,T,Brows,ve,cg", [(6, 6, 128, 200, 2, True, 384), (10, 5, 128, 130, 1, True, 1280),
                                                   (2, 1, 64, 64, 1, True, 64), (6, 6, 128, 97, 3, False, 0),
                                                   (12, 12, 128, 300, 1, True, 1536), (4, 2, 64, 150, 2, True, 200)])
def test_qkv_rope_qknorm_ve(H, Hkv, D, T, Brows, ve, cg):
    """q|k|v projection against the oracle's step functions.  On value-embedding layers the gate's
    pre-activation comes from the gate rows packed after each kv head's v rows (the GEMM reads the
    bf16 copy of the block input, like q, k and v; the reference uses the fp64 input, and the bf16
    rounding moves a gate by far less than the tolerance)."""
    C = H * D
    M = Brows * T
    V = 512
    g = torch.Generator().manual_seed(H * 100 + D)
    x = torch.randn((M, C), generator=g) * 3.0
    xb = x.to(torch.bfloat16)
    x64 = x.double().numpy()
    ssp = torch.from_numpy(_ssp_of(x64)).float()
    wq, wk, wv = (_rand_bf16((n, C), 0.02, seed=s) for n, s in ((H * D, 1), (Hkv * D, 2), (Hkv * D, 3)))
    B = binding()
    c_g = cg if ve else C
    wg = _rand_bf16((Hkv, c_g), 0.05, seed=5)
    wqkv = B.ops.pack_qkv(wq, wk, wv, wg if ve else None, D)
    tokens = torch.randint(0, V, (M,), generator=g, dtype=torch.int32)
    vet = _rand_bf16((V, Hkv * D), 0.02, seed=4)
    rope = B.ops.rope_table(T, D, 10000.0, DEV)
    q, k, v = B.ops.qkv(xb.to(DEV), wqkv.to(DEV), T, H, Hkv, D, rope, 1e-6, ssp.to(DEV),
                        ve, 1.5, vet.to(DEV) if ve else None, tokens.to(DEV), V)
    torch.cuda.synchronize()
    a = O.rms_norm(x64, 1e-6)
    cos, sin = O.rope_tables(T, D, 10000.0)
    for b in range(Brows):
        sl = slice(b * T, (b + 1) * T)
        qr = O.rms_norm(O.apply_rope((a[sl] @ bf16_np(wq).T).reshape(T, H, D), cos, sin), 1e-6)
        kr = O.rms_norm(O.apply_rope((a[sl] @ bf16_np(wk).T).reshape(T, Hkv, D), cos, sin), 1e-6)
        vr = (a[sl] @ bf16_np(wv).T).reshape(T, Hkv, D)
        if ve:
            gate = 1.5 * O.sigmoid(a[sl, :c_g] @ bf16_np(wg).T)
            vr = vr + gate[:, :, None] * bf16_np(vet)[tokens[sl].numpy()].reshape(T, Hkv, D)
        np.testing.assert_allclose(bf16_np(q[sl]).reshape(T, H, D), qr, rtol=1e-2, atol=2e-2)
        np.testing.assert_allclose(bf16_np(k[sl]).reshape(T, Hkv, D), kr, rtol=1e-2, atol=2e-2)
        # v carries the bf16 rounding of the GEMM input x (<= 2^-9 relative per element): over C
        # terms of x_c w_c (|x| ~ 3, |w| ~ 0.02) scaled by rs ~ 1/3 its spread is
        # sqrt(C) * 2^-9 * 3 * 0.02 / 3 ~ 1e-3, so 6e-3 covers the largest of ~1e5 outputs
        np.testing.assert_allclose(bf16_np(v[sl]).reshape(T, Hkv, D), vr, rtol=1e-2, atol=6e-3)


def test_rope_table_values():
    B = binding()
    t = B.ops.rope_table(2048, 128, 10000.0, DEV).cpu().double().numpy()   # [D/2, T, 2]
    cos, sin = O.rope_tables(2048, 128, 10000.0)                           # [T, D/2]
    np.testing.assert_allclose(t[..., 0].T, cos, atol=1e-6)
    np.testing.assert_allclose(t[..., 1].T, sin, atol=1e-6)


# ------------------------------------------------------------------------ attention

def _unit_rms(t):
    return t / t.pow(2).mean(-1, keepdim=True).sqrt()


@pytest.mark.parametrize("Bn,T,H,Hkv,D,window", [
    (1, 64, 2, 1, 64, -1), (2, 200, 6, 6, 128, -1), (2, 200, 6, 6, 128, 37), (1, 333, 10, 5, 128, 128),
    (1, 130, 2, 1, 64, 0), (1, 97, 4, 2, 128, 1), (2, 300, 6, 6, 128, 512), (1, 1030, 6, 6, 128, 256)])
def test_attention_windowed_gqa(Bn, T, H, Hkv, D, window):
    g = torch.Generator().manual_seed(T + H + window)
    q = _unit_rms(torch.randn((Bn * T, H, D), generator=g)).to(torch.bfloat16)
    k = _unit_rms(torch.randn((Bn * T, Hkv, D), generator=g)).to(torch.bfloat16)
    v = (torch.randn((Bn * T, Hkv, D), generator=g) * 0.5).to(torch.bfloat16)
    y = binding().ops.attention(q.reshape(Bn * T, -1).to(DEV), k.reshape(Bn * T, -1).to(DEV),
                                v.reshape(Bn * T, -1).to(DEV), Bn, T, H, Hkv, D, window)
    torch.cuda.synchronize()
    for b in range(Bn):
        sl = slice(b * T, (b + 1) * T)
        ref = O.attention(bf16_np(q[sl]), bf16_np(k[sl]), bf16_np(v[sl]), window)
        got = bf16_np(y[sl]).reshape(T, H, D)
        np.testing.assert_allclose(got, ref, rtol=2e-2, atol=1e-2)
