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


def test_gemm_resid_f32_in_place():
    M, N, K = 300, 768, 3072
    A = _rand_bf16((M, K), seed=5)
    Bm = _rand_bf16((N, K), scale=0.02, seed=6)
    x = torch.randn((M, N), generator=torch.Generator().manual_seed(7))
    xd = x.to(DEV)
    _ops().gemm(A.to(DEV), Bm.to(DEV), "resid_f32", out=xd, resid=xd)
    torch.cuda.synchronize()
    ref = x.double().numpy() + bf16_np(A) @ bf16_np(Bm).T
    np.testing.assert_allclose(xd.cpu().double().numpy(), ref, rtol=1e-5, atol=2e-4)


def test_gemm_relu2_and_softcap():
    M, N, K = 257, 1024, 768
    A = _rand_bf16((M, K), seed=8)
    Bm = _rand_bf16((N, K), scale=0.05, seed=9)
    acc = bf16_np(A) @ bf16_np(Bm).T
    h = _ops().gemm(A.to(DEV), Bm.to(DEV), "relu2_bf16")
    z = _ops().gemm(A.to(DEV), Bm.to(DEV), "softcap_f32", cap=15.0)
    torch.cuda.synchronize()
    np.testing.assert_allclose(bf16_np(h), O.relu2(acc), rtol=2 ** -7, atol=1e-3)
    # the soft-cap uses the hardware tanh (tanh.approx.f32, relative error below 2^-10 by its
    # documentation), so |cap * tanh| may err by up to cap * 2^-10 on top of the fp32 accumulation
    np.testing.assert_allclose(z.cpu().double().numpy(), O.softcap(acc, 15.0), rtol=0, atol=15.0 * 2 ** -10)
    assert float(z.abs().max()) < 15.0


# ------------------------------------------------------------------------ row kernels

@pytest.mark.parametrize("C,M", [(128, 67), (768, 1000), (1280, 33), (1536, 17)])
def test_rownorm_mix_and_gate(C, M):
    g = torch.Generator().manual_seed(C)
    x = torch.randn((M, C), generator=g) * 0.7
    y = torch.randn((M, C), generator=g) * 0.3
    Hkv, c_g = 3, C // 2
    wg = _rand_bf16((Hkv, c_g), scale=0.05, seed=C + 1)
    xo = torch.empty((M, C), device=DEV)
    xn, gate = _ops().rownorm(x.to(DEV), y.to(DEV), 1.1, 0.25, xo, 1e-6, wg.to(DEV), c_g, 2.0, True)
    torch.cuda.synchronize()
    xm = 1.1 * x.double().numpy() + 0.25 * y.double().numpy()
    np.testing.assert_allclose(xo.cpu().double().numpy(), xm, rtol=1e-6, atol=1e-6)
    a = O.rms_norm(xm, 1e-6)
    np.testing.assert_allclose(bf16_np(xn), a, rtol=2 ** -8, atol=1e-6)
    gref = 2.0 * O.sigmoid(a[:, :c_g] @ bf16_np(wg).T)
    np.testing.assert_allclose(gate.cpu().double().numpy(), gref, rtol=1e-5, atol=1e-5)


def test_rownorm_backout_form():
    M, C = 100, 768
    g = torch.Generator().manual_seed(11)
    x = torch.randn((M, C), generator=g)
    xm = torch.randn((M, C), generator=g)
    xn, _ = _ops().rownorm(x.to(DEV), xm.to(DEV), 1.0, -0.5)
    torch.cuda.synchronize()
    ref = O.rms_norm(x.double().numpy() - 0.5 * xm.double().numpy(), 1e-6)
    np.testing.assert_allclose(bf16_np(xn), ref, rtol=2 ** -8, atol=1e-6)


@pytest.mark.parametrize("embed_norm", [False, True])
def test_embed_smear(embed_norm):
    from dataclasses import replace
    from synth import get_workload, make_weights
    cfg = replace(get_workload("tiny_all").model, embed_norm=embed_norm, smear_gate_channels=64)
    wts = make_weights(cfg)
    B_, T = 3, 50
    tok = torch.randint(0, cfg.vocab_size, (B_, T), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    x0 = _ops().embed_smear(tok.to(DEV), wts["wte"].to(DEV), wts["smear"].to(DEV), 64, embed_norm, cfg.rms_eps)
    torch.cuda.synchronize()
    W = O.OracleWeights.from_synth(cfg, wts)
    for b in range(B_):
        ref = O.embed_smear(cfg, W, tok[b].numpy())
        np.testing.assert_allclose(x0[b * T:(b + 1) * T].cpu().double().numpy(), ref, rtol=1e-5, atol=1e-6)


def test_embed_token_out_of_range_sets_status():
    V, C = 512, 128
    wte = _rand_bf16((V, C), 0.02, seed=1).to(DEV)
    tok = torch.tensor([[1, 2, V + 5, 3]], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    x0 = _ops().embed_smear(tok, wte, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6
    assert torch.all(x0[2] == 0) and torch.isfinite(x0).all()


# ------------------------------------------------------------------------ q|k|v epilogue

@pytest.mark.parametrize("H,Hkv,D,T,Brows,ve", [(6, 6, 128, 200, 2, True), (10, 5, 128, 130, 1, True),
                                                (2, 1, 64, 64, 1, True), (6, 6, 128, 97, 3, False)])
def test_qkv_rope_qknorm_ve(H, Hkv, D, T, Brows, ve):
    C = H * D
    M = Brows * T
    V = 512
    g = torch.Generator().manual_seed(H * 100 + D)
    xn = (torch.randn((M, C), generator=g)).to(torch.bfloat16)
    wq, wk, wv = (_rand_bf16((n, C), 0.02, seed=s) for n, s in ((H * D, 1), (Hkv * D, 2), (Hkv * D, 3)))
    wqkv = torch.cat([wq, wk, wv], 0)
    tokens = torch.randint(0, V, (M,), generator=g, dtype=torch.int32)
    gate = torch.rand((M, Hkv), generator=g) if ve else None
    vet = _rand_bf16((V, Hkv * D), 0.02, seed=4) if ve else None
    B = binding()
    rope = B.ops.rope_table(T, D, 10000.0, DEV)
    q, k, v = B.ops.qkv(xn.to(DEV), wqkv.to(DEV), T, H, Hkv, D, rope, 1e-6,
                        gate.to(DEV) if ve else None, vet.to(DEV) if ve else None, tokens.to(DEV), V)
    torch.cuda.synchronize()
    a = bf16_np(xn)
    cos, sin = O.rope_tables(T, D, 10000.0)
    for b in range(Brows):
        sl = slice(b * T, (b + 1) * T)
        qr = O.rms_norm(O.apply_rope((a[sl] @ bf16_np(wq).T).reshape(T, H, D), cos, sin), 1e-6)
        kr = O.rms_norm(O.apply_rope((a[sl] @ bf16_np(wk).T).reshape(T, Hkv, D), cos, sin), 1e-6)
        vr = (a[sl] @ bf16_np(wv).T).reshape(T, Hkv, D)
        if ve:
            vr = vr + gate[sl].double().numpy()[:, :, None] * bf16_np(vet)[tokens[sl].numpy()].reshape(T, Hkv, D)
        np.testing.assert_allclose(bf16_np(q[sl]).reshape(T, H, D), qr, rtol=1e-2, atol=2e-2)
        np.testing.assert_allclose(bf16_np(k[sl]).reshape(T, Hkv, D), kr, rtol=1e-2, atol=2e-2)
        np.testing.assert_allclose(bf16_np(v[sl]).reshape(T, Hkv, D), vr, rtol=1e-2, atol=2e-3)


def test_rope_table_values():
    B = binding()
    t = B.ops.rope_table(2048, 128, 10000.0, DEV).cpu().double().numpy()
    cos, sin = O.rope_tables(2048, 128, 10000.0)
    np.testing.assert_allclose(t[..., 0], cos, atol=1e-6)
    np.testing.assert_allclose(t[..., 1], sin, atol=1e-6)


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
