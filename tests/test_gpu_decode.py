"""KV-cache prefill + single-token decode (C ABI, CUDA kernels) against the fp64 oracle.

The forward is causal, so the logits a decode step produces at position p must equal row p of
the oracle's forward over the whole sequence; prefill logits must equal rows 0..T0-1.  The
tiny case covers GQA (H = 2, Hkv = 1), D = 64 and windows shorter than the prefill (the
layer's cache ring wraps); d12 covers D = 128 and the window-512 ring at full size."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from synth import get_workload, make_tokens, make_weights
from tests.helpers import assert_parity, binding, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _decode_run(m, tok, T0, T_max, positions):
    cache = m.kv_cache(tok.shape[0], T_max)
    pre = m.prefill(tok[:, :T0].contiguous().to(DEV), cache, T_max)
    steps = []
    for p in positions:
        steps.append(m.decode_step(tok[:, p - 1].contiguous().to(DEV), tok[:, p].contiguous().to(DEV), p, cache,
                                   T_max).clone())
    assert m.status() == 0
    return pre, torch.stack(steps, 1)


def test_decode_tiny_gqa_windows_wrap():
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, n_layer=3, window_left=(16, 16, -1), has_ve=(1, 0, 1), seq_len_ctx=64)
    wts = make_weights(cfg, init="dense")
    tok = torch.randint(0, cfg.vocab_size, (2, 64), generator=torch.Generator().manual_seed(21), dtype=torch.int32)
    m = binding().Model(cfg, to_device(wts))
    T0 = 20
    pos = list(range(T0, 64))
    pre, dec = _decode_run(m, tok, T0, 64, pos)
    ref = O.forward(cfg, O.OracleWeights.from_synth(cfg, wts), tok.numpy())
    assert_parity(pre.cpu().numpy(), ref[:, :T0], "prefill")
    assert_parity(dec.cpu().numpy(), ref[:, T0:], "decode")
    full = m.forward(tok.to(DEV)).cpu().numpy()
    np.testing.assert_allclose(dec.cpu().numpy(), full[:, T0:], rtol=0, atol=2e-2)
    np.testing.assert_array_equal(pre.cpu().numpy(), full[:, :T0])   # prefill is the forward itself


def test_decode_d12_tail_positions():
    wl = get_workload("d12")
    cfg = wl.model
    wts = make_weights(cfg, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)
    m = binding().Model(cfg, to_device(wts))
    T0 = wl.T - 8
    pos = list(range(T0, wl.T))
    _, dec = _decode_run(m, tok, T0, wl.T, pos)
    full = m.forward(tok.to(DEV))
    got = dec.cpu().numpy()
    assert_parity(got, full[:, T0:].cpu().numpy(), "decode vs forward")
    ref = O.forward_row(cfg, O.OracleWeights.from_synth(cfg, wts), tok[0].numpy(), positions=pos)
    assert_parity(got[0], ref, "decode vs oracle row 0")


def test_decode_argument_errors():
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, seq_len_ctx=64)
    m = binding().Model(cfg, to_device(make_weights(cfg, init="dense")))
    tok = torch.zeros((1,), dtype=torch.int32, device=DEV)
    cache = m.kv_cache(1, 32)
    lib = binding().lib()
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    out = torch.empty((1, cfg.vocab_size), device=DEV)
    args = lambda pos, cap_bytes, T_max: (m.handle, tok.data_ptr(), tok.data_ptr(), 1, pos, cache.data_ptr(),
                                          cap_bytes, T_max, out.data_ptr(), ws.data_ptr(), ws.numel(), None)
    assert lib.nc_decode_step(*args(0, cache.numel(), 32)) == 1          # pos must be >= 1
    assert lib.nc_decode_step(*args(32, cache.numel(), 32)) == 1         # pos < T_max
    assert lib.nc_decode_step(*args(5, cache.numel(), 65)) == 2          # T_max > seq_len_ctx
    assert lib.nc_decode_step(*args(5, cache.numel() - 1, 32)) == 3      # cache too small
    assert m.launch_count(kv=True) == 2 + 5 * cfg.n_layer


def test_decode_step_replays_from_a_cuda_graph():
    """After a first call on the device (per-device kernel set-up), a decode step makes no host
    synchronisation or allocation, so a caller can capture it in a CUDA graph: replays give the
    eager step's logits bit for bit (the cache append at the position rewrites the same rows)."""
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, n_layer=3, window_left=(16, 16, -1), has_ve=(1, 0, 1), seq_len_ctx=64)
    wts = make_weights(cfg, init="dense")
    tok = torch.randint(0, cfg.vocab_size, (2, 64), generator=torch.Generator().manual_seed(22), dtype=torch.int32)
    m = binding().Model(cfg, to_device(wts))
    T0, p = 40, 40
    cache = m.kv_cache(2, 64)
    m.prefill(tok[:, :T0].contiguous().to(DEV), cache, 64)
    prev, cur = tok[:, p - 1].contiguous().to(DEV), tok[:, p].contiguous().to(DEV)
    out = torch.empty((2, cfg.vocab_size), dtype=torch.float32, device=DEV)
    m.decode_step(prev, cur, p, cache, 64, out=out)
    eager = out.clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            m.decode_step(prev, cur, p, cache, 64, out=out)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert m.status() == 0


def test_decode_twelve_rows():
    """B = 12 (one group of 16 token rows, 12 of them filled; a window that wraps on the first
    layer): the steps equal the forward's rows and the oracle's."""
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, n_layer=2, window_left=(8, -1), has_ve=(0, 1), seq_len_ctx=64)
    wts = make_weights(cfg, init="dense")
    tok = torch.randint(0, cfg.vocab_size, (12, 40), generator=torch.Generator().manual_seed(23), dtype=torch.int32)
    m = binding().Model(cfg, to_device(wts))
    T0 = 30
    pos = list(range(T0, 40))
    _, dec = _decode_run(m, tok, T0, 64, pos)
    ref = O.forward(cfg, O.OracleWeights.from_synth(cfg, wts), tok.numpy())
    assert_parity(dec.cpu().numpy(), ref[:, T0:], "decode, 12 batch rows")
    full = m.forward(tok.to(DEV)).cpu().numpy()
    np.testing.assert_allclose(dec.cpu().numpy(), full[:, T0:], rtol=0, atol=2e-2)


def test_decode_twenty_rows():
    """B = 20: the step's products take the tokens in groups of 16, so the second group (4 rows)
    exercises a partly filled group; the steps equal the oracle's rows and the forward's."""
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, n_layer=2, window_left=(8, -1), has_ve=(1, 0), seq_len_ctx=64)
    wts = make_weights(cfg, init="dense")
    tok = torch.randint(0, cfg.vocab_size, (20, 36), generator=torch.Generator().manual_seed(24), dtype=torch.int32)
    m = binding().Model(cfg, to_device(wts))
    T0 = 32
    pos = list(range(T0, 36))
    _, dec = _decode_run(m, tok, T0, 64, pos)
    ref = O.forward(cfg, O.OracleWeights.from_synth(cfg, wts), tok.numpy())
    assert_parity(dec.cpu().numpy(), ref[:, T0:], "decode, 20 batch rows")
    full = m.forward(tok.to(DEV)).cpu().numpy()
    np.testing.assert_allclose(dec.cpu().numpy(), full[:, T0:], rtol=0, atol=2e-2)


def test_decode_from_the_first_positions():
    """A prefill of one token, then decode steps at positions 1..12: with fewer cached keys than
    the attention's eight splits, most splits are empty and the new key's partial dominates; a
    window of 4 makes the ring wrap from position 5 on."""
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, n_layer=2, window_left=(4, -1), has_ve=(1, 0), seq_len_ctx=64)
    wts = make_weights(cfg, init="dense")
    tok = torch.randint(0, cfg.vocab_size, (3, 13), generator=torch.Generator().manual_seed(25), dtype=torch.int32)
    m = binding().Model(cfg, to_device(wts))
    pre, dec = _decode_run(m, tok, 1, 64, list(range(1, 13)))
    ref = O.forward(cfg, O.OracleWeights.from_synth(cfg, wts), tok.numpy())
    assert_parity(pre.cpu().numpy(), ref[:, :1], "prefill of one token")
    assert_parity(dec.cpu().numpy(), ref[:, 1:13], "decode, positions 1..12")


def test_decode_d12_twenty_rows_persistent_lm_head():
    """d12 weights with B = 20 (two groups of 16 token rows): the lm_head's product runs on
    persistent CTAs over 4,096 vocabulary blocks for each group; steps at positions 14 and 15 equal
    the forward's rows and the oracle's."""
    wl = get_workload("d12")
    cfg = wl.model
    wts = make_weights(cfg, seed=wl.seed, init=wl.init)
    tok = torch.randint(0, cfg.vocab_size, (20, 16), generator=torch.Generator().manual_seed(26), dtype=torch.int32)
    m = binding().Model(cfg, to_device(wts))
    _, dec = _decode_run(m, tok, 14, 64, [14, 15])
    full = m.forward(tok.to(DEV)).cpu().numpy()
    assert_parity(dec.cpu().numpy(), full[:, 14:16], "decode vs forward, d12, 20 rows")
    ref = O.forward_row(cfg, O.OracleWeights.from_synth(cfg, wts), tok[19].numpy(), positions=[14, 15])
    assert_parity(dec[19].cpu().numpy(), ref, "decode vs oracle, d12, row 19")


@pytest.mark.parametrize("windows", [(0, -1), (1, 2)])
def test_decode_windows_of_zero_to_two_keys(windows):
    """Windows W = 0, 1, 2: a query sees only itself (no cached key: every split is empty and the
    new key's partial is the whole softmax) or one or two cached keys; the ring has W + 1 slots."""
    wl = get_workload("tiny_all")
    cfg = replace(wl.model, n_layer=2, window_left=windows, has_ve=(1, 1), seq_len_ctx=64)
    wts = make_weights(cfg, init="dense")
    tok = torch.randint(0, cfg.vocab_size, (2, 12), generator=torch.Generator().manual_seed(27), dtype=torch.int32)
    m = binding().Model(cfg, to_device(wts))
    _, dec = _decode_run(m, tok, 3, 64, list(range(3, 12)))
    ref = O.forward(cfg, O.OracleWeights.from_synth(cfg, wts), tok.numpy())
    assert_parity(dec.cpu().numpy(), ref[:, 3:12], f"decode, windows {windows}")
