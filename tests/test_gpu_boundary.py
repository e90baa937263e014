"""Boundary behaviour of the C ABI on a GPU: argument errors, device status word, host-buffer
entry point, per-kernel timing."""
import ctypes

import numpy as np
import pytest
import torch

from synth import get_workload, make_tokens, make_weights
from tests.helpers import binding, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tiny():
    wl = get_workload("tiny_all")
    wts = make_weights(wl.model, init="dense")
    B = binding()
    m = B.Model(wl.model, to_device(wts))
    return wl, m, make_tokens(wl)


def test_argument_errors(tiny):
    wl, m, tok = tiny
    B = binding()
    lib = B.lib()
    tok_d = tok.to(DEV)
    logits = torch.empty((wl.B, wl.T, wl.model.vocab_size), device=DEV)
    ws = m.workspace(wl.B, wl.T)
    s = torch.cuda.current_stream().cuda_stream
    assert lib.nc_forward(m.handle, tok_d.data_ptr(), wl.B, wl.T, logits.data_ptr(), ws.data_ptr(), ws.numel() - 1, s) == 3
    assert lib.nc_forward(m.handle, tok_d.data_ptr(), wl.B, wl.T, logits.data_ptr(), ws.data_ptr() + 16, ws.numel(), s) == 1
    assert lib.nc_forward(m.handle, tok_d.data_ptr(), 0, wl.T, logits.data_ptr(), ws.data_ptr(), ws.numel(), s) == 1
    n = ctypes.c_size_t()
    assert lib.nc_workspace_bytes(m.handle, 1, wl.model.seq_len_ctx + 1, ctypes.byref(n)) == 2
    big = torch.zeros((1, wl.model.seq_len_ctx + 1), dtype=torch.int32, device=DEV)
    with pytest.raises(B.NcError):
        m.forward(big)
    assert m.status() == 0


def test_token_out_of_range_reported_and_cleared(tiny):
    wl, m, tok = tiny
    bad = tok.clone()
    bad[0, 5] = wl.model.vocab_size + 3
    bad[1, 0] = -1
    out = m.forward(bad.to(DEV))
    assert m.status() == 6
    assert torch.isfinite(out).all()
    assert m.status() == 0


def test_forward_host_matches_device(tiny):
    wl, m, tok = tiny
    dev = m.forward(tok.to(DEV)).cpu()
    host_tok = tok.pin_memory()
    host_out = torch.empty((wl.B, wl.T, wl.model.vocab_size), dtype=torch.float32).pin_memory()
    m.forward_host(host_tok, host_out)
    assert torch.equal(dev, host_out)


def test_timing_counts_launches(tiny):
    wl, m, tok = tiny
    m.timing(True)
    m.forward(tok.to(DEV))
    m.forward(tok.to(DEV))
    m.timing(False)
    t = m.timing_read()
    L = wl.model.n_layer
    assert t["embed_smear"][1] == 2 and t["lmhead_softcap"][1] == 2
    assert t["qkv_rope_qknorm_ve"][1] == 2 * L and t["proj_residual"][1] == 2 * L
    assert m.launch_count() == 2 + 5 * L
    assert sum(n for _, n in t.values()) == 2 * m.launch_count()
    assert all(ms >= 0 for ms, _ in t.values())
