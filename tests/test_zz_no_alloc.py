"""nc_forward_static_scratch: the forward for callers that cannot allocate device memory.

Such callers (code inside a framework that owns all device memory, or a serving loop that
must not stall on cudaMalloc/cudaFree) get their scratch from a fixed array built into the
library.  This checks, through the C ABI, that two calls in a row give the same logits as
nc_forward with a caller workspace, and that sizes above the array's limit are refused
before any device work.  The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from synth import get_workload, make_tokens, make_weights
from tests.helpers import MAX_ABS, MEAN_REL, binding, parity, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT = 32 * 1024 * 1024


def _fn():
    lib = binding().lib()
    f = lib.nc_forward_static_scratch
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return f


@pytest.mark.parametrize("name,B,T", [("tiny_all", 2, 64), ("d12", 1, 512)])
def test_static_scratch_matches_workspace_forward(name, B, T):
    wl = get_workload(name)
    wts = make_weights(wl.model, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)[:B, :T].contiguous().to(DEV)
    m = binding().Model(wl.model, to_device(wts))
    assert m.workspace_bytes(B, T) <= LIMIT
    ref = m.forward(tok)
    assert m.status() == 0
    fn = _fn()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full((B, T, wl.model.vocab_size), float("nan"), device=DEV)
        assert fn(m.handle, tok.data_ptr(), B, T, out.data_ptr(), stream) == 0
        assert m.status() == 0
        max_abs, mean_rel = parity(out.cpu().numpy(), ref.cpu().numpy())
        assert np.isfinite(out.cpu().numpy()).all()
        assert max_abs <= MAX_ABS and mean_rel <= MEAN_REL


def test_static_scratch_rejects_sizes_above_limit():
    wl = get_workload("d12")
    wts = make_weights(wl.model, seed=wl.seed, init=wl.init)
    m = binding().Model(wl.model, to_device(wts))
    B, T = 8, 2048
    assert m.workspace_bytes(B, T) > LIMIT
    tok = torch.zeros((B, T), dtype=torch.int32, device=DEV)
    out = torch.zeros((1,), device=DEV)
    assert _fn()(m.handle, tok.data_ptr(), B, T, out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 3
    assert _fn()(None, tok.data_ptr(), B, T, out.data_ptr(), None) == 1
