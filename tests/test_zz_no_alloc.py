"""nc_forward_static_scratch: the forward for callers that cannot allocate device memory.

Such callers (code inside a framework that owns all device memory, or a serving loop that
must not stall on cudaMalloc/cudaFree) get their scratch from a fixed array built into the
library.  This checks, through the C ABI, that two calls in a row give bit for bit the logits
of nc_forward with a caller workspace (the same kernels on the same inputs), with a call on
other tokens and a larger batch in between so that the second checked call starts from that
call's leftovers in the shared array, and that sizes above the array's limit are refused
before any device work.  The file name makes pytest collect it last.
"""
import ctypes

import torch
import pytest

from synth import get_workload, make_tokens, make_weights
from tests.helpers import binding, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT = 32 * 1024 * 1024


def _fn():
    lib = binding().lib()
    f = lib.nc_forward_static_scratch
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return f


def _static(m, tok, V):
    B, T = tok.shape
    out = torch.full((B, T, V), float("nan"), device=DEV)
    rc = _fn()(m.handle, tok.data_ptr(), B, T, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    assert m.status() == 0
    return out


# (workload, checked batch B x T, the larger batch of the call in between)
@pytest.mark.parametrize("name,B,T,B2,T2", [("tiny_all", 2, 64, 4, 64), ("d12", 1, 512, 2, 640)])
def test_static_scratch_matches_workspace_forward(name, B, T, B2, T2):
    wl = get_workload(name)
    V = wl.model.vocab_size
    wts = make_weights(wl.model, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)[:B, :T].contiguous().to(DEV)
    other = torch.randint(0, V, (B2, T2), generator=torch.Generator().manual_seed(77),
                          dtype=torch.int32).to(DEV)
    m = binding().Model(wl.model, to_device(wts))
    assert m.workspace_bytes(B2, T2) <= LIMIT and m.workspace_bytes(B2, T2) > m.workspace_bytes(B, T)
    ref = m.forward(tok)
    ref_other = m.forward(other)
    assert m.status() == 0
    assert torch.equal(_static(m, tok, V), ref)
    assert torch.equal(_static(m, other, V), ref_other)   # different tokens, larger batch
    assert torch.equal(_static(m, tok, V), ref)           # starts from the larger call's leftovers


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
