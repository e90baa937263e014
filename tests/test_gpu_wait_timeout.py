"""Failure detection without a GPU fault: a bounded device-side wait that runs out.

Every wait of the tcgen05 kernels on an mbarrier is bounded in time.  nc_op_test_wait_timeout runs
the GEMM kernel with a 1 ms limit and withholds, for one pair tile, the signal that its accumulator
is ready, so that the epilogue waiting for it gives up.  The kernel must record
NC_ERR_DEVICE_TIMEOUT, return (the stream synchronises), and leave the context usable: TMEM freed,
no copy or tensor-core operation left in flight.  The proof of the last part is that the same
GEMM, and a whole forward of a model, give bit-identical results before and after.
"""
import time

import pytest
import torch

from synth import get_workload, make_tokens, make_weights
from tests.helpers import binding, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"
NC_ERR_DEVICE_TIMEOUT = 5


def _rand_bf16(shape, seed):
    return (torch.randn(shape, generator=torch.Generator().manual_seed(seed)) * 0.5).to(torch.bfloat16).to(DEV)


def test_wait_runs_out_and_context_stays_usable():
    B = binding()
    wl = get_workload("tiny_all")
    model = B.Model(wl.model, to_device(make_weights(wl.model, init="dense")))
    tok = make_tokens(wl).to(DEV)
    before = model.forward(tok)
    assert model.status() == 0
    # two pair tiles (256 x 256 each), one per CTA pair: tile 0's accumulator signal is withheld
    M, N, K = 256, 512, 256
    A, Bm = _rand_bf16((M, K), 1), _rand_bf16((N, K), 2)
    ref = B.ops.gemm(A, Bm, "bf16")
    torch.cuda.synchronize()
    out = torch.zeros((M, N), dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.perf_counter()
    assert B.ops.test_wait_timeout(A, Bm, out, 1_000_000, 0, status) == 0
    torch.cuda.synchronize()   # the kernel returned
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == NC_ERR_DEVICE_TIMEOUT
    assert elapsed < 5.0
    # tile 1 (output columns 256..511) was computed normally
    assert torch.equal(out[:, 256:], ref[:, 256:])
    # the same GEMM and the model's forward, bit for bit as before the timeout
    assert torch.equal(B.ops.gemm(A, Bm, "bf16"), ref)
    after = model.forward(tok)
    assert model.status() == 0
    assert torch.equal(after, before)
