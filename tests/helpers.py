"""Shared helpers for the GPU parity tests (the oracle is the reference everywhere)."""
import functools

import numpy as np
import torch

import oracle as O
from synth import get_workload, make_tokens, make_weights

# Tolerances for the full forward (bf16 tensor-core inputs, fp32 accumulation):
# max |logit - oracle| and sum|g - o| / sum|o|.
MAX_ABS = 5e-2
MEAN_REL = 1e-2


@functools.lru_cache(maxsize=None)
def ensure_built():
    from decoder_only_forward_02_b300 import build
    build.build()
    return True


def binding():
    ensure_built()
    from decoder_only_forward_02_b300 import binding as B
    return B


def to_device(wts: dict, device="cuda"):
    return {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in wts.items()}


def parity(g: np.ndarray, o: np.ndarray):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    d = np.abs(g - o)
    return float(d.max()), float(d.sum() / np.abs(o).sum())


# (label, max_abs, mean_rel) of every whole-forward comparison in this session, printed as a table
# at the end of the run (conftest.pytest_terminal_summary) so that the headroom to the bounds shows.
MARGINS = []


# (label, value, bound) of every backward comparison (relative errors of gradients, or the largest
# ratio of an error to its per-element bound), printed as a second table.
GRAD_MARGINS = []


def assert_parity(g, o, what=""):
    max_abs, mean_rel = parity(g, o)
    MARGINS.append((what, max_abs, mean_rel))
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    assert max_abs <= MAX_ABS and mean_rel <= MEAN_REL, f"{what}: max_abs={max_abs:.3e} mean_rel={mean_rel:.3e}"
    return max_abs, mean_rel


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


@functools.lru_cache(maxsize=4)
def workload_inputs(name: str, init: str = None):
    wl = get_workload(name)
    wts = make_weights(wl.model, seed=wl.seed, init=init or wl.init)
    tok = make_tokens(wl)
    return wl, wts, tok
