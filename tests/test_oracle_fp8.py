"""Pins of the FP8 (e4m3, tensorwise-scaled) forward oracle (oracle/fp8.py), on CPU."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import fp8 as F8
from synth import get_workload, make_tokens, make_weights

rng = np.random.default_rng(77)


def test_round_e4m3_matches_torch_float8():
    mags = 2.0 ** rng.uniform(-12, np.log2(448.0), 20000)
    x = np.concatenate([mags * rng.choice([-1.0, 1.0], mags.size),
                        [0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -6, 240.0, 232.0, 17.0]])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(F8.round_e4m3(x), ref)
    assert F8.round_e4m3(np.array([1000.0, -460.0]))[0] == 448.0     # saturates
    assert F8.round_e4m3(np.array([-460.0]))[0] == -448.0


def test_fp8_linear_exact_on_the_grid_at_unit_scale():
    grid = np.unique(np.abs(F8.round_e4m3(rng.uniform(-448, 448, 4000))))
    x = rng.choice(grid, (9, 16)) * rng.choice([-1.0, 1.0], (9, 16))
    w = rng.choice(grid, (5, 16)) * rng.choice([-1.0, 1.0], (5, 16))
    x[0, 0], w[0, 0] = 448.0, -448.0                       # amax 448: both scales are 1
    np.testing.assert_array_equal(F8.fp8_linear(x, w), x @ w.T)


def test_fp8_linear_scaling_commutes_with_powers_of_two():
    x, w = rng.normal(size=(7, 32)), rng.normal(size=(11, 32))
    base = F8.fp8_linear(x, w)
    np.testing.assert_array_equal(F8.fp8_linear(8.0 * x, w), 8.0 * base)
    np.testing.assert_array_equal(F8.fp8_linear(x, 0.25 * w), 0.25 * base)


def test_fp8_linear_error_bound():
    # each quantised operand errs by at most 2^-4 relative (3 mantissa bits, half a spacing) or by
    # half the subnormal spacing 2^-10 / scale in absolute terms
    x, w = rng.normal(size=(64, 96)), rng.normal(size=(48, 96))
    sx, sw = F8.tensor_scale(x), F8.tensor_scale(w)
    ex = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 / sx
    ew = 2.0 ** -4 * np.abs(w) + 2.0 ** -10 / sw
    bound = (ex @ np.abs(w).T) + (np.abs(x) @ ew.T) + (ex @ ew.T)
    err = np.abs(F8.fp8_linear(x, w) - x @ w.T)
    assert np.all(err <= bound * (1 + 1e-12))
    assert np.linalg.norm(err) / np.linalg.norm(x @ w.T) < 0.05


@pytest.mark.parametrize("name", ["tiny_all", "tiny"])
def test_batched_forward_equals_the_forward_oracle(name):
    wl = get_workload(name)
    cfg = wl.model
    W = O.OracleWeights.from_synth(cfg, make_weights(cfg, init="dense"))
    tok = make_tokens(wl).numpy()
    np.testing.assert_allclose(F8.forward_batched(cfg, W, tok), O.forward(cfg, W, tok), rtol=1e-12, atol=1e-12)


def test_fp8_forward_stays_close_to_bf16_forward():
    # not a pin: the e4m3 forward of the tiny model tracks the exact one (|logit| < 15)
    wl = get_workload("tiny_all")
    cfg = wl.model
    W = O.OracleWeights.from_synth(cfg, make_weights(cfg, init="dense"))
    tok = make_tokens(wl).numpy()
    z8, z = F8.forward_fp8(cfg, W, tok), O.forward(cfg, W, tok)
    assert np.all(np.abs(z8) < cfg.softcap)
    assert np.abs(z8 - z).max() < 0.5 and np.abs(z8 - z).mean() < 0.05
