"""bench.py's work accounting, which sets the headline percentage: visible query-key pairs
against a brute-force count, and the model FLOPs per token against the window-aware counts
F_tok = L*2*(C*H*D + 2*C*Hkv*D + H*D*C + 2*C*F) + 2*C*V + sum over layers of 4*H*D*n_keys,
evaluated independently for the four full-size configurations."""
import math

import pytest

import bench
from synth import get_workload


@pytest.mark.parametrize("T,W", [(1, 0), (5, 0), (5, 2), (16, 3), (16, 15), (16, 16), (16, -1), (100, 7),
                                 (2048, 512)])
def test_window_pairs_brute_force(T, W):
    brute = sum((i + 1) if W < 0 else min(i + 1, W + 1) for i in range(T))
    assert bench.window_pairs(T, W) == brute


@pytest.mark.parametrize("name,per_token", [("d12", 242_053_248), ("d20", 865_482_880),
                                            ("d12_long", 307_523_712), ("d24", 1_547_026_944)])
def test_model_flops_per_token(name, per_token):
    wl = get_workload(name)
    assert math.isclose(bench.model_flops(wl.model, wl.B, wl.T), per_token * wl.B * wl.T, rel_tol=1e-12)


def test_d12_forward_is_3_966_tflop():
    wl = get_workload("d12")
    assert abs(bench.model_flops(wl.model, wl.B, wl.T) / 1e12 - 3.966) < 5e-4
