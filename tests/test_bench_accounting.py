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


def test_decode_step_bytes_d12():
    """d12, B = 8, position 2047: per layer 2304 x 768 q|k|v weights (+ 96 gate rows x 768 on the
    six value-embedding layers), 768 x 768 out-projection and two 3072 x 768 MLP matrices, the
    32768 x 768 lm_head, all bf16; the cache read is 512 keys on the nine window-512 layers and
    2047 on the three full ones, 8 rows x 6 heads x 128 x 2 bytes x (key, value) per key."""
    wl = get_workload("d12")
    cfg = wl.model
    assert sum(1 for v in cfg.has_ve if v) == 6
    per_layer = 2304 * 768 + 768 * 768 + 2 * 3072 * 768
    weights = 2 * (12 * per_layer + 6 * 96 * 768 + 32768 * 768)
    cache = (9 * 512 + 3 * 2047) * 8 * 6 * 128 * 2 * 2
    assert bench.decode_step_bytes(cfg, 8, 2047) == (weights, cache)
    assert weights == 221_085_696 and cache == 264_167_424
