"""fp64 CPU oracle for the nanochat-style decoder-only GPT forward pass (``forward``), its
next-token cross-entropy and bits per byte (``loss``), and the gradient of that loss with
respect to every weight (``backward``), and the forward with FP8 (e4m3) tensorwise-scaled
linear layers (``fp8``).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package; only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` use it.  It shares no code with the
CUDA path.
"""
from .forward import (
    OracleWeights, rms_norm, rope_tables, apply_rope, attention, relu2, softcap,
    sigmoid, embed_smear, block, forward_row, forward, param_shapes, param_count,
)
from .loss import cross_entropy, loss_stats

__all__ = [
    "OracleWeights", "rms_norm", "rope_tables", "apply_rope", "attention", "relu2",
    "softcap", "sigmoid", "embed_smear", "block", "forward_row", "forward",
    "param_shapes", "param_count", "cross_entropy", "loss_stats",
]
