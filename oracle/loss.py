"""Plain fp64 NumPy statement of the next-token cross-entropy and bits per byte.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Sources (web pages, cited by title and section):

* [ARC] "nanochat — 架构与原理", section 2 component table (metrics row: bits
  per byte computed by the loss evaluation) and section 7 code map (the bpb
  metric beside the loss evaluation).
* [RPT] "NanoChat基础训练报告", loss progression table (training loss and
  validation bits per byte).

READING (the pages name the quantities but do not define them): the loss of a
position is the cross-entropy, in nats, of the soft-capped logits against the
token that follows it; a negative target marks an ignored position.  Bits per
byte sums the losses of the positions whose target token has a nonzero byte
length and divides by ln 2 times the sum of those byte lengths (tokens of zero
length, the special tokens, carry no bytes and are left out of both sums).

Pinned by the CPU tests in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

f64 = np.float64


def cross_entropy(logits: np.ndarray, targets: np.ndarray) -> np.ndarray:
    """Per-position loss [N] in nats: log(sum_v exp(z[n, v])) - z[n, targets[n]].

    logits [N, V] (any float type, evaluated in fp64); positions with a
    negative target get 0.  The log-sum-exp is taken around the row maximum,
    which leaves the value unchanged and keeps exp in range.
    """
    z = np.asarray(logits, dtype=f64)
    t = np.asarray(targets, dtype=np.int64)
    out = np.zeros(z.shape[0], dtype=f64)
    for n in range(z.shape[0]):
        if t[n] < 0:
            continue
        row = z[n]
        mx = row.max()
        out[n] = mx + math.log(np.exp(row - mx).sum()) - row[t[n]]
    return out


def loss_stats(losses: np.ndarray, targets: np.ndarray,
               token_bytes: Optional[np.ndarray] = None) -> Tuple[float, float]:
    """(mean loss over positions with a target >= 0, bits per byte).

    Bits per byte is NaN without token_bytes or when no counted target has a
    nonzero byte length; the mean is NaN when no position is counted.
    """
    l = np.asarray(losses, dtype=f64)
    t = np.asarray(targets, dtype=np.int64)
    counted = t >= 0
    mean = float(l[counted].sum() / counted.sum()) if counted.any() else float("nan")
    if token_bytes is None:
        return mean, float("nan")
    nb = np.where(counted, np.asarray(token_bytes, dtype=np.int64)[np.where(counted, t, 0)], 0)
    with_bytes = nb > 0
    if not with_bytes.any():
        return mean, float("nan")
    bpb = float(l[with_bytes].sum() / (math.log(2.0) * nb[with_bytes].sum()))
    return mean, bpb
