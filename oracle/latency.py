"""Latency model and cascade-depth rules of the DyTC scheduler (oracle).

Test infrastructure: only tests/, the smoke check and bench.py's CPU legs use
this package.

[CAS-blog] §3.2: every draft configuration's latency is predicted as
latency = b0 + b1 * seq_len + b2 * layer_depth, with the b fitted offline.
Reading: layer_depth = layers the pass runs, seq_len = the committed context;
the fit is ordinary least squares over measured points.

[CAS-blog] §4.1 item 1: maximum cascade depth K = min(3, log2(layers / 12)),
read as a count of levels, so its floor; §4.2 problem 3: one level fewer when
seq_len > 512.  At least one level always remains, and the levels kept are
the first K (cheapest first).
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np


def fit_latency(seq_len: Sequence[float], depth: Sequence[float], ms: Sequence[float]) -> np.ndarray:
    """(b0, b1, b2) minimising sum (b0 + b1 s + b2 d - ms)^2, by numpy's least squares."""
    A = np.stack([np.ones(len(ms)), np.asarray(seq_len, dtype=np.float64), np.asarray(depth, dtype=np.float64)], 1)
    beta, _, rank, _ = np.linalg.lstsq(A, np.asarray(ms, dtype=np.float64), rcond=None)
    if rank < 3:
        raise ValueError("the points do not determine the three coefficients")
    return beta


def predict(beta: Sequence[float], seq_len: float, depth: float) -> float:
    return float(beta[0] + beta[1] * seq_len + beta[2] * depth)


def cascade_depth(n_layers: int, n_levels: int, seq_len: int) -> int:
    k = math.floor(min(3.0, math.log2(n_layers / 12.0)))
    if seq_len > 512:
        k -= 1
    return max(1, min(k, n_levels))
