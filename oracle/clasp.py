"""CLaSp dynamic-programming layer-skip search (oracle).

[CLaSp] §三 (the dynamic-programming paragraph): dp[i][j] is the largest
cosine similarity to the "optimal" hidden state reachable after the first i
transformer layers with j of them skipped.  §二 and §三: the target is the
full hidden state of the last accepted token from the last verify pass.
§三: the DP is approximate (the no-after-effect property does not hold),
yet close to brute force.  §三 (sequence parallelism): state (i, j) needs
only states (i-1, .), and all j of one i go through layer i together under
a mask without duplicating the KV cache.

Reading used here (the pages give no formula):
  * g_i = the full model's residual after layer i for the last accepted
    token tau at position p; g_0 = E[tau];
  * state(0, 0) = E[tau];  for i = 1..L and j in [max(0, n-(L-i)), min(i, n)]:
        keep = f_i(state(i-1, j))      if (i-1, j) is a state
        skip = state(i-1, j-1)         if (i-1, j-1) is a state
    state(i, j) = the candidate with the larger cos(., g_i); a tie keeps;
  * f_i is layer i run on one row at position p that sees the committed
    slots [0, p) and its own K/V (nothing is written to the cache);
  * the answer is the skip set backtracked from (L, n).
The oracle runs each j as its own one-row pass (the batching is a GPU
concern; it does not change what is computed).
"""
from __future__ import annotations

import itertools
from typing import Dict, List, Sequence, Tuple

import numpy as np

from .decode import Session
from .model import layer_forward


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.dot(a, b) / (np.linalg.norm(a) * np.linalg.norm(b)))


def _own_vis(p: int) -> np.ndarray:
    vis = np.zeros((1, p + 1), dtype=bool)
    vis[0, :] = True  # cache slots [0, p) + the row's own local K/V column
    return vis


def layer_on_state(sess: Session, i: int, h: np.ndarray, p: int) -> np.ndarray:
    cfg = sess.cfg
    out = layer_forward(cfg, sess.Wt.layer(i), sess.cache.k[i], sess.cache.v[i], h[None, :], np.array([p]), None,
                        _own_vis(p), False)
    return out[0]


def dp_search(sess: Session, n: int):
    """Return (skip set, dp value, table) for the current target.

    table[i][j] = (value, 'keep'|'skip', keep cosine or None, skip cosine or None):
    the state's cosine to g_i, the choice, and both candidates' cosines (the
    margin between them is how close the decision was)."""
    tgt = sess.target
    L, p = sess.cfg.n_layers, tgt.pos
    g = tgt.states
    states: Dict[int, np.ndarray] = {0: g[0].copy()}
    table: List[Dict[int, tuple]] = [{0: (cosine(g[0], g[0]), "keep", None, None)}]
    for i in range(1, L + 1):
        new: Dict[int, np.ndarray] = {}
        row: Dict[int, tuple] = {}
        for j in range(max(0, n - (L - i)), min(i, n) + 1):
            best = None
            c_keep = c_skip = None
            if j in states:
                keep = layer_on_state(sess, i - 1, states[j], p)
                c_keep = cosine(keep, g[i])
                best = (c_keep, "keep", keep)
            if j - 1 in states:
                c_skip = cosine(states[j - 1], g[i])
                if best is None or c_skip > best[0]:
                    best = (c_skip, "skip", states[j - 1])
            new[j] = best[2]
            row[j] = (best[0], best[1], c_keep, c_skip)
        states = new
        table.append(row)
    skip, j = [], n
    for i in range(L, 0, -1):
        if table[i][j][1] == "skip":
            skip.append(i - 1)
            j -= 1
    return tuple(sorted(skip)), table[L][n][0], table


def dp_select(sess: Session, n: int):
    skip, val, _ = dp_search(sess, n)
    return skip, val


def skipped_state(sess: Session, skip: Sequence[int]) -> np.ndarray:
    """Residual after all L layers of tau at p with the layers in `skip` bypassed."""
    tgt = sess.target
    h = tgt.states[0].copy()
    sk = set(skip)
    for i in range(sess.cfg.n_layers):
        if i not in sk:
            h = layer_on_state(sess, i, h, tgt.pos)
    return h


def brute_force(sess: Session, n: int):
    """max over all C(L, n) skip sets of cos(state_S, g_L); returns (best set, best value, all values)."""
    L = sess.cfg.n_layers
    g_L = sess.target.states[L]
    vals = {}
    for S in itertools.combinations(range(L), n):
        vals[S] = cosine(skipped_state(sess, S), g_L)
    best = max(vals, key=lambda s: vals[s])
    return best, vals[best], vals
