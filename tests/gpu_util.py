"""Helpers shared by the GPU parity tests (not collected as tests)."""
import numpy as np

import ssd_inputs as si
from oracle import decode, model

NEAR_TIE = 0.05  # top-1 minus top-2 logit below which a token may differ
LOGIT_TOL = 3e-2
HIDDEN_COS = 0.999
# Draft exit: the stop decision compares the draft's top-1 probability p1 with a threshold.
# ln p1 = x_top - logsumexp(x); logits within LOGIT_TOL move each term by at most LOGIT_TOL,
# so a decision where |ln p1 - ln thr| < 2 * LOGIT_TOL may go either way.
NEAR_THR = 2 * LOGIT_TOL


def near_thr(p1, thr):
    return abs(np.log(p1) - np.log(thr)) < NEAR_THR


def cos(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def oracle_ar_with_gaps(W, prompt, n):
    """Oracle greedy tokens and the top-1/top-2 gap of the logits each was chosen from."""
    s = decode.Session(W)
    first, logits = s.prefill(prompt)
    toks, gaps = [first], [model.top_gap(logits[-1])]
    while len(toks) < n:
        nxt, row = s.ar_step()
        toks.append(nxt)
        gaps.append(model.top_gap(row))
    return toks, gaps


def first_mismatch(a, b):
    for i, (x, y) in enumerate(zip(a, b)):
        if x != y:
            return i
    return None


def gpu_ar_resync(eng, prompt, oracle_toks, gaps):
    """Run GPU greedy decoding step by step against the oracle; at a mismatch that is a
    near-tie in the oracle, count it and continue from the oracle's token.  Returns
    (near-tie count, hard mismatches)."""
    first = eng.prefill(prompt)
    t0 = len(prompt)
    near, hard = 0, []
    cur = first
    for i in range(len(oracle_toks)):
        if i > 0:
            cur = eng.decode_ar(1)[0]
        if cur != oracle_toks[i]:
            if gaps[i] < NEAR_TIE:
                near += 1
                eng.rollback(t0 + i, int(oracle_toks[i]))
                cur = oracle_toks[i]
            else:
                hard.append((i, cur, oracle_toks[i], gaps[i]))
                break
    return near, hard


def cfg_variant(name, **kw):
    return si.CONFIGS[name].replace(**kw) if kw else si.CONFIGS[name]
