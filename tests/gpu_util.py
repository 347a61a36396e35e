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


# ---------------------------------------------------------------------------------------------------
# The oracle follows a GPU generation (ssd_generate's per-cycle log, OPT_CYCLE_LOG): every decision the
# GPU took -- each draft token, each verify row's argmax, each tree expansion's top-2, each DP mask --
# is recomputed by the oracle on the GPU's own inputs and compared.  Where they differ, the oracle's
# gap at that decision must be a near-tie (counted); the oracle then continues with the GPU's decision,
# so every later cycle is still compared on identical inputs.


class Follow:
    def __init__(self, W, prompt, gpu_first, int8_tokens=True):
        self.int8_tokens = int8_tokens
        self.W = W
        self.cfg = W.cfg
        self.s = decode.Session(W)
        self.near = 0  # near-tie decisions where the GPU and the oracle differ
        self.decisions = 0
        first, logits = self.s.prefill(prompt)
        self.tie(first == gpu_first, model.top_gap(logits[-1]), "first token")
        self.s.pending = int(gpu_first)

    def tie(self, same: bool, gap: float, what):
        self.decisions += 1
        if not same:
            assert gap < NEAR_TIE, (what, gap)
            self.near += 1

    def check_verify_rows(self, e, cyc, n_rows):
        for r in range(n_rows):
            self.tie(e["argmax"][r] == cyc.argmax[r], cyc.gaps[r], ("verify row", e["t"], r))

    def linear(self, e, skip, act_int8=False, exit_layers=0, exit_thr=0.0, k=None):
        s = self.s
        assert (e["t"], e["tokens"][0]) == (s.t, s.pending), (e["t"], s.t, e["tokens"][0], s.pending)
        drafts = [x for x in e["tokens"][1:] if x >= 0]
        gaps, am, probs = [], [], []
        s.draft_linear(skip, len(drafts), act_int8, gaps=gaps, force=drafts, argmax=am, probs=probs,
                       exit_layers=exit_layers)
        for r in range(len(drafts)):
            self.tie(am[r] == drafts[r], gaps[r], ("draft", e["t"], r))
        if exit_thr > 0:
            for r, p1 in enumerate(probs):
                stop_here = r == len(drafts) - 1 and len(drafts) < k
                if (p1 < exit_thr) != stop_here:
                    assert near_thr(p1, exit_thr), ("draft exit", e["t"], r, p1, exit_thr)
                    self.near += 1
        cyc = s.verify_linear(drafts, follow=(e["n_acc"], e["bonus"]))
        self.check_verify_rows(e, cyc, len(drafts) + 1)
        if e["argmax"][: len(drafts) + 1] == cyc.argmax:
            assert (e["n_acc"], e["bonus"]) == (cyc.n_accepted, cyc.bonus)
        return drafts, cyc

    def tree(self, e, parents, expansions, levels, level_exit=()):
        """expansions: (node, level) in the order they ran; levels: (skip, int8) per level.  With
        self.int8_tokens False the children of int8-level expansions are not compared (a deep int8
        forward's decisions depend on code flips; see int8_logits_check)."""
        s = self.s
        assert (e["t"], e["tokens"][0]) == (s.t, s.pending)
        assert e["parents"] == list(parents), (e["parents"], parents)
        tokens = e["tokens"]
        depth = decode.tree_depths(parents)
        kids = {}
        for c in range(1, len(parents)):
            kids.setdefault(parents[c], []).append(c)
        for u, l in expansions:
            skip, int8 = levels[l]
            rows = []
            top = s.draft_node(u, parents, depth, tokens[u], skip, int8, level_exit[l] if level_exit else 0,
                               rows=rows)
            if int8 and not self.int8_tokens:
                continue
            x = np.sort(np.asarray(rows[0], dtype=np.float64))[::-1]
            g01, g12 = float(x[0] - x[1]), float(x[1] - x[2])
            for r, c in enumerate(kids.get(u, [])):
                self.tie(tokens[c] == top[r], g01 if r == 0 else min(g01, g12), ("expansion", e["t"], u, r))
        cyc = s.verify_tree(tokens, parents, follow=(e["path"], e["bonus"]))
        self.check_verify_rows(e, cyc, len(parents))
        if e["argmax"] == cyc.argmax:
            assert (e["path"], e["bonus"]) == (cyc.path, cyc.bonus)
        return cyc

    def dytc(self, e, dy: decode.DyTC):
        plan = dy.plan(self.s.t)
        self.tree(e, plan.parents, plan.expansions, self.cfg.levels, self.cfg.level_exit)
        tokens = e["tokens"]
        gpu = decode.Cycle(tokens[1:], e["argmax"], [], e["n_acc"], e["bonus"], e["path"])
        dy.update(plan, tokens, gpu)  # the oracle's EMA arithmetic on the GPU's acceptance
        assert e["ema"][: len(dy.a)] == dy.a, (e["ema"], dy.a)  # same float64 operations: identical

    def vcascade(self, e, lo, hi, k):
        """Vertical cascade cycle: the lower level's drafts, the higher level's check and the chain it hands
        the target, all on the GPU's chain."""
        s, cfg = self.s, self.cfg
        assert (e["t"], e["tokens"][0]) == (s.t, s.pending)
        chain = [x for x in e["tokens"][1:] if x >= 0]
        (sk_lo, i8_lo), (sk_hi, i8_hi) = cfg.levels[lo], cfg.levels[hi]
        t = s.t
        lg, lam = [], []
        m = len(chain) - 1  # the chain's last entry: a lower-level draft the higher level agreed with, or its correction
        d = s.draft_linear(sk_lo, k, i8_lo, gaps=lg, argmax=lam, force=chain[:m],
                           exit_layers=decode.level_exit(cfg, lo))
        for r in range(m):
            self.tie(lam[r] == chain[r], lg[r], ("lower draft", t, r))
        rows = [s.pending] + d
        logits, _ = decode.forward(self.W, s.cache, rows, range(t, t + k + 1), range(t, t + k + 1),
                                   decode.causal_vis(t, k + 1), skip=sk_hi, act_int8=i8_hi,
                                   exit_layers=decode.level_exit(cfg, hi))
        ham = [int(a) for a in decode.argmax_f32(logits)]
        hg = [decode.top_gap(r) for r in logits]
        for r in range(m + 1):
            self.tie(ham[r] == chain[r], hg[r], ("higher check", t, r))
        if m + 1 < k:  # the chain stopped early: the higher level rejected the lower draft at m
            self.tie(ham[m] != d[m], min(hg[m], lg[m]), ("higher rejects", t, m))
        cyc = s.verify_linear(chain, follow=(e["n_acc"], e["bonus"]))
        self.check_verify_rows(e, cyc, len(chain) + 1)
        return cyc

    def dp(self, e, n):
        from oracle import clasp

        s = self.s
        o_mask, o_val, _ = clasp.dp_search(s, n)
        self.decisions += 1
        if tuple(e["mask"]) != tuple(o_mask):
            got = clasp.cosine(clasp.skipped_state(s, e["mask"]), s.target.states[self.cfg.n_layers])
            assert got >= o_val - 1e-3, (e["mask"], o_mask, got, o_val)
            self.near += 1
        assert abs(e["dp_value"] - o_val) < 2e-3, (e["dp_value"], o_val)
        return tuple(e["mask"])


def tree_cycle_against_oracle(eng, s, toks, parents, expansions, levels, level_exit=(), int8_tokens=True):
    """One teacher-forced tree cycle: every expansion of the GPU's tree recomputed by the oracle on the
    GPU's tokens (top-2 compared, near-ties counted), then both verify the GPU's tree: every node's
    logits within tolerance, and the oracle follows the GPU's acceptance.  Returns the near-tie count."""
    near = 0
    depth = decode.tree_depths(parents)
    kids = {}
    for c in range(1, len(parents)):
        kids.setdefault(parents[c], []).append(c)
    for u, l in expansions:
        skip, int8 = levels[l]
        rows = []
        top = s.draft_node(u, parents, depth, toks[u], skip, int8, level_exit[l] if level_exit else 0, rows=rows)
        if int8 and not int8_tokens:  # a deep int8 forward's decisions are not compared
            continue
        x = np.sort(np.asarray(rows[0], dtype=np.float64))[::-1]
        for r, c in enumerate(kids.get(u, [])):
            if toks[c] != top[r]:
                assert (x[0] - x[1] if r == 0 else min(x[0] - x[1], x[1] - x[2])) < NEAR_TIE, (u, r, toks, top)
                near += 1
    n_acc, path, bonus = eng.verify(toks, parents)
    lo = []
    cyc = s.verify_tree(toks, parents, follow=(path, bonus), logits_out=lo)
    for c in range(len(parents)):
        err = float(np.max(np.abs(eng.logits(c) - lo[0][c])))
        assert err < LOGIT_TOL, (c, err)
    if (path, bonus) != (cyc.path, cyc.bonus):
        am = [int(np.argmax(eng.logits(c))) for c in range(len(parents))]
        bad = [c for c in range(len(parents)) if am[c] != cyc.argmax[c]]
        assert bad and all(cyc.gaps[c] < NEAR_TIE for c in bad), (path, bonus, cyc)
        near += 1
    return near


def oracle_cands(table, L, n):
    """The oracle's DP table (clasp.dp_search) as an [L+1, n+1, 2] array of (keep, skip) cosines (NaN absent)."""
    c = np.full((L + 1, n + 1, 2), np.nan)
    for i in range(L + 1):
        for j, e in table[i].items():
            if e[2] is not None:
                c[i, j, 0] = e[2]
            if e[3] is not None:
                c[i, j, 1] = e[3]
    return c


def compare_dp_tables(val, back, cands, L, n, tol=2e-3):
    """Compare the GPU's DP table with the oracle's candidate cosines, layer by layer from the bottom: every
    cell's decision (keep / skip, a tie keeps) and value must match until the first layer where a decision
    differs; there each differing cell must be a near-tie (|keep - skip| < tol).  The layers above depend on
    the differing cells' states and are not compared.  Returns (layer of the first difference or None,
    number of differing cells there)."""
    assert abs(float(val[0, 0]) - 1.0) < 1e-6
    for i in range(1, L + 1):
        lo, hi = max(0, n - (L - i)), min(i, n)
        flips = []
        for j in range(lo, hi + 1):
            kc, sc = cands[i, j]
            o_skip = np.isnan(kc) or (not np.isnan(sc) and sc > kc)
            o_val = sc if o_skip else kc
            if bool(back[i, j]) != o_skip:
                assert not np.isnan(kc) and not np.isnan(sc) and abs(kc - sc) < tol, (i, j, kc, sc, back[i, j])
                flips.append(j)
            else:
                assert abs(float(val[i, j]) - o_val) < tol, (i, j, float(val[i, j]), o_val)
        if flips:
            return i, len(flips)
    return None, 0


def int8_prefix_free(eng, W, token, skip, k, shallow):
    """An int8 draft with no committed prefix (the pending token at position 0): each draft row's attention
    sees only the drafts' own keys, so both sides quantize values that differ only by float32 rounding of
    their products (with a prefix, the prefilled cache's 16-bit hi/lo operand rounding, ~1e-5 relative,
    already flips many codes).  Leaves the engine at committed length 0."""
    eng.rollback(0, int(token))
    d = eng.draft(skip, k, act_int8=True)
    g = eng.logits(0)
    s = decode.Session(W, 64)
    s.pending = int(token)
    r8, r16, am, gaps = [], [], [], []
    s.draft_linear(skip, k, act_int8=True, rows=r8, force=d, argmax=am, gaps=gaps)
    s.draft_linear(skip, k, act_int8=False, rows=r16, force=d)
    dev, q = int8_logits_check(g, r8[-1], r16[-1], shallow)
    near = 0
    if shallow:
        for r in range(k):
            if am[r] != d[r]:
                assert gaps[r] < NEAR_TIE, (r, d, am, gaps)
                near += 1
    return near, dev, q


def int8_logits_check(gpu_row, o_int8, o_16, shallow: bool):
    """GPU logits of an int8-activation forward against the oracle's.  Per-token int8 codes make the forward
    discontinuous: a code flips when an element sits within rounding noise of a .5 boundary, and the flip
    moves the next layer's inputs by a quantization step, which flips more codes downstream (the oracle
    against itself with float32 instead of float64 products: 0 to 0.03 after one or two layers, up to 0.33
    and cos 0.998 after four).  The yardstick is the quantization's own effect on this forward,
    q = oracle int8 logits - oracle 16-bit logits.  A shallow forward (one layer run) has few flips: its
    logits must agree within max(LOGIT_TOL, q/4) in max-abs, which a missing or wrong quantization misses
    by about 4x.  A deep forward's flips have spread: its deviation must stay within twice q (RMS), which
    bounds gross errors only; its decisions are not compared."""
    g, a, b = (np.asarray(x, dtype=np.float64) for x in (gpu_row, o_int8, o_16))
    q = float(np.max(np.abs(a - b)))
    dev = float(np.max(np.abs(g - a)))
    if shallow:
        assert dev <= max(LOGIT_TOL, 0.25 * q), ("shallow int8 logits", dev, q)
    else:
        rms = lambda x: float(np.sqrt(np.mean(x * x)))
        assert rms(g - a) <= 2.0 * rms(a - b) + 1e-3, ("deep int8 logits", rms(g - a), rms(a - b))
    return dev, q
