"""Greedy decoding, speculative cycles, acceptance/rollback and DyTC (oracle).

Sequence bookkeeping (shared reading of [CLaSp] §一 and §三):
  * the cache holds committed tokens x_0..x_{t-1} in slots 0..t-1;
  * the pending token x_t (last emitted, not yet run through the model) is
    the first row of the next draft/verify;
  * a linear cycle drafts d_1..d_K with the skipped-layer model (slots
    t..t+K-1), then verifies rows [x_t, d_1..d_K] at positions t..t+K with
    the full model in one pass ([CLaSp] §三 stage 2);
  * greedy acceptance: n = the longest prefix with argmax(row r-1) == d_r;
    the bonus token is argmax(row n), the full model's prediction that
    overrides the first rejected draft ([CLaSp] §一, §三); slots t..t+n are
    kept, the rest of the new slots are dropped (rollback), the pending
    token becomes the bonus and the committed length t + n + 1.
  Greedy acceptance makes the output identical to plain greedy decoding,
  the losslessness the pages claim ([CAS-blog] §1, [CAS-paper] abstract,
  [CLaSp] §四).

Tree cycles ([CAS-paper] abstract: DyTC, a dynamic tree of multi-level
drafts, verified in one pass): node c sits in slot t + c at position
t + depth(c) and sees the committed prefix plus its ancestors; acceptance
walks from the root to the child whose token equals the current argmax;
the accepted path is then compacted into slots t+1..t+n.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

import ssd_inputs as si

from .model import KVCache, Weights, argmax_f32, causal_vis, forward, top1_prob, top2_f32, top_gap


@dataclasses.dataclass
class Target:
    """Full-model states of the last accepted token: the CLaSp DP target."""
    token: int
    pos: int
    states: List[np.ndarray]  # residual after i layers, i = 0..L


@dataclasses.dataclass
class Cycle:
    drafts: List[int]
    argmax: List[int]
    gaps: List[float]  # top-1 - top-2 of the verify logits per row
    n_accepted: int
    bonus: int
    path: List[int]


class Session:
    """One request (batch 1): KV cache, committed length t, pending token."""

    def __init__(self, Wt: Weights, max_ctx: Optional[int] = None):
        self.Wt = Wt
        self.cfg = Wt.cfg
        self.max_ctx = self.cfg.max_ctx if max_ctx is None else max_ctx
        self.cache = KVCache(self.cfg, self.max_ctx)
        self.t = 0
        self.pending: Optional[int] = None
        self.target: Optional[Target] = None

    # -- prefill / autoregressive ------------------------------------------
    def prefill(self, tokens: Sequence[int]):
        tokens = [int(x) for x in tokens]
        n, t = len(tokens), self.t
        logits, states = forward(self.Wt, self.cache, tokens, range(t, t + n), range(t, t + n), causal_vis(t, n))
        self.t = t + n
        self.pending = int(argmax_f32(logits[-1]))
        self.target = Target(tokens[-1], t + n - 1, [s[-1].copy() for s in states])
        return self.pending, logits

    def ar_step(self):
        """Run the pending token through the full model; return (new pending token, logits row)."""
        t = self.t
        logits, states = forward(self.Wt, self.cache, [self.pending], [t], [t], causal_vis(t, 1))
        self.target = Target(self.pending, t, [s[0].copy() for s in states])
        self.t = t + 1
        self.pending = int(argmax_f32(logits[0]))
        return self.pending, logits[0]

    def rollback(self, new_len: int) -> None:
        """Truncate the committed length (slots >= new_len become scratch)."""
        assert 0 <= new_len <= self.t
        self.t = new_len

    # -- linear speculative cycle --------------------------------------------
    def draft_linear(self, skip: Sequence[int], k: int, act_int8: bool = False,
                     gaps: Optional[List[float]] = None, force: Optional[Sequence[int]] = None,
                     exit_thr: float = 0.0, probs: Optional[List[float]] = None,
                     rows: Optional[List[np.ndarray]] = None, exit_layers: int = 0,
                     argmax: Optional[List[int]] = None) -> List[int]:
        """Up to K drafts with the layer-skipped model; draft r runs in slot t + r and sees slots [0, t + r].

        Draft exit ([CLaSp] §四): after draft r, if the draft model's top-1
        softmax probability p1 is below exit_thr, drafting stops; draft r is
        kept (it is the last one) and no further draft is generated, so
        1 <= len(result) <= k.  exit_thr = 0 never stops early (p1 > 0).
        gaps / probs / rows (optional) receive, per draft step, the top-1
        minus top-2 logit, p1 and the logits row; force (optional) feeds the
        given tokens as drafts instead of the argmax (used to follow another
        implementation, so every step is computed on the same inputs as
        there; entries that are None, or past its end, take the argmax);
        argmax (optional) receives the oracle's own greedy token of
        each step, forced or not.  exit_layers: the draft model's early exit
        (model.forward)."""
        t, x, out = self.t, self.pending, []
        for r in range(k):
            logits, _ = forward(self.Wt, self.cache, [x], [t + r], [t + r], causal_vis(t + r, 1), skip=skip,
                                act_int8=act_int8, exit_layers=exit_layers)
            if gaps is not None:
                gaps.append(top_gap(logits[0]))
            if rows is not None:
                rows.append(logits[0].copy())
            p1 = top1_prob(logits[0])
            if probs is not None:
                probs.append(p1)
            own = int(argmax_f32(logits[0]))
            if argmax is not None:
                argmax.append(own)
            x = own if force is None or r >= len(force) or force[r] is None else int(force[r])
            out.append(x)
            if p1 < exit_thr:
                break
        return out

    def verify_linear(self, drafts: Sequence[int], follow: Optional[Tuple[int, int]] = None,
                      logits_out: Optional[List[np.ndarray]] = None) -> Cycle:
        """Verify [pending, drafts] in one full-model pass and accept greedily.

        The returned Cycle is the oracle's own decision.  follow = (n, bonus)
        commits another implementation's decision instead (the state then
        continues from n accepted drafts and that bonus token), so the two can
        be compared cycle by cycle through a near-tie."""
        t, K = self.t, len(drafts)
        rows = [self.pending] + [int(d) for d in drafts]
        logits, states = forward(self.Wt, self.cache, rows, range(t, t + K + 1), range(t, t + K + 1),
                                 causal_vis(t, K + 1))
        if logits_out is not None:
            logits_out.append(logits)
        am = [int(a) for a in argmax_f32(logits)]
        n = 0
        while n < K and am[n] == rows[n + 1]:
            n += 1
        bonus = am[n]
        cyc = Cycle(list(rows[1:]), am, [top_gap(r) for r in logits], n, bonus, list(range(n + 1)))
        if follow is not None:
            n, bonus = int(follow[0]), int(follow[1])
            assert 0 <= n <= K
        self.target = Target(rows[n], t + n, [s[n].copy() for s in states])
        self.t = t + n + 1
        self.pending = bonus
        return cyc

    # -- tree cycle --------------------------------------------------------------
    def tree_vis(self, parents: Sequence[int]) -> np.ndarray:
        """Node c (slot t + c) sees slots [0, t) and its ancestors-or-self."""
        t, N = self.t, len(parents)
        vis = np.zeros((N, t + N), dtype=bool)
        for c in range(N):
            vis[c, :t] = True
            a = c
            while a >= 0:
                vis[c, t + a] = True
                a = parents[a]
        return vis

    def draft_node(self, node: int, parents: Sequence[int], depth: Sequence[int], token: int,
                   skip: Sequence[int], act_int8: bool, exit_layers: int = 0,
                   rows: Optional[List[np.ndarray]] = None):
        """One draft expansion of `node`: return its (top-1, top-2) continuation tokens.
        rows (optional) receives the expansion's logits row."""
        t = self.t
        vis = self.tree_vis(list(parents[: node + 1]))[node: node + 1]
        logits, _ = forward(self.Wt, self.cache, [token], [t + depth[node]], [t + node], vis, skip=skip,
                            act_int8=act_int8, exit_layers=exit_layers)
        if rows is not None:
            rows.append(logits[0].copy())
        return top2_f32(logits[0])

    def verify_tree(self, tokens: Sequence[int], parents: Sequence[int],
                    follow: Optional[Tuple[Sequence[int], int]] = None,
                    logits_out: Optional[List[np.ndarray]] = None) -> Cycle:
        """Tree verify and greedy walk; the returned Cycle is the oracle's own decision.
        follow = (path, bonus) commits another implementation's accepted path instead
        (compaction, target and pending token follow it), as in verify_linear."""
        t, N = self.t, len(tokens)
        depth = tree_depths(parents)
        logits, states = forward(self.Wt, self.cache, list(tokens), [t + d for d in depth], range(t, t + N),
                                 self.tree_vis(parents))
        if logits_out is not None:
            logits_out.append(logits)
        am = [int(a) for a in argmax_f32(logits)]
        children: Dict[int, List[int]] = {}
        for c in range(1, N):
            children.setdefault(parents[c], []).append(c)
        path, cur = [0], 0
        while True:
            nxt = [c for c in children.get(cur, []) if tokens[c] == am[cur]]
            if not nxt:
                break
            cur = nxt[0]
            path.append(cur)
        n = len(path) - 1
        bonus = am[cur]
        cyc = Cycle([int(x) for x in tokens[1:]], am, [top_gap(r) for r in logits], n, bonus, list(path))
        if follow is not None:
            path, bonus = [int(x) for x in follow[0]], int(follow[1])
            n, cur = len(path) - 1, path[-1]
        for i in range(1, n + 1):  # compact the accepted path's KV into slots t+1..t+n
            self.cache.copy_slot(t + i, t + path[i])
        self.target = Target(int(tokens[cur]), t + n, [s[cur].copy() for s in states])
        self.t = t + n + 1
        self.pending = bonus
        return cyc


def tree_depths(parents: Sequence[int]) -> List[int]:
    d = []
    for c, p in enumerate(parents):
        d.append(0 if p < 0 else d[p] + 1)
    return d


# ----------------------------------------------------------------------------
# DyTC: dynamic tree cascade routing
# ----------------------------------------------------------------------------


def level_costs(cfg: si.ModelConfig) -> List[float]:
    """Latency prediction per cascade level, as a fraction of one verify pass.

    [CAS-blog] §3.2 gives latency = b0 + b1 * seq_len + b2 * layer_depth; at
    batch 1 a pass streams the weights of the layers it runs plus the
    lm_head, so the reading here is b0 = lm_head bytes, b2 = bytes of one
    layer, b1 = 0, normalised by the full pass.
    """
    hd, d, F = cfg.head_dim, cfg.d_model, cfg.ffn
    w_layer = 2 * (cfg.qkv_rows * d + d * cfg.n_q_heads * hd + 2 * F * d + d * F)
    w_lm = 2 * cfg.vocab * d
    full = cfg.n_layers * w_layer + w_lm
    out = []
    for l, (skip, _) in enumerate(cfg.levels):
        n_run = len(set(range(cfg.n_layers - level_exit(cfg, l))) - set(skip))
        out.append((n_run * w_layer + w_lm) / full)
    return out


def level_exit(cfg: si.ModelConfig, l: int) -> int:
    """Early-exit layer count of cascade level l (0 when the config gives none)."""
    return cfg.level_exit[l] if l < len(cfg.level_exit) else 0


@dataclasses.dataclass
class TreePlan:
    parents: List[int]
    depth: List[int]
    prob: List[float]
    cap: List[int]  # highest level a node may be expanded with (level of the expansion that made it)
    expansions: List[Tuple[int, int]]  # (node, level index 0-based), in order


class DyTC:
    """Acceptance-rate EMA + latency-aware tree construction.

    EMA ([CAS-blog] §3.1): a_l <- alpha * rate_l + (1 - alpha) * a_l, alpha = 0.2,
    initial 0.65 (the blog's 0.6-0.7 starting threshold, §4.1 item 2).

    Tree rule (the pages give only "heuristics of acceptance rates and
    latency prediction", [CAS-paper] abstract and method sketch; this
    reading is stated in full so the GPU host can restate it):
      * the root has p = 1; expanding node u with level l gives a rank-0
        child with p(u) a_l and a rank-1 child with p(u) (1 - a_l) a_l;
      * E = 1 + sum of p over non-root nodes, T = 1 + sum of c_l over the
        expansions made;
      * candidates: unexpanded nodes of depth < max_depth, levels up to the
        node's cap (the level that created it; root: any level), so every
        layer a child runs was also run for all of its ancestors (nested
        skip sets);
      * gain(u, l) = p(u) a_l + p(u) (1 - a_l) a_l; pick the largest gain/c_l,
        ties to the lower node index, then the lower level;
      * expand while gain/c_l > E/T and a node slot is free; the rank-1
        child is added only if a slot is still free.
    """

    def __init__(self, cfg: si.ModelConfig, costs: Optional[Sequence[float]] = None, rules: bool = False,
                 betas: Optional[Sequence[Sequence[float]]] = None):
        """costs: fixed level costs (default: the byte ratio of level_costs); betas: latency
        models (16-bit, int8) instead, costs taken at plan time as latency(seq_len, layers run,
        level's mode) / latency(seq_len, L, 16-bit); rules: use only the first
        latency.cascade_depth(L, levels, seq_len) levels."""
        self.cfg = cfg
        self.a = [cfg.ema_init] * len(cfg.levels)
        self.c = list(level_costs(cfg) if costs is None else costs)
        self.rules = rules
        self.betas = betas

    def plan(self, seq_len: int = 0) -> TreePlan:
        from .latency import cascade_depth, predict

        cfg = self.cfg
        nl = len(cfg.levels)
        if self.betas is not None:
            full = predict(self.betas[0], seq_len, cfg.n_layers)
            self.c = []
            for l, (skip, int8) in enumerate(cfg.levels):
                run = len(set(range(cfg.n_layers - level_exit(cfg, l))) - set(skip))
                self.c.append(predict(self.betas[1 if int8 else 0], seq_len, run) / full)
        if self.rules:
            nl = cascade_depth(cfg.n_layers, nl, seq_len)
        parents, depth, prob, cap, expanded = [-1], [0], [1.0], [nl - 1], [False]
        exps: List[Tuple[int, int]] = []
        E, T = 1.0, 1.0
        while True:
            best = None
            for u in range(len(parents)):
                if expanded[u] or depth[u] >= cfg.tree_max_depth:
                    continue
                for l in range(cap[u] + 1):
                    a = self.a[l]
                    gain = prob[u] * a + prob[u] * (1.0 - a) * a
                    score = gain / self.c[l]
                    if best is None or score > best[0]:
                        best = (score, u, l)
            if best is None or len(parents) - 1 >= cfg.tree_max_nodes or not best[0] > E / T:
                break
            _, u, l = best
            a = self.a[l]
            expanded[u] = True
            exps.append((u, l))
            for p in (prob[u] * a, prob[u] * (1.0 - a) * a):
                if len(parents) - 1 >= cfg.tree_max_nodes:
                    break
                parents.append(u)
                depth.append(depth[u] + 1)
                prob.append(p)
                cap.append(l)
                expanded.append(False)
                E += p
            T += self.c[l]
        return TreePlan(parents, depth, prob, cap, exps)

    def update(self, plan: TreePlan, tokens: Sequence[int], cyc: Cycle) -> None:
        """One EMA step from the verify result: every expanded node on the accepted walk
        (including the node where the walk stopped) is an event of its level, a success
        when the target's argmax there equals its rank-0 child's token."""
        nl = len(self.a)
        level_of = {u: l for u, l in plan.expansions}
        first_child = {}
        for c in range(1, len(plan.parents)):
            first_child.setdefault(plan.parents[c], c)
        ev, ok = [0] * nl, [0] * nl
        for u in cyc.path:
            if u in level_of:
                l = level_of[u]
                ev[l] += 1
                ok[l] += int(cyc.argmax[u] == tokens[first_child[u]])
        alpha = self.cfg.ema_alpha
        for l in range(nl):
            if ev[l]:
                self.a[l] = alpha * (ok[l] / ev[l]) + (1.0 - alpha) * self.a[l]


def run_tree_cycle(sess: Session, dytc: DyTC):
    """Plan the tree, run its draft expansions in order, verify, update the EMA."""
    cfg = sess.cfg
    plan = dytc.plan(sess.t)
    N = len(plan.parents)
    tokens = [sess.pending] + [0] * (N - 1)
    kids: Dict[int, List[int]] = {}
    for c in range(1, N):
        kids.setdefault(plan.parents[c], []).append(c)
    for u, l in plan.expansions:
        skip, int8 = cfg.levels[l]
        top = sess.draft_node(u, plan.parents, plan.depth, tokens[u], skip, int8, level_exit(cfg, l))
        for rank, c in enumerate(kids.get(u, [])):
            tokens[c] = top[rank]
    cyc = sess.verify_tree(tokens, plan.parents)
    dytc.update(plan, tokens, cyc)
    return plan, tokens, cyc


# ----------------------------------------------------------------------------
# end-to-end drivers
# ----------------------------------------------------------------------------


def generate_ar(Wt: Weights, prompt: Sequence[int], n_gen: int, max_ctx: Optional[int] = None) -> List[int]:
    sess = Session(Wt, max_ctx)
    first, _ = sess.prefill(prompt)
    out = [first]
    while len(out) < n_gen:
        nxt, _ = sess.ar_step()
        out.append(nxt)
    return out[:n_gen]


@dataclasses.dataclass
class SpecResult:
    tokens: List[int]
    cycles: List[Cycle]
    masks: List[Tuple[int, ...]]  # skip set in force, per DP refresh (CLaSp) or the static one
    dp_values: List[float]
    conf: List[List[float]] = dataclasses.field(default_factory=list)  # per cycle: each draft's top-1 probability


def generate_spec(Wt: Weights, prompt: Sequence[int], n_gen: int, max_ctx: Optional[int] = None,
                  skip: Optional[Sequence[int]] = None, k: Optional[int] = None, act_int8: bool = False,
                  dp_n_skip: Optional[int] = None, dp_interval: Optional[int] = None,
                  exit_thr: float = 0.0, early_exit: int = 0) -> SpecResult:
    """Linear speculative generation: static skip set, or CLaSp DP-selected skip set
    refreshed every `dp_interval` verify steps (and once right after prefill);
    exit_thr > 0 ends each cycle's drafting at the first draft whose top-1
    probability is below it ([CLaSp] §四); early_exit = e drafts with the last e
    layers cut off as well ([CAS-blog] §2.1 item 2)."""
    from .clasp import dp_select

    cfg = Wt.cfg
    k = cfg.draft_k if k is None else k
    dp_n = cfg.dp_n_skip if dp_n_skip is None else dp_n_skip
    dp_every = cfg.dp_interval if dp_interval is None else dp_interval
    sess = Session(Wt, max_ctx)
    first, _ = sess.prefill(prompt)
    out, cycles, masks, values, conf = [first], [], [], [], []
    cur = tuple(cfg.skip if skip is None else skip)
    if dp_n:
        cur, val = dp_select(sess, dp_n)
        masks.append(cur)
        values.append(val)
    else:
        masks.append(cur)
    while len(out) < n_gen:
        probs: List[float] = []
        drafts = sess.draft_linear(cur, k, act_int8, exit_thr=exit_thr, probs=probs, exit_layers=early_exit)
        conf.append(probs)
        cyc = sess.verify_linear(drafts)
        cycles.append(cyc)
        out += drafts[: cyc.n_accepted] + [cyc.bonus]
        if dp_n and dp_every and len(cycles) % dp_every == 0 and len(out) < n_gen:
            cur, val = dp_select(sess, dp_n)
            masks.append(cur)
            values.append(val)
    return SpecResult(out[:n_gen], cycles, masks, values, conf)


def hcascade_chain(lens: Sequence[int]) -> Tuple[List[int], List[int]]:
    """Horizontal cascade ([CAS-paper] abstract: the classic cascade DyTC is compared with; the
    horizontal form drafts the earlier positions of a chain with the more accurate levels and the later
    ones with the cheaper levels): (parents, level of each draft position) of a chain whose first
    lens[-1] drafts come from the highest level, then lens[-2] from the next, ..., lens[0] from L1."""
    levels = [l for l in range(len(lens) - 1, -1, -1) for _ in range(lens[l])]
    return [-1] + list(range(len(levels))), levels


def generate_hcascade(Wt: Weights, prompt: Sequence[int], n_gen: int, lens: Sequence[int],
                      max_ctx: Optional[int] = None):
    """Generation with horizontal-cascade chains drafted node by node at their levels, each chain
    verified in one pass (tree verify over a chain)."""
    cfg = Wt.cfg
    parents, levels = hcascade_chain(lens)
    depth = tree_depths(parents)
    sess = Session(Wt, max_ctx)
    first, _ = sess.prefill(prompt)
    out, cycles = [first], []
    while len(out) < n_gen:
        tokens = [sess.pending]
        for r, l in enumerate(levels):
            skip, int8 = cfg.levels[l]
            tokens.append(sess.draft_node(r, parents, depth, tokens[r], skip, int8, level_exit(cfg, l))[0])
        cyc = sess.verify_tree(tokens, parents)
        cycles.append(cyc)
        out += [tokens[c] for c in cyc.path[1:]] + [cyc.bonus]
    return out[:n_gen], cycles


def generate_vcascade(Wt: Weights, prompt: Sequence[int], n_gen: int, lo: int, hi: int, k: int,
                      max_ctx: Optional[int] = None):
    """Vertical cascade (the other classic cascade DyTC is compared with, [CAS-paper] abstract): the
    drafts of level `hi` come from level `lo`.  Each cycle: `lo` drafts k tokens; `hi` runs the
    pending token and those drafts as one pass (causal, slots t..t+k) and keeps the longest prefix
    its greedy predictions agree with, then its own prediction where they first differ (k tokens at
    most); the target verifies that chain."""
    cfg = Wt.cfg
    skip_lo, i8_lo = cfg.levels[lo]
    skip_hi, i8_hi = cfg.levels[hi]
    sess = Session(Wt, max_ctx)
    first, _ = sess.prefill(prompt)
    out, cycles = [first], []
    while len(out) < n_gen:
        t = sess.t
        d = sess.draft_linear(skip_lo, k, i8_lo, exit_layers=level_exit(cfg, lo))
        rows = [sess.pending] + d
        logits, _ = forward(Wt, sess.cache, rows, range(t, t + k + 1), range(t, t + k + 1), causal_vis(t, k + 1),
                            skip=skip_hi, act_int8=i8_hi, exit_layers=level_exit(cfg, hi))
        am = [int(a) for a in argmax_f32(logits)]
        n = 0
        while n < k and am[n] == d[n]:
            n += 1
        drafts = d[:n] + ([am[n]] if n < k else [])
        cyc = sess.verify_linear(drafts)
        cycles.append(cyc)
        out += drafts[: cyc.n_accepted] + [cyc.bonus]
    return out[:n_gen], cycles


def generate_tree(Wt: Weights, prompt: Sequence[int], n_gen: int, max_ctx: Optional[int] = None,
                  costs: Optional[Sequence[float]] = None, rules: bool = False,
                  betas: Optional[Sequence[Sequence[float]]] = None):
    sess = Session(Wt, max_ctx)
    dytc = DyTC(Wt.cfg, costs, rules, betas)
    first, _ = sess.prefill(prompt)
    out, records = [first], []
    while len(out) < n_gen:
        plan, tokens, cyc = run_tree_cycle(sess, dytc)
        records.append((plan, tokens, cyc, list(dytc.a)))
        out += [tokens[c] for c in cyc.path[1:]] + [cyc.bonus]
    return out[:n_gen], records
