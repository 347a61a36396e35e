"""Expected values for the full-size workloads, written by the CPU oracle alone.

    python tests/golden/make_scale_goldens.py [--out DIR] [llama3_70b_clasp] [llama2_13b_cascade] [llama3_8b_clasp]

Writes scale_<workload>.npz into DIR (default tests/golden; all three workloads when none is named);
tests/test_gpu_scale.py compares the GPU path with tests/golden/scale_<workload>.npz.

The models are far too large for the float64 oracle (64-280 GB of float64
weights), so the oracle runs with compute="f32": weights widened exactly to
float32, projection products taken in float32, everything else in float64
(pinned against the float64 oracle by
tests/test_oracle.py::test_f32_products_match_f64).  Only oracle/ and the
seeded input generators are called.

What each file holds (a logits "sample" is the row at 4096 fixed seeded
vocabulary indices followed by the row's own 64 largest entries):

llama3_8b_clasp  -- CLaSp on the Llama-3-8B shape ([CLaSp] §三): prompt of
    1024 ids, DP (16 of 32 layers) right after prefill and every 32 verify
    steps, linear drafts of 6, 512 tokens.  Prefill: first token, its top-1 /
    top-2 gap, the last prompt token's residual after every layer (float16)
    and a logits sample.  Per cycle: committed length before it, the drafts
    and each draft step's gap, the verify argmax and gap of every row, the
    accepted count and bonus token.  Per DP run: the cycle it precedes, the
    mask, dp[L][n] and both candidates' cosines of every (i, j) cell.  Cycle
    0 also keeps logits samples of its draft steps and verify rows.
llama2_13b_cascade -- CAS-Spec cascade on the Llama-2-13B shape (fp16)
    ([CAS-blog] §2.2, [CAS-paper] abstract): prompt 256.  Prefill as above
    (full logits row), the full logits of three int8 drafts of the first
    prompt token at position 0 (no prefix) -- one layer run, level L2 (30 %
    skipped + int8), level L3 (all layers + int8) -- each with its 16-bit
    twin, then 4 DyTC tree
    cycles: acceptance estimates before and after, the plan (parents,
    expansions), every expansion's three largest logits (ids, values), the
    tree tokens, verify argmax and gaps, accepted path and bonus.
llama3_70b_clasp -- the Llama-3-70B shape ([CLaSp] §四, 44 of 80 layers
    skipped): prompt of 2048 ids.  Prefill as for the 8B shape, then the DP
    for 44 skipped layers (45 rows per layer) on the last prompt token.
"""
from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import ssd_inputs as si  # noqa: E402
from oracle import clasp, decode  # noqa: E402
from oracle.model import Weights, top_gap  # noqa: E402

N_SAMPLE, N_TOP = 4096, 64


def log(*a):
    print(time.strftime("%H:%M:%S"), *a, flush=True)


def sample_idx(V: int) -> np.ndarray:
    return np.sort(np.random.default_rng(20261203).choice(V, min(N_SAMPLE, V), replace=False)).astype(np.int32)


def logit_sample(row: np.ndarray, base: np.ndarray):
    top = np.argsort(-np.asarray(row, dtype=np.float64), kind="stable")[:N_TOP].astype(np.int32)
    idx = np.concatenate([base, top])
    return idx, np.asarray(row, dtype=np.float64)[idx].astype(np.float32)


def dp_record(table, L: int, n: int) -> np.ndarray:
    cands = np.full((L + 1, n + 1, 2), np.nan, dtype=np.float64)
    for i in range(L + 1):
        for j, e in table[i].items():
            if e[2] is not None:
                cands[i, j, 0] = e[2]
            if e[3] is not None:
                cands[i, j, 1] = e[3]
    return cands


def mask_u8(skip, L):
    m = np.zeros(L, dtype=np.uint8)
    m[list(skip)] = 1
    return m


def prefill_record(sess, prompt, out, base):
    t0 = time.time()
    first, logits = sess.prefill(prompt)
    log(f"prefill of {len(prompt)} tokens: {time.time() - t0:.0f} s, first token {first}")
    out["first"] = np.int32(first)
    out["first_gap"] = np.float64(top_gap(logits[-1]))
    out["h_last"] = np.stack(sess.target.states).astype(np.float16)
    if base is None:
        out["prefill_logits"] = logits[-1].astype(np.float32)
    else:
        i, v = logit_sample(logits[-1], base)
        out["prefill_idx"], out["prefill_val"] = i, v
    return first


def clasp_8b(path):
    cfg = si.CONFIGS["llama3_8b_clasp"]
    L, n, K, every = cfg.n_layers, cfg.dp_n_skip, cfg.draft_k, cfg.dp_interval
    W = Weights(cfg, keep_bits=False, compute="f32", evict=False, cache_bytes=40 << 30)
    sess = decode.Session(W, cfg.max_ctx)
    prompt = si.prompt(cfg)
    base = sample_idx(cfg.vocab)
    out = {}
    first = prefill_record(sess, prompt, out, base)
    toks = [first]
    dp_at, dp_mask, dp_val, dp_cands = [], [], [], []

    def run_dp(at):
        t0 = time.time()
        skip, val, table = clasp.dp_search(sess, n)
        dp_at.append(at)
        dp_mask.append(mask_u8(skip, L))
        dp_val.append(val)
        dp_cands.append(dp_record(table, L, n))
        log(f"DP before cycle {at}: {skip} value {val:.6f} ({time.time() - t0:.0f} s)")
        return skip

    skip = run_dp(0)
    c_t, c_d, c_dg, c_am, c_vg, c_n, c_b = [], [], [], [], [], [], []
    t_start = time.time()
    while len(toks) < cfg.n_gen:
        c = len(c_t)
        c_t.append(sess.t)
        gaps, drows, vrows = [], [], []
        drafts = sess.draft_linear(skip, K, gaps=gaps, rows=drows if c == 0 else None)
        cyc = sess.verify_linear(drafts, logits_out=vrows if c == 0 else None)
        if c == 0:
            s = [logit_sample(r, base) for r in drows]
            out["draft0_idx"] = np.stack([a for a, _ in s])
            out["draft0_val"] = np.stack([b for _, b in s])
            s = [logit_sample(r, base) for r in vrows[0]]
            out["verify0_idx"] = np.stack([a for a, _ in s])
            out["verify0_val"] = np.stack([b for _, b in s])
        c_d.append(drafts)
        c_dg.append(gaps)
        c_am.append(cyc.argmax)
        c_vg.append(cyc.gaps)
        c_n.append(cyc.n_accepted)
        c_b.append(cyc.bonus)
        toks += drafts[: cyc.n_accepted] + [cyc.bonus]
        if c % 16 == 0:
            el = time.time() - t_start
            log(f"cycle {c}: {len(toks)} tokens, n_acc {cyc.n_accepted}, {el / (c + 1):.1f} s/cycle")
        if (c + 1) % every == 0 and len(toks) < cfg.n_gen:
            skip = run_dp(c + 1)
    out.update(tokens=np.asarray(toks[: cfg.n_gen], dtype=np.int32), cyc_t=np.asarray(c_t, dtype=np.int32),
               cyc_drafts=np.asarray(c_d, dtype=np.int32), cyc_draft_gaps=np.asarray(c_dg),
               cyc_argmax=np.asarray(c_am, dtype=np.int32), cyc_gaps=np.asarray(c_vg),
               cyc_n=np.asarray(c_n, dtype=np.int32), cyc_bonus=np.asarray(c_b, dtype=np.int32),
               dp_at=np.asarray(dp_at, dtype=np.int32), dp_mask=np.stack(dp_mask), dp_val=np.asarray(dp_val),
               dp_cands=np.stack(dp_cands).astype(np.float32))
    out["meta"] = np.array(json.dumps({"workload": cfg.name, "prompt_len": cfg.prompt_len, "n_gen": cfg.n_gen,
                                       "k": K, "dp_n_skip": n, "dp_interval": every, "compute": "f32"}))
    np.savez_compressed(path, **out)


def cascade_13b(path, n_cycles=4):
    cfg = si.CONFIGS["llama2_13b_cascade"]
    L = cfg.n_layers
    W = Weights(cfg, keep_bits=True, compute="f32", evict=False, cache_bytes=20 << 30)
    sess = decode.Session(W, cfg.max_ctx)
    prompt = si.prompt(cfg)
    out = {}
    prefill_record(sess, prompt, out, None)
    # int8 drafts with no committed prefix (the first prompt token pending at position 0), each with its
    # 16-bit twin (the same step without int8): one layer run (shallow), and levels L2 and L3 (deep)
    one = tuple(i for i in range(L) if i != L // 2)
    for name, skip in (("i8one", one), ("l2", cfg.levels[1][0]), ("l3", cfg.levels[2][0])):
        s0 = decode.Session(W, 64)
        s0.pending = int(prompt[0])
        r8, r16 = [], []
        d = s0.draft_linear(skip, 1, act_int8=True, rows=r8)
        s0.draft_linear(skip, 1, act_int8=False, rows=r16, force=d)
        out[f"{name}_token"] = np.int32(d[0])
        out[f"{name}_gap"] = np.float64(top_gap(r8[0]))
        out[f"{name}_logits"] = r8[0].astype(np.float32)
        out[f"{name}_logits16"] = r16[0].astype(np.float32)
        log(f"{name} int8 draft token {d[0]}, int8 effect {float(np.max(np.abs(r8[0] - r16[0]))):.3f}")
    dytc = decode.DyTC(cfg)
    recs = []
    for c in range(n_cycles):
        t0 = time.time()
        ema0 = list(dytc.a)
        t_before = sess.t
        plan = dytc.plan(sess.t)
        N = len(plan.parents)
        tokens = [sess.pending] + [0] * (N - 1)
        kids = {}
        for ch in range(1, N):
            kids.setdefault(plan.parents[ch], []).append(ch)
        top3 = []
        for u, l in plan.expansions:
            skip, int8 = cfg.levels[l]
            rows = []
            top = sess.draft_node(u, plan.parents, plan.depth, tokens[u], skip, int8, decode.level_exit(cfg, l),
                                  rows=rows)
            x = rows[0].astype(np.float32)
            order = np.lexsort((np.arange(x.size), -x))[:3]
            top3.append((order.tolist(), rows[0][order].tolist()))
            for r, ch in enumerate(kids.get(u, [])):
                tokens[ch] = top[r]
        cyc = sess.verify_tree(tokens, plan.parents)
        dytc.update(plan, tokens, cyc)
        recs.append({"t": t_before, "ema_before": ema0, "ema_after": list(dytc.a), "parents": plan.parents,
                     "expansions": plan.expansions, "top3": top3, "tokens": [int(x) for x in tokens],
                     "argmax": cyc.argmax, "gaps": cyc.gaps, "path": cyc.path, "bonus": cyc.bonus})
        log(f"tree cycle {c}: {N} nodes, {len(plan.expansions)} expansions, path {cyc.path} "
            f"({time.time() - t0:.0f} s)")
    out["cycles"] = np.array(json.dumps(recs))
    out["meta"] = np.array(json.dumps({"workload": cfg.name, "prompt_len": cfg.prompt_len, "compute": "f32"}))
    np.savez_compressed(path, **out)


def clasp_70b(path):
    cfg = si.CONFIGS["llama3_70b_clasp"]
    L, n = cfg.n_layers, cfg.dp_n_skip
    # one layer's float32 matrices kept (3.4 GB): every layer is generated again for each pass over the model
    W = Weights(cfg, keep_bits=False, compute="f32", evict=True, cache_bytes=4 << 30)
    prompt = si.prompt(cfg)
    sess = decode.Session(W, len(prompt) + 64)
    base = sample_idx(cfg.vocab)
    out = {}
    prefill_record(sess, prompt, out, base)
    t0 = time.time()
    skip, val, table = clasp.dp_search(sess, n)
    log(f"DP n={n}: {skip} value {val:.6f} ({time.time() - t0:.0f} s)")
    out.update(dp_mask=mask_u8(skip, L), dp_val=np.float64(val), dp_cands=dp_record(table, L, n).astype(np.float32))
    out["meta"] = np.array(json.dumps({"workload": cfg.name, "prompt_len": len(prompt), "dp_n_skip": n,
                                       "compute": "f32"}))
    np.savez_compressed(path, **out)


JOBS = {"llama3_70b_clasp": clasp_70b, "llama2_13b_cascade": cascade_13b, "llama3_8b_clasp": clasp_8b}


def main(args):
    out_dir = HERE
    if args[:1] == ["--out"]:
        out_dir, args = args[1], args[2:]
        os.makedirs(out_dir, exist_ok=True)
    si.build_host()
    for name in args or list(JOBS):
        path = os.path.join(out_dir, f"scale_{name}.npz")
        log(f"== {name} -> {path}")
        t0 = time.time()
        JOBS[name](path)
        log(f"== {name} done in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main(sys.argv[1:])
