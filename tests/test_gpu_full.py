"""GPU parity at the workloads' real shapes.

* Llama-3-8B shape, all 32 layers: prefill logits and every layer's hidden
  state against the oracle, the CLaSp DP (n = 16), three teacher-forced
  speculative cycles (the oracle drafts on the GPU's drafts and follows its
  acceptance; near-ties resynchronise instead of ending the test), an int8
  draft's logits, a draft-equals-target cycle (all K drafts accepted, the
  cache kept and rolled back), then greedy steps.
* Llama-3-70B and Llama-2-13B shapes cut to a few layers: the same kernels at
  the real d_model, heads, FFN and vocabulary against the oracle, including
  the 13B DyTC tree (every expansion, every verify row), the int8 cascade
  levels' logits and a DyTC generation recomputed cycle by cycle.
* 70B and 13B at full size on the GPU alone: properties that hold at any
  size (speculative output == autoregressive output; the DP keeps n layers
  skipped and n = 0 reproduces the full model).

The oracle runs in its float32-product mode here (weights exact in float32,
products in float32, the rest float64; pinned against float64 in
tests/test_oracle.py), which keeps these runs within minutes.
"""
import gc

import numpy as np
import pytest

import ssd_inputs as si
from oracle import clasp, decode
from oracle.model import Weights

from gpu_util import (HIDDEN_COS, LOGIT_TOL, NEAR_TIE, Follow, cos, int8_logits_check, int8_prefix_free,
                      tree_cycle_against_oracle)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__

    __graft_entry__.build()


def free():
    gc.collect()
    torch.cuda.empty_cache()


def oracle_weights(cfg):
    return Weights(cfg, keep_bits=False, compute="f32", evict=False, cache_bytes=48 << 30)


def check_prefill(eng, sess, prompt, row):
    """Prefill on both sides: logits and every layer's residual of the last prompt token; a first token
    that differs must be a near-tie, and the oracle then continues from the GPU's token."""
    first = eng.prefill(prompt)
    o_first, o_logits = sess.prefill(prompt)
    err = float(np.max(np.abs(eng.logits(0) - o_logits[-1])))
    assert err < LOGIT_TOL, err
    cs = [cos(eng.hidden(l, row), sess.target.states[l]) for l in range(sess.cfg.n_layers + 1)]
    assert min(cs) >= HIDDEN_COS, cs
    if first != o_first:
        assert decode.model.top_gap(o_logits[-1]) < NEAR_TIE
        sess.pending = first
    return first


def check_cycle(eng, sess, skip, k):
    """One teacher-forced speculative cycle: the oracle drafts on the GPU's drafts (every step compared,
    the last step's logits too), both verify the same rows (every row's logits compared), and the oracle
    follows the GPU's acceptance.  Returns the near-tie count."""
    near = 0
    drafts = eng.draft(skip, k)
    gaps, am, rows = [], [], []
    sess.draft_linear(skip, k, gaps=gaps, force=drafts, argmax=am, rows=rows)
    err = float(np.max(np.abs(eng.logits(0) - rows[-1])))
    assert err < LOGIT_TOL, ("draft logits", err)
    for r in range(k):
        if am[r] != drafts[r]:
            assert gaps[r] < NEAR_TIE, (r, drafts, am, gaps)
            near += 1
    n_acc, path, bonus = eng.verify([sess.pending] + drafts)
    lo = []
    cyc = sess.verify_linear(drafts, follow=(n_acc, bonus), logits_out=lo)
    for r in range(k + 1):
        err = float(np.max(np.abs(eng.logits(r) - lo[0][r])))
        assert err < LOGIT_TOL, ("verify logits", r, err)
    if (n_acc, bonus) != (cyc.n_accepted, cyc.bonus):
        assert cyc.gaps[min(n_acc, cyc.n_accepted)] < NEAR_TIE, (n_acc, bonus, cyc)
        near += 1
    assert eng.position() == (sess.t, sess.pending)
    return near


def check_dp(eng, sess, n):
    mask, val = eng.dp_select(n)
    o_mask, o_val, _ = clasp.dp_search(sess, n)
    assert len(mask) == n
    if mask != o_mask:
        got = clasp.cosine(clasp.skipped_state(sess, mask), sess.target.states[sess.cfg.n_layers])
        assert got >= o_val - 1e-3, (mask, o_mask, got, o_val)
    assert abs(val - o_val) < 2e-3, (val, o_val)


def test_llama3_8b_full_depth_against_oracle():
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = si.CONFIGS["llama3_8b"]
    prompt = si.prompt(cfg)
    eng = ssd.Engine(cfg, ssd.DeviceWeights(cfg))
    sess = decode.Session(oracle_weights(cfg))
    check_prefill(eng, sess, prompt, (len(prompt) - 1) % 64)
    check_dp(eng, sess, 16)
    near = 0
    for _ in range(2):
        near += check_cycle(eng, sess, cfg.skip, cfg.draft_k)
    # draft == target: nothing skipped, so every draft is accepted; the kept KV then serves the next pass
    t0 = sess.t
    drafts = eng.draft((), cfg.draft_k)
    n_acc, _, bonus = eng.verify([sess.pending] + drafts)
    assert n_acc == cfg.draft_k
    o = sess.draft_linear((), cfg.draft_k, force=drafts)
    cyc = sess.verify_linear(o, follow=(n_acc, bonus))
    assert cyc.n_accepted == cfg.draft_k or min(cyc.gaps) < NEAR_TIE
    assert eng.position() == (sess.t, sess.pending) == (t0 + cfg.draft_k + 1, bonus)
    for _ in range(3):
        got = eng.decode_ar(1)[0]
        want, row = sess.ar_step()
        if got != want:  # resynchronise on the oracle's token
            assert decode.model.top_gap(row) < NEAR_TIE
            near += 1
            eng.rollback(sess.t, want)
        assert float(np.max(np.abs(eng.logits(0) - row))) < LOGIT_TOL
    # int8 activations at d 4096 / F 14336, prefix-free: one layer run (shallow), the static draft's 16 (deep)
    n8, dev1, q1 = int8_prefix_free(eng, sess.Wt, prompt[0], tuple(i for i in range(cfg.n_layers) if i != 9), 2, True)
    near += n8
    _, dev16, q16 = int8_prefix_free(eng, sess.Wt, prompt[0], cfg.skip, 2, False)
    print(f"8B int8 logits deviation: one layer {dev1:.4f} (int8 effect {q1:.3f}); 16 layers {dev16:.4f} ({q16:.3f})")
    assert near <= 3, near
    assert eng.stats()["mma_fallbacks"] == 0
    del eng
    free()


@pytest.mark.parametrize("layers", [2])
def test_llama3_70b_shapes_against_oracle(layers):
    import self_speculative_decoding_layer_gb300 as ssd

    full = si.CONFIGS["llama3_70b_clasp"]
    cfg = full.replace(n_layers=layers, prompt_len=64, n_gen=32)
    prompt = si.prompt(cfg)
    eng = ssd.Engine(cfg, ssd.DeviceWeights(cfg))
    sess = decode.Session(oracle_weights(cfg))
    check_prefill(eng, sess, prompt, len(prompt) - 1)
    check_dp(eng, sess, 1)
    assert check_cycle(eng, sess, (1,), full.draft_k) <= 2
    del eng
    free()


@pytest.mark.parametrize("level_exit", [(), (2, 0, 0)])
def test_llama2_13b_shapes_cascade_against_oracle(level_exit):
    """(2, 0, 0): L1 also exits 2 layers early ([CAS-blog] §2.2)."""
    import self_speculative_decoding_layer_gb300 as ssd

    levels = (((0, 1, 2), False), ((1,), True), ((), True))
    cfg = si.CONFIGS["llama2_13b_cascade"].replace(n_layers=4, prompt_len=48, n_gen=32, levels=levels,
                                                   level_exit=level_exit)
    prompt = si.prompt(cfg)
    w = ssd.DeviceWeights(cfg)
    eng = ssd.Engine(cfg, w)
    W = oracle_weights(cfg)
    sess = decode.Session(W)
    check_prefill(eng, sess, prompt, len(prompt) - 1)
    near = 0
    # one teacher-forced tree cycle on the GPU's own tree: same plan, every expansion, every verify row
    toks, parents = eng.draft_tree(levels=levels, level_exit=level_exit)
    plan = decode.DyTC(cfg).plan(sess.t)
    assert parents == plan.parents and toks[0] == sess.pending
    near += tree_cycle_against_oracle(eng, sess, toks, parents, plan.expansions, levels, level_exit,
                                      int8_tokens=False)
    assert near <= 3, near
    # a whole DyTC generation (EMA updates included) recomputed cycle by cycle; lossless on the GPU
    e2 = ssd.Engine(cfg, w)
    e2.prefill(prompt)
    e2.set_option(ssd.OPT_CYCLE_LOG, 1)
    toks2 = e2.generate(24, ssd.POLICY_DYTC, levels=levels, level_exit=level_exit)
    e3 = ssd.Engine(cfg, w)
    e3.prefill(prompt)
    assert toks2 == e3.generate(24, ssd.POLICY_AR)
    f = Follow(W, prompt, toks2[0], int8_tokens=False)
    dy = decode.DyTC(cfg)
    for e in e2.cycle_log():
        f.dytc(e, dy)
    assert f.near <= 3, f.near
    # int8 activations with fp16 weights at d 5120 / F 13824, prefix-free: one layer run, levels L2 and L3
    int8_prefix_free(eng, W, prompt[0], (0, 1, 3), 2, True)
    for l in (1, 2):
        int8_prefix_free(eng, W, prompt[0], levels[l][0], 2, False)
    del eng, e2, e3, w
    free()


def test_llama3_70b_full_size_properties():
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = si.CONFIGS["llama3_70b_clasp"]
    prompt = si.prompt(cfg, 256)
    w = ssd.DeviceWeights(cfg)
    eng = ssd.Engine(cfg, w)
    eng.prefill(prompt)
    mask0, val0 = eng.dp_select(0)  # n = 0: the full model reproduces its own target
    assert mask0 == () and abs(val0 - 1.0) < 1e-4
    t0, p0 = eng.position()
    ar = eng.generate(24, ssd.POLICY_AR)
    eng.rollback(t0, p0)
    sp = eng.generate(24, ssd.POLICY_CLASP, dp_n_skip=44, dp_interval=2, k=cfg.draft_k, dp_at_start=False)
    assert sp == ar
    st = eng.stats()
    assert st["dp_runs"] >= 1 and st["mma_fallbacks"] == 0
    del eng, w
    free()


def test_llama2_13b_full_size_tree_is_lossless():
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = si.CONFIGS["llama2_13b_cascade"]
    prompt = si.prompt(cfg)
    w = ssd.DeviceWeights(cfg)
    eng = ssd.Engine(cfg, w)
    eng.prefill(prompt)
    t0, p0 = eng.position()
    ar = eng.generate(24, ssd.POLICY_AR)
    eng.rollback(t0, p0)
    tr = eng.generate(24, ssd.POLICY_DYTC)
    assert tr == ar
    assert eng.stats()["cycles"] > 0
    del eng, w
    free()
