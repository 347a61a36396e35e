"""Pins of the CPU oracle against things other than itself: hand-worked values,
closed forms, library routines, brute force and the method's exact invariants."""
import math
import os

import numpy as np
import pytest

import ssd_inputs as si
from oracle import clasp, decode, latency, model, quant
from oracle.model import ArrayWeights, KVCache, Weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                out.append(line.split())
    return out


def hand_cfg(**kw):
    base = dict(name="hand", n_layers=1, d_model=2, n_q_heads=1, n_kv_heads=1, head_dim=2, ffn=1, vocab=3,
                rms_eps=0.0, prompt_len=3, n_gen=1)
    base.update(kw)
    return si.ModelConfig(**base)


def zero_layer(cfg):
    d, hd, F = cfg.d_model, cfg.head_dim, cfg.ffn
    return dict(wq=np.zeros((cfg.n_q_heads * hd, d)), wk=np.zeros((cfg.n_kv_heads * hd, d)),
                wv=np.zeros((cfg.n_kv_heads * hd, d)), wo=np.zeros((d, cfg.n_q_heads * hd)),
                wg=np.zeros((F, d)), wu=np.zeros((F, d)), wd=np.zeros((d, F)), g_attn=np.ones(d), g_ffn=np.ones(d))


# ---------------------------------------------------------------- model pieces


def test_rmsnorm_closed_form():
    x = np.array([[3.0, 4.0], [-2.0, -2.0]])
    g = np.array([1.0, 0.5])
    y = model.rmsnorm(x, g, 1e-5)
    assert np.allclose(y[0], np.array([3.0, 4.0]) / math.sqrt(12.5 + 1e-5) * g, rtol=0, atol=1e-15)
    assert np.allclose(y[1], np.array([-1.0, -0.5]) / math.sqrt(1.0 + 1e-5 / 4.0), rtol=0, atol=1e-15)


def test_silu_closed_forms():
    assert model.silu(np.array([0.0]))[0] == 0.0
    assert model.silu(np.array([1.0]))[0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), abs=1e-15)
    assert model.silu(np.array([40.0]))[0] == pytest.approx(40.0, abs=1e-12)
    assert abs(model.silu(np.array([-40.0]))[0]) < 1e-15


def test_rope_hand_values():
    for row in _rows("rope_hd4.txt"):
        v = [float(x) for x in row]
        pos, x, want = int(v[0]), np.array(v[1:5]), np.array(v[5:9])
        y = model.rope(x.reshape(1, 1, 4), np.array([pos]), 10000.0).reshape(4)
        assert np.allclose(y, want, atol=1e-14), (pos, y, want)


def test_rope_relative_position_and_norm():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    d = []
    for m, n in [(5, 2), (103, 100), (2003, 2000)]:
        qm = model.rope(q, np.array([m]), 10000.0)
        kn = model.rope(k, np.array([n]), 10000.0)
        assert np.linalg.norm(qm) == pytest.approx(np.linalg.norm(q), rel=1e-13)
        d.append(float(np.sum(qm * kn)))
    assert d[0] == pytest.approx(d[1], rel=1e-9) and d[0] == pytest.approx(d[2], rel=1e-9)


def test_attention_matches_library_sdpa_with_gqa():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    R, S, Hq, Hkv, hd = 5, 11, 8, 2, 16
    q = rng.standard_normal((R, Hq, hd))
    k = rng.standard_normal((S, Hkv, hd))
    v = rng.standard_normal((S, Hkv, hd))
    vis = rng.random((R, S)) < 0.6
    vis[:, 0] = True
    o = model.attention(q, k, v, vis)
    tq = torch.tensor(q).permute(1, 0, 2)  # [Hq, R, hd]
    tk = torch.tensor(k).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
    tv = torch.tensor(v).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(vis))
    assert np.allclose(o, ref.permute(1, 0, 2).numpy(), atol=1e-12)


def test_identity_layers_give_norm_embedding_logits():
    cfg = hand_cfg(d_model=4, vocab=4, n_layers=2, head_dim=4, ffn=2)
    E = 2.0 * np.eye(4)
    W = ArrayWeights(cfg, E, E, np.ones(4), [zero_layer(cfg), zero_layer(cfg)])
    logits, states = model.forward(W, KVCache(cfg, 8), [2], [0], [0], model.causal_vis(0, 1))
    want = np.zeros(4)
    want[2] = 4.0  # e_2 . (e_2 / rms(e_2)), rms(2 e_2) = sqrt(4/4)
    assert np.allclose(logits[0], want, atol=1e-15)
    assert all(np.array_equal(s, states[0]) for s in states)


def test_early_exit_at_zero_layers_left_gives_norm_embedding_logits():
    """Exiting before every layer: the lm_head reads the embedding through the final norm,
    whatever the layers would have done (here they are far from identity)."""
    cfg = hand_cfg(d_model=4, vocab=4, n_layers=2, head_dim=4, ffn=2)
    E = 2.0 * np.eye(4)
    busy = zero_layer(cfg)
    busy["wg"] = np.ones((2, 4))
    busy["wu"] = np.ones((2, 4))
    busy["wd"] = np.ones((4, 2))
    W = ArrayWeights(cfg, E, E, np.ones(4), [busy, busy])
    logits, states = model.forward(W, KVCache(cfg, 8), [2], [0], [0], model.causal_vis(0, 1), exit_layers=2)
    want = np.zeros(4)
    want[2] = 4.0
    assert np.allclose(logits[0], want, atol=1e-15)
    full, _ = model.forward(W, KVCache(cfg, 8), [2], [0], [0], model.causal_vis(0, 1))
    assert not np.allclose(full[0], want)  # the layers do change the result when they run


def test_uniform_attention_averages_values_causally():
    cfg = hand_cfg()
    lay = zero_layer(cfg)
    lay["wv"] = np.eye(2)
    lay["wo"] = np.eye(2)  # q = 0 -> uniform attention; FFN zero
    lay["wk"] = np.array([[0.3, -1.0], [2.0, 0.5]])
    E = np.array([[1.0, 1.0], [3.0, -1.0], [-2.0, 2.0]])
    W = ArrayWeights(cfg, E, np.eye(3, 2), np.ones(2), [lay])
    _, states = model.forward(W, KVCache(cfg, 4), [0, 1, 2], [0, 1, 2], [0, 1, 2], model.causal_vis(0, 3))
    a = [np.array([1.0, 1.0]), np.array([3.0, -1.0]) / math.sqrt(5.0), np.array([-1.0, 1.0])]
    want = [E[0] + a[0], E[1] + (a[0] + a[1]) / 2, E[2] + (a[0] + a[1] + a[2]) / 3]
    assert np.allclose(states[1], np.array(want), atol=1e-14)


def test_ffn_gate_up_down_by_hand():
    cfg = hand_cfg()
    lay = zero_layer(cfg)
    lay["wg"] = np.array([[1.0, 0.0]])
    lay["wu"] = np.array([[0.0, 1.0]])
    lay["wd"] = np.array([[1.0], [0.0]])
    lay["g_ffn"] = np.array([1.0, 2.0])
    E = np.array([[3.0, 4.0], [0.0, 1.0], [1.0, 0.0]])
    W = ArrayWeights(cfg, E, np.eye(3, 2), np.ones(2), [lay])
    _, states = model.forward(W, KVCache(cfg, 2), [0], [0], [0], model.causal_vis(0, 1))
    b0, b1 = 3.0 / math.sqrt(12.5), 2.0 * 4.0 / math.sqrt(12.5)
    gate = b0 / (1.0 + math.exp(-b0))
    assert np.allclose(states[1][0], [3.0 + gate * b1, 4.0], atol=1e-14)


def test_sharp_attention_retrieves_matching_position():
    """RoPE'd q.k is largest at equal offsets: a row whose query equals a key's
    content attends (sharply) to the key at its own relative offset 0."""
    cfg = hand_cfg(d_model=4, head_dim=4, vocab=4, ffn=1)
    lay = zero_layer(cfg)
    lay["wq"] = 60.0 * np.eye(4)
    lay["wk"] = 60.0 * np.eye(4)
    lay["wv"] = np.eye(4)
    lay["wo"] = np.eye(4)
    E = np.eye(4)
    W = ArrayWeights(cfg, E, np.eye(4), np.ones(4), [lay])
    _, st = model.forward(W, KVCache(cfg, 4), [1, 2, 1], [0, 1, 2], [0, 1, 2], model.causal_vis(0, 3))
    # row 2 (token 1) matches itself far more than token 1 at distance 2 or token 2
    delta = st[1][2] - st[0][2]
    assert delta[1] > 0.9 * np.max(np.abs(delta)) and np.argmax(delta) == 1


def test_argmax_and_top2_ties_go_to_lower_id():
    x = np.array([0.5, 2.0, 2.0, 1.0, 2.0])
    assert model.argmax_f32(x) == 1
    assert model.top2_f32(x) == (1, 2)
    assert model.top_gap(np.array([1.0, 3.0, 2.5])) == pytest.approx(0.5)


def test_top1_prob_closed_forms_and_library():
    from scipy.special import logsumexp

    assert model.top1_prob(np.zeros(1024)) == pytest.approx(1.0 / 1024, rel=1e-12)
    # two tied maxima, the rest exp(-1000) = 0 in float64
    assert model.top1_prob(np.array([-1000.0, 3.0, 3.0, -1000.0])) == pytest.approx(0.5, rel=1e-12)
    # exp(ln 3) / (1 + exp(ln 3)) = 3/4 (logits rounded to float32 first)
    x = np.array([0.0, math.log(3.0)], dtype=np.float32)
    assert model.top1_prob(x) == pytest.approx(1.0 / (1.0 + math.exp(-float(x[1]))), rel=1e-12)
    # large offsets must not overflow: the probability is shift invariant
    rng = np.random.default_rng(3)
    for _ in range(5):
        v = rng.normal(0.0, 3.0, 777).astype(np.float32)
        ref = math.exp(float(v.max()) - logsumexp(v.astype(np.float64)))
        assert model.top1_prob(v) == pytest.approx(ref, rel=1e-12)
        assert model.top1_prob(v + np.float32(4096.0)) == pytest.approx(
            math.exp(float((v + np.float32(4096.0)).max()) - logsumexp((v + np.float32(4096.0)).astype(np.float64))),
            rel=1e-12)


# ---------------------------------------------------------------- int8


def test_int8_golden_codes():
    rows = {r[0]: r[1:] for r in _rows("int8_codes.txt")}
    x = np.array([float(v) for v in rows["x"]])
    codes, scale = quant.quantize_rows(x)
    assert codes[0].tolist() == [int(v) for v in rows["q"]]
    assert scale[0] == np.float32(float(rows["scale"][0]))


def test_int8_error_bound_and_range():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 999)) * rng.uniform(0.01, 10, size=(7, 1))
    codes, scale = quant.quantize_rows(x)
    assert codes.min() >= -127 and codes.max() <= 127
    assert np.all(np.max(np.abs(codes), axis=1) == 127)
    xh = quant.fake_quant_rows(x)
    assert np.all(np.abs(x - xh) <= scale[:, None].astype(np.float64) * (0.5 + 1e-6) + 1e-7 * np.abs(x))


def test_int8_zero_row():
    x = np.zeros((2, 5))
    x[1, 3] = -4.0
    xh = quant.fake_quant_rows(x)
    assert np.all(xh[0] == 0.0) and xh[1, 3] == -127.0 * float(np.float32(np.float32(4.0) / np.float32(127.0)))
    assert np.all(np.delete(xh[1], 3) == 0.0)


# ---------------------------------------------------------------- cache + decoding invariants


@pytest.fixture(scope="module")
def tiny():
    return Weights(si.CONFIGS["tiny"])


@pytest.fixture(scope="module")
def tiny_gqa():
    return Weights(si.CONFIGS["tiny"].replace(name="tiny_gqa", n_kv_heads=2, gamma_sigma=0.1))


def test_prefill_equals_incremental(tiny_gqa):
    cfg = tiny_gqa.cfg
    p = si.prompt(cfg, 12)
    a = decode.Session(tiny_gqa, 64)
    _, la = a.prefill(p)
    b = decode.Session(tiny_gqa, 64)
    b.prefill(p[:5])
    for tok in p[5:]:
        _, lb = b.prefill([tok])
    assert np.allclose(la[-1], lb[-1], atol=1e-11)
    for i in range(cfg.n_layers):
        assert np.allclose(a.cache.k[i][:12], b.cache.k[i][:12], atol=1e-12)


def test_rollback_equals_fresh_cache(tiny):
    p = si.prompt(tiny.cfg, 30)
    a = decode.Session(tiny, 64)
    a.prefill(p[:20])
    a.prefill(p[20:30])
    a.rollback(20)
    _, la = a.prefill(p[20:25])
    b = decode.Session(tiny, 64)
    _, lb = b.prefill(p[:25])
    assert np.allclose(la[-1], lb[-1], atol=1e-11)


def test_spec_equals_autoregressive(tiny):
    cfg = tiny.cfg
    p = si.prompt(cfg)
    ar = decode.generate_ar(tiny, p, cfg.n_gen)
    sp = decode.generate_spec(tiny, p, cfg.n_gen)
    assert sp.tokens == ar
    assert sum(c.n_accepted + 1 for c in sp.cycles) + 1 >= cfg.n_gen


def test_spec_int8_and_gqa_equal_autoregressive(tiny_gqa):
    p = si.prompt(tiny_gqa.cfg, 20)
    ar = decode.generate_ar(tiny_gqa, p, 30)
    assert decode.generate_spec(tiny_gqa, p, 30, skip=(0, 3), k=3, act_int8=True).tokens == ar
    assert decode.generate_spec(tiny_gqa, p, 30, skip=(0, 1, 2, 3), k=5).tokens == ar


def test_draft_equal_target_accepts_everything(tiny):
    p = si.prompt(tiny.cfg)
    sp = decode.generate_spec(tiny, p, 40, skip=(), k=4)
    assert all(c.n_accepted == 4 for c in sp.cycles)


def _softmax_max(row):
    from scipy.special import softmax

    return float(softmax(np.asarray(row).astype(np.float32).astype(np.float64)).max())


def test_draft_exit_stops_after_first_low_confidence_draft(tiny):
    """[CLaSp] §四 draft exit: drafting ends with the first draft whose top-1 softmax
    probability is below the threshold; that draft is the last one kept."""
    cfg = tiny.cfg
    K, skip = 6, (0, 3)
    s = decode.Session(tiny)
    s.prefill(si.prompt(cfg))
    lengths = set()
    for cyc in range(6):
        rows = []
        full = s.draft_linear(skip, K, rows=rows)
        p = [_softmax_max(r) for r in rows]
        q = np.sort(p)
        thr = 0.5 * (q[cyc % (K - 1)] + q[cyc % (K - 1) + 1])  # the 1 + cyc % 5 least confident drafts fall below
        expect = next((r + 1 for r in range(K) if p[r] < thr), K)
        got = s.draft_linear(skip, K, exit_thr=thr)
        assert got == full[:expect], (cyc, p, thr)
        lengths.add(len(got))
        assert s.draft_linear(skip, K, exit_thr=0.0) == full
        assert s.draft_linear(skip, K, exit_thr=1.5) == full[:1]
        s.verify_linear(full[:expect])
    assert len(lengths) >= 2, lengths  # the thresholds really cut the drafts at different depths


def test_draft_exit_generation_equals_autoregressive(tiny):
    cfg = tiny.cfg
    p = si.prompt(cfg)
    ar = decode.generate_ar(tiny, p, cfg.n_gen)
    probe = decode.Session(tiny)
    probe.prefill(p)
    probs = []
    probe.draft_linear((0, 3), 8, probs=probs)
    thr = float(np.median(probs))
    sp = decode.generate_spec(tiny, p, cfg.n_gen, skip=(0, 3), k=6, exit_thr=thr)
    assert sp.tokens == ar
    n = [len(c.drafts) for c in sp.cycles]
    assert min(n) >= 1 and max(n) <= 6 and len(set(n)) >= 2, n
    # a threshold above 1 keeps exactly one draft per cycle: the same cycles as draft length 1
    one = decode.generate_spec(tiny, p, 24, k=6, exit_thr=1.5)
    k1 = decode.generate_spec(tiny, p, 24, k=1)
    assert one.tokens == k1.tokens == ar[:24]
    assert [(c.drafts, c.n_accepted, c.bonus) for c in one.cycles] == [(c.drafts, c.n_accepted, c.bonus)
                                                                       for c in k1.cycles]


def test_early_exit_equals_skipping_the_last_layers(tiny):
    """[CAS-blog] §2.1 item 2: an early exit after layer L-e-1 gives the same logits as running
    the model with the last e layers bypassed, and leaves those layers' KV slots unwritten."""
    cfg = tiny.cfg
    p = si.prompt(cfg, 16)
    for e, skip in ((1, ()), (2, (0,)), (3, ())):
        a = decode.Session(tiny, 64)
        b = decode.Session(tiny, 64)
        a.prefill(p)
        b.prefill(p)
        for L_ in range(cfg.n_layers):
            a.cache.k[L_][16:] = 7.0
        la, _ = model.forward(tiny, a.cache, [5], [16], [16], model.causal_vis(16, 1), skip=skip, exit_layers=e)
        lb, _ = model.forward(tiny, b.cache, [5], [16], [16], model.causal_vis(16, 1),
                              skip=tuple(skip) + tuple(range(cfg.n_layers - e, cfg.n_layers)))
        assert np.allclose(la, lb, atol=1e-12)
        for L_ in range(cfg.n_layers - e, cfg.n_layers):
            assert np.all(a.cache.k[L_][16] == 7.0)
        for L_ in set(range(cfg.n_layers - e)) - set(skip):
            assert not np.all(a.cache.k[L_][16] == 7.0)


def test_early_exit_drafts_are_lossless(tiny):
    cfg = tiny.cfg
    p = si.prompt(cfg)
    ar = decode.generate_ar(tiny, p, 40)
    sp = decode.generate_spec(tiny, p, 40, skip=(1,), k=4, early_exit=2)
    assert sp.tokens == ar
    cyc = decode.Session(tiny)
    cyc.prefill(p)
    ref = decode.Session(tiny)
    ref.prefill(p)
    assert cyc.draft_linear((1,), 4, exit_layers=2) == ref.draft_linear((1, 2, 3), 4)


def test_cascade_levels_with_early_exit():
    """L1 of the cascade with a 4-layer early exit ([CAS-blog] §2.2): 70 % of the first L-4
    layers skipped, nested around L2's skips, and the exit layers outside its skip set."""
    lv0 = si.cascade_levels(40)
    assert lv0 == si.CONFIGS["llama2_13b_cascade"].levels
    assert len(lv0[0][0]) == 28 and len(lv0[1][0]) == 12
    lv = si.cascade_levels(40, 4)
    l1, l2 = set(lv[0][0]), set(lv[1][0])
    assert len(l1) == round(0.7 * 36) and max(l1) < 36
    assert {i for i in l2 if i < 36} <= l1
    assert lv[1:] == lv0[1:]
    cfg = si.CONFIGS["llama2_13b_cascade"].replace(levels=lv, level_exit=(4, 0, 0))
    c = decode.level_costs(cfg)
    n_run = 40 - 25 - 4
    assert c[0] * 25703219200 == pytest.approx(n_run * 634388480 + 327680000, rel=1e-14)


def test_tree_generation_with_early_exit_level_is_lossless():
    cfg = si.CONFIGS["tiny"].replace(name="tiny_cascade_exit", tree=True,
                                     levels=(((1,), False), ((1,), True), ((), True)), level_exit=(2, 0, 0))
    W = Weights(cfg)
    p = si.prompt(cfg)
    ar = decode.generate_ar(W, p, 40)
    toks, recs = decode.generate_tree(W, p, 40)
    assert toks == ar
    assert any(len(r[0].parents) > 2 for r in recs)


def test_chain_tree_equals_linear(tiny):
    p = si.prompt(tiny.cfg)
    a = decode.Session(tiny, 128)
    a.prefill(p)
    b = decode.Session(tiny, 128)
    b.prefill(p)
    drafts = a.draft_linear((1, 2), 4)
    b.draft_linear((1, 2), 4)
    ca = a.verify_linear(drafts)
    cb = b.verify_tree([b.pending] + drafts, [-1, 0, 1, 2, 3])
    assert ca.argmax == cb.argmax and ca.n_accepted == cb.n_accepted and ca.bonus == cb.bonus
    assert np.allclose(a.cache.k[0][: a.t], b.cache.k[0][: b.t], atol=1e-12)


def test_tree_generation_equals_autoregressive():
    cfg = si.CONFIGS["tiny"].replace(name="tiny_cascade", tree=True,
                                     levels=(((0, 1, 2), False), ((1,), True), ((), True)))
    W = Weights(cfg)
    p = si.prompt(cfg)
    ar = decode.generate_ar(W, p, 40)
    toks, recs = decode.generate_tree(W, p, 40)
    assert toks == ar
    assert any(len(r[0].parents) > 2 for r in recs)


def test_tree_compaction_moves_accepted_branch(tiny):
    """Accept along a non-first branch: its KV must end up in the contiguous slots."""
    p = si.prompt(tiny.cfg)
    s = decode.Session(tiny, 128)
    s.prefill(p)
    t = s.t
    ref = decode.Session(tiny, 128)
    ref.prefill(p)
    la, _ = ref.ar_step()
    # node 1 = a wrong token, node 2 = the true continuation (sibling), node 3 child of 2
    wrong = (la + 1) % tiny.cfg.vocab
    lb, _ = ref.ar_step()
    ref.ar_step()  # runs lb in slot t + 2
    cyc = s.verify_tree([s.pending, wrong, la, lb], [-1, 0, 0, 2])
    assert cyc.path[:3] == [0, 2, 3] and cyc.n_accepted >= 2
    assert np.allclose(s.cache.k[1][t + 1], ref.cache.k[1][t + 1], atol=1e-12)
    assert np.allclose(s.cache.k[3][t + 2], ref.cache.k[3][t + 2], atol=1e-12)


# ---------------------------------------------------------------- DyTC


def test_dytc_plan_hand_worked():
    """gain/c at a = 0.65 with the 13B level costs, worked by hand: root at L1
    (2.8405 > 1), node 1 at L1 (1.8463 > E/T = 1.4344), then the best score
    1.2001 (node 3) falls below E/T = 1.5130 and planning stops."""
    cfg = si.CONFIGS["llama2_13b_cascade"]
    c = decode.level_costs(cfg)
    assert c[0] == pytest.approx(7940341760 / 25703219200, rel=1e-15)
    assert c[1] == pytest.approx(18090557440 / 25703219200, rel=1e-15)
    assert c[2] == 1.0
    plan = decode.DyTC(cfg).plan()
    assert plan.parents == [-1, 0, 0, 1, 1]
    assert plan.expansions == [(0, 0), (1, 0)]
    assert plan.prob == pytest.approx([1.0, 0.65, 0.2275, 0.4225, 0.147875])


def test_dytc_respects_budget_depth_and_caps():
    cfg = si.CONFIGS["llama2_13b_cascade"]
    d = decode.DyTC(cfg)
    d.a = [0.99, 0.99, 0.99]
    plan = d.plan()
    assert len(plan.parents) - 1 <= cfg.tree_max_nodes and max(plan.depth) <= cfg.tree_max_depth
    lvl = dict(plan.expansions)
    for u, l in plan.expansions:
        par = plan.parents[u]
        if par >= 0:
            assert l <= lvl[par]
    assert all(plan.parents[c] < c for c in range(1, len(plan.parents)))


def test_cascade_depth_rule_hand_values():
    """[CAS-blog] §4.1 item 1 and §4.2 problem 3, worked by hand: log2(40/12) = 1.74 -> 1,
    log2(80/12) = 2.74 -> 2, log2(96/12) = 3 -> 3, log2(200/12) > 3 -> 3; seq_len > 512 drops one."""
    cd = latency.cascade_depth
    assert [cd(40, 3, 256), cd(80, 3, 100), cd(80, 3, 600), cd(96, 3, 512), cd(96, 3, 513)] == [1, 2, 1, 3, 2]
    assert [cd(200, 3, 0), cd(32, 3, 0), cd(24, 3, 0), cd(47, 3, 0), cd(48, 3, 0), cd(10, 3, 0)] == [3, 1, 1, 1, 2, 1]
    assert [cd(96, 2, 0), cd(96, 1, 0), cd(24, 3, 600)] == [2, 1, 1]


def test_latency_fit_exact_and_normal_equations():
    """Noise-free points of a known model give it back; on noisy points the residual is
    orthogonal to (1, s, d) (the least-squares condition); a 3-point system by Cramer's rule."""
    s = np.array([128, 256, 512, 1024] * 3, dtype=float)
    d = np.repeat([8.0, 16.0, 32.0], 4)
    beta = np.array([0.21, 3e-5, 0.061])
    y = beta[0] + beta[1] * s + beta[2] * d
    assert np.allclose(latency.fit_latency(s, d, y), beta, rtol=1e-10, atol=1e-13)
    rng = np.random.default_rng(5)
    yn = y + rng.normal(0, 0.01, y.size)
    b = latency.fit_latency(s, d, yn)
    r = yn - (b[0] + b[1] * s + b[2] * d)
    assert abs(r.sum()) < 1e-10 and abs((r * s).sum()) < 1e-7 and abs((r * d).sum()) < 1e-9
    S, D, Y = [100.0, 300.0, 100.0], [4.0, 4.0, 10.0], [1.0, 1.5, 2.2]
    b = latency.fit_latency(S, D, Y)
    # by hand: b1 = (1.5 - 1.0) / 200, b2 = (2.2 - 1.0) / 6, b0 = 1.0 - 100 b1 - 4 b2
    assert np.allclose(b, [1.0 - 100 * 0.0025 - 4 * 0.2, 0.0025, 0.2], rtol=1e-12)
    with pytest.raises(ValueError):
        latency.fit_latency([100, 100, 100, 100], [1, 2, 3, 4], [1, 2, 3, 4])


def test_dytc_latency_model_costs_and_depth_rule():
    """Costs from latency models (16-bit, int8), worked by hand for the 13B cascade; the depth
    rule keeps only L1 on 40 layers (log2(40/12) < 2)."""
    cfg = si.CONFIGS["llama2_13b_cascade"]
    b16, b8 = (1.0, 0.001, 0.1), (1.0, 0.001, 0.05)
    d = decode.DyTC(cfg, betas=(b16, b8))
    d.plan(200)
    full = 1.0 + 0.2 + 4.0
    assert d.c == pytest.approx([(1.2 + 0.1 * 12) / full, (1.2 + 0.05 * 28) / full, (1.2 + 0.05 * 40) / full],
                                rel=1e-15)
    r = decode.DyTC(cfg, rules=True)
    r.a = [0.99, 0.99, 0.99]
    plan = r.plan(100)
    assert plan.expansions and all(l == 0 for _, l in plan.expansions)
    deep = cfg.replace(n_layers=80, levels=si.cascade_levels(80))
    r2 = decode.DyTC(deep, rules=True)
    r2.a = [0.05, 0.99, 0.99]  # L1 is poor: the planner wants L2 or L3 where it may use them
    assert any(l == 1 for _, l in r2.plan(100).expansions)  # 2 levels on 80 layers
    assert all(l == 0 for _, l in r2.plan(600).expansions)  # past 512: one level fewer
    free = decode.DyTC(deep)
    free.a = r2.a
    assert any(l >= 1 for _, l in free.plan(600).expansions)  # without the rule L2 is still used


def test_hcascade_chain_layout():
    """Highest level first: lens (L1, L2, L3) = (2, 1, 3) gives L3 L3 L3 L2 L1 L1 along one chain."""
    parents, levels = decode.hcascade_chain([2, 1, 3])
    assert parents == [-1, 0, 1, 2, 3, 4, 5]
    assert levels == [2, 2, 2, 1, 0, 0]
    assert decode.hcascade_chain([0, 0, 1]) == ([-1, 0], [2])


def test_hcascade_single_level_equals_linear_drafts():
    """A one-level horizontal cascade is a linear draft at that level: the same drafts, acceptance and
    output as the linear cycle, and lossless."""
    levels = (((1, 2), False), ((1,), True), ((), True))
    cfg = si.CONFIGS["tiny"].replace(name="tiny_hc", tree=True, levels=levels)
    W = Weights(cfg)
    p = si.prompt(cfg)
    toks, cycles = decode.generate_hcascade(W, p, 30, [4, 0, 0])
    lin = decode.generate_spec(W, p, 30, skip=(1, 2), k=4)
    assert toks == lin.tokens == decode.generate_ar(W, p, 30)
    assert [(c.drafts, c.n_accepted, c.bonus) for c in cycles] == [(c.drafts, c.n_accepted, c.bonus)
                                                                   for c in lin.cycles]
    mixed, cyc2 = decode.generate_hcascade(W, p, 30, [2, 1, 1])
    assert mixed == toks
    assert all(len(c.drafts) == 4 for c in cyc2)


def test_vcascade_invariants():
    """Vertical cascade: lossless; when the higher level is the target itself its chain is the
    target's own greedy continuation, so the target accepts all of it; when both levels are the same
    model the higher level keeps every lower-level draft."""
    levels = (((0, 1, 2), False), ((1,), True), ((), False))
    cfg = si.CONFIGS["tiny"].replace(name="tiny_vc", tree=True, levels=levels)
    W = Weights(cfg)
    p = si.prompt(cfg)
    ar = decode.generate_ar(W, p, 40)
    toks, cycles = decode.generate_vcascade(W, p, 40, 0, 1, 4)
    assert toks == ar
    toks2, cyc2 = decode.generate_vcascade(W, p, 40, 0, 2, 4)
    assert toks2 == ar
    assert all(c.n_accepted == len(c.drafts) for c in cyc2)
    assert all(1 <= len(c.drafts) <= 4 for c in cyc2)
    same = cfg.replace(levels=(((1, 2), False), ((1, 2), False), ((), False)))
    toks3, cyc3 = decode.generate_vcascade(Weights(same), p, 30, 0, 1, 4)
    assert toks3 == ar[:30]
    lin = decode.generate_spec(Weights(same), p, 30, skip=(1, 2), k=4)
    assert [(c.drafts, c.n_accepted) for c in cyc3] == [(c.drafts, c.n_accepted) for c in lin.cycles]


def test_ema_closed_form():
    cfg = si.CONFIGS["llama2_13b_cascade"]
    d = decode.DyTC(cfg)
    plan = decode.TreePlan([-1, 0, 0], [0, 1, 1], [1, .5, .5], [2, 0, 0], [(0, 0)])
    rates = [1, 0, 0, 1, 1]
    for r in rates:
        toks = [5, 7, 8]
        am = [7 if r else 9, 0, 0]
        d.update(plan, toks, decode.Cycle([7, 8], am, [1, 1, 1], 1 if r else 0, 0, [0, 1] if r else [0]))
    want = 0.65 * 0.8 ** 5 + sum(0.2 * 0.8 ** (len(rates) - 1 - k) * r for k, r in enumerate(rates))
    assert d.a[0] == pytest.approx(want, rel=1e-14)
    assert d.a[1] == 0.65 and d.a[2] == 0.65


# ---------------------------------------------------------------- CLaSp DP


@pytest.mark.parametrize("L", [4, 6, 8])
def test_dp_against_brute_force(L):
    cfg = si.CONFIGS["tiny"].replace(name=f"tiny{L}", n_layers=L)
    W = Weights(cfg)
    s = decode.Session(W, 64)
    s.prefill(si.prompt(cfg, 16))
    agree = 0
    for n in range(1, L // 2 + 1):
        sk, val, _ = clasp.dp_search(s, n)
        assert len(sk) == n
        bs, bv, vals = clasp.brute_force(s, n)
        assert val <= bv + 1e-12
        assert clasp.cosine(clasp.skipped_state(s, sk), s.target.states[L]) == pytest.approx(val, abs=1e-12)
        top = sorted(vals.values())[::-1]
        if sk == bs:
            agree += 1
        else:  # a miss is allowed only where the optimum is nearly tied
            assert top[0] - top[1] < 1e-3 or bv - val < 1e-3
    assert agree >= 1


def test_dp_n0_keeps_all_layers(tiny):
    s = decode.Session(tiny, 64)
    s.prefill(si.prompt(tiny.cfg, 16))
    sk, val, _ = clasp.dp_search(s, 0)
    assert sk == () and val == pytest.approx(1.0, abs=1e-12)


def test_dp_all_skipped(tiny):
    s = decode.Session(tiny, 64)
    s.prefill(si.prompt(tiny.cfg, 16))
    L = tiny.cfg.n_layers
    sk, val, _ = clasp.dp_search(s, L)
    assert sk == tuple(range(L))
    assert val == pytest.approx(clasp.cosine(s.target.states[0], s.target.states[L]), abs=1e-14)


def test_dp_refresh_generation_equals_autoregressive(tiny):
    p = si.prompt(tiny.cfg)
    ar = decode.generate_ar(tiny, p, 40)
    sp = decode.generate_spec(tiny, p, 40, dp_n_skip=2, dp_interval=3)
    assert sp.tokens == ar and len(sp.masks) > 2


def test_dp_tie_keeps():
    """Identity layers make every candidate equal to the embedding, so every
    comparison is an exact tie; a tie keeps, so the one skip lands on layer 0
    (the only (1, 1) state) and layer 1 is kept."""
    cfg = hand_cfg(d_model=4, vocab=4, n_layers=2, head_dim=4, ffn=2)
    E = np.eye(4) + 0.5
    W = ArrayWeights(cfg, E, E, np.ones(4), [zero_layer(cfg), zero_layer(cfg)])
    s = decode.Session(W, 8)
    s.prefill([1, 2, 3])
    sk, val, table = clasp.dp_search(s, 1)
    assert sk == (0,) and val == pytest.approx(1.0, abs=1e-15)
    assert table[2][1][1] == "keep"


# ---------------------------------------------------------------- branching trees against fresh prefills


def _fresh_logits(W, prompt, path_tokens):
    """Logits after prompt + path_tokens, by a fresh causal prefill of the whole sequence."""
    s = decode.Session(W, 128)
    _, logits = s.prefill(list(prompt) + list(path_tokens))
    return logits[-1]


def _branching_tree():
    # root 0; 1, 2 its rank-0/rank-1 children; 3, 4 under 1; 5, 6 under 2; 7 under 5
    return [-1, 0, 0, 1, 1, 2, 2, 5]


def _path(tokens, parents, c):
    out = []
    while c >= 0:
        out.append(tokens[c])
        c = parents[c]
    return out[::-1]


def test_branching_draft_nodes_equal_fresh_prefills(tiny):
    """A tree expanded with the full model as its draft level (nothing skipped, no int8): every
    expansion's logits must equal those of its own root-to-node token path computed by a fresh
    causal prefill of prompt + path -- a different code path (causal visibility, contiguous
    slots) from the tree expansion (node c in slot t + c at position t + depth(c), seeing the
    prefix and its ancestors).  The tree branches at the root and at nodes 1, 2 and 5, so a
    slot/position mix-up (e.g. position t + c) or a wrong ancestor mask changes some row; the
    children are the (top-1, top-2) of each expansion, and the rank-0 spine is greedy decoding."""
    p = si.prompt(tiny.cfg, 24)
    parents = _branching_tree()
    depth = decode.tree_depths(parents)
    s = decode.Session(tiny, 128)
    s.prefill(p)
    tokens = [s.pending] + [0] * (len(parents) - 1)
    kids = {}
    for c in range(1, len(parents)):
        kids.setdefault(parents[c], []).append(c)
    for u in (0, 1, 2, 5):  # parents before children
        rows = []
        top = s.draft_node(u, parents, depth, tokens[u], (), False, rows=rows)
        fresh = _fresh_logits(tiny, p, _path(tokens, parents, u))
        assert np.allclose(rows[0], fresh, rtol=0, atol=1e-9), (u, float(np.max(np.abs(rows[0] - fresh))))
        assert top == model.top2_f32(fresh)
        for r, c in enumerate(kids[u]):
            tokens[c] = top[r]
    ar = decode.generate_ar(tiny, p, 4)
    assert [tokens[0], tokens[1], tokens[3]] == ar[:3]


def test_branching_tree_verify_equals_fresh_prefills(tiny):
    """Tree verification over the same branching tree: each node's logits row equals the fresh
    causal prefill of its root-to-node path, and the walk accepts along the rank-0 spine (the
    full model agrees with its own greedy drafts)."""
    p = si.prompt(tiny.cfg, 24)
    parents = _branching_tree()
    ar = decode.generate_ar(tiny, p, 6)
    V = tiny.cfg.vocab
    # rank-0 spine = greedy tokens; the other branches hold arbitrary tokens
    tokens = [ar[0], ar[1], (ar[1] + 5) % V, ar[2], (ar[2] + 9) % V, 17, 29, 41]
    s = decode.Session(tiny, 128)
    s.prefill(p)
    out = []
    cyc = s.verify_tree(tokens, parents, logits_out=out)
    for c in range(len(parents)):
        fresh = _fresh_logits(tiny, p, _path(tokens, parents, c))
        assert np.allclose(out[0][c], fresh, rtol=0, atol=1e-9), c
    assert cyc.path == [0, 1, 3] and cyc.bonus == ar[3]


def test_follow_commits_the_given_decision(tiny):
    """verify_linear / verify_tree with follow= commit another implementation's acceptance: the
    state afterwards equals that of a session that committed the same tokens by prefill."""
    p = si.prompt(tiny.cfg, 20)
    a = decode.Session(tiny, 128)
    first, _ = a.prefill(p)
    d = a.draft_linear((1, 2), 3)
    a.verify_linear(d, follow=(1, 7))  # accept the first draft, bonus 7
    assert (a.t, a.pending) == (22, 7) and a.target.token == d[0] and a.target.pos == 21
    t = decode.Session(tiny, 128)
    t.prefill(p)
    t.verify_tree([t.pending, 3, d[0], 5], [-1, 0, 0, 2], follow=([0, 2], 7))
    assert (t.t, t.pending) == (22, 7) and t.target.token == d[0]
    b = decode.Session(tiny, 128)
    b.prefill(list(p) + [first, d[0]])
    _, la = a.prefill([7])
    _, lt = t.prefill([7])
    _, lb = b.prefill([7])
    assert np.allclose(la[-1], lb[-1], atol=1e-11) and np.allclose(lt[-1], lb[-1], atol=1e-11)


def test_f32_products_match_f64(tiny_gqa):
    """The float32-product mode used for the full-size workloads against the float64 oracle:
    logits within 1e-4 and the same greedy tokens wherever the top-1/top-2 gap exceeds 1e-3."""
    cfg = tiny_gqa.cfg
    W32 = Weights(cfg, compute="f32")
    p = si.prompt(cfg, 40)
    a, b = decode.Session(tiny_gqa, 128), decode.Session(W32, 128)
    _, la = a.prefill(p)
    _, lb = b.prefill(p)
    assert float(np.max(np.abs(la - lb))) < 1e-4
    for sa_, sb_ in zip(a.target.states, b.target.states):
        assert float(np.max(np.abs(sa_ - sb_))) < 1e-5
    da = a.draft_linear((0, 3), 4, act_int8=True)
    db = b.draft_linear((0, 3), 4, act_int8=True, force=da)
    ca, cb = a.verify_linear(da), b.verify_linear(db)
    for r, (x, y) in enumerate(zip(ca.argmax, cb.argmax)):
        assert x == y or ca.gaps[r] < 1e-3
