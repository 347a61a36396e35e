"""GPU parity on the small workloads: every pass of the hot path through the C ABI
against the CPU oracle on the same seeded inputs."""
import numpy as np
import pytest

import ssd_inputs as si
from oracle import clasp, decode
from oracle.model import Weights

from gpu_util import (HIDDEN_COS, LOGIT_TOL, NEAR_TIE, Follow, cos, first_mismatch, gpu_ar_resync, near_thr,
                      oracle_ar_with_gaps, tree_cycle_against_oracle)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CFGS = {
    "tiny": si.CONFIGS["tiny"],
    # GQA (2 query heads per KV head), random RMSNorm gains, ragged FFN width
    "tiny_gqa": si.CONFIGS["tiny"].replace(name="tiny_gqa", n_kv_heads=2, gamma_sigma=0.1, ffn=720),
    # fp16 storage, head_dim 128, 6 layers
    "tiny_fp16": si.CONFIGS["tiny"].replace(name="tiny_fp16", dtype="fp16", n_layers=6, n_q_heads=2, n_kv_heads=2,
                                            head_dim=128, skip=(1, 3, 4)),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__

    __graft_entry__.build()


@pytest.fixture(scope="module")
def oracle_w():
    return {k: Weights(c) for k, c in CFGS.items()}


@pytest.fixture(scope="module")
def dev_w():
    import self_speculative_decoding_layer_gb300 as ssd

    return {k: ssd.DeviceWeights(c) for k, c in CFGS.items()}


def make(name, dev_w, impl=0, graphs=1, **kw):
    """An engine on the product library, or on the test library when a cross-check kernel is selected."""
    import self_speculative_decoding_layer_gb300 as ssd

    e = ssd.Engine(CFGS[name], dev_w[name], xcheck=impl != 0, **kw)
    e.set_option(ssd.OPT_GEMM_IMPL, impl)
    e.set_option(ssd.OPT_USE_GRAPHS, graphs)
    return e


def gpu_ar(name, dev_w, prompt, n):
    """The GPU's own plain greedy decoding (for losslessness checks on the GPU alone)."""
    import self_speculative_decoding_layer_gb300 as ssd

    e = make(name, dev_w)
    e.prefill(prompt)
    return e.generate(n, ssd.POLICY_AR)


@pytest.mark.parametrize("name", list(CFGS))
def test_device_weights_match_host_generator(name, dev_w):
    cfg = CFGS[name]
    w = dev_w[name]
    specs = {s.name: s for s in si.layer_specs(cfg, cfg.n_layers - 1)}
    qkv = w.tensors[3 + 6 * (cfg.n_layers - 1)].view(torch.int16).cpu().numpy().view(np.uint16)
    nq = cfg.n_q_heads * cfg.head_dim
    nk = cfg.n_kv_heads * cfg.head_dim
    assert np.array_equal(qkv[:nq], si.host_values(specs["wq"], cfg))
    assert np.array_equal(qkv[nq + nk:], si.host_values(specs["wv"], cfg))
    g = {s.name: s for s in si.global_specs(cfg)}
    emb = w.embed.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(emb, si.host_values(g["embed"], cfg))
    gf = w.final_norm.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(gf, si.host_values(g["final_norm"], cfg))


# tensor-core paths: 0 by shape, 4 split-K in a cluster, 5 stream-K; 1 the CUDA-core cross-check kernel
@pytest.mark.parametrize("impl", [0, 1, 4, 5])
@pytest.mark.parametrize("name", list(CFGS))
def test_prefill_logits_and_hidden(name, impl, oracle_w, dev_w):
    cfg = CFGS[name]
    prompt = si.prompt(cfg, 45)  # one 45-row chunk (ragged against every tile)
    eng = make(name, dev_w, impl)
    first = eng.prefill(prompt)
    s = decode.Session(oracle_w[name])
    o_first, o_logits = s.prefill(prompt)
    g = eng.logits(0)
    err = float(np.max(np.abs(g - o_logits[-1])))
    assert err < LOGIT_TOL, err
    for l in range(cfg.n_layers + 1):
        c = cos(eng.hidden(l, 44), s.target.states[l])
        assert c >= HIDDEN_COS, (l, c)
    if first != o_first:
        assert decode.model.top_gap(o_logits[-1]) < NEAR_TIE


@pytest.mark.parametrize("name", list(CFGS))
def test_prefill_chunks_equal_single_pass(name, dev_w):
    """A 100-token prompt (two chunks: 64 + 36 rows) equals prefill in 4 pieces."""
    cfg = CFGS[name]
    prompt = si.prompt(cfg, 100)
    a = make(name, dev_w)
    a.prefill(prompt)
    la = a.logits(0)
    b = make(name, dev_w)
    for off in (0, 30, 64, 90):
        end = {0: 30, 30: 64, 64: 90, 90: 100}[off]
        b.prefill(prompt[off:end])
    lb = b.logits(0)
    assert float(np.max(np.abs(la - lb))) < 1e-2


@pytest.mark.parametrize("graphs", [1, 0])
@pytest.mark.parametrize("name", list(CFGS))
def test_autoregressive_tokens_match_oracle(name, graphs, oracle_w, dev_w):
    cfg = CFGS[name]
    prompt = si.prompt(cfg)
    toks, gaps = oracle_ar_with_gaps(oracle_w[name], prompt, 48)
    eng = make(name, dev_w, graphs=graphs)
    near, hard = gpu_ar_resync(eng, prompt, toks, gaps)
    assert not hard, hard
    assert near <= 2


@pytest.mark.parametrize("impl", [0, 1, 4, 5])
@pytest.mark.parametrize("name", list(CFGS))
def test_linear_cycles_match_oracle(name, impl, oracle_w, dev_w):
    """Teacher-forced cycles: the oracle drafts on the GPU's drafts (every step compared), verifies the
    same rows (every row's logits compared) and follows the GPU's acceptance; int8 drafts every other
    cycle, with the last draft step's logits compared."""
    cfg = CFGS[name]
    prompt = si.prompt(cfg)
    eng = make(name, dev_w, impl)
    s = decode.Session(oracle_w[name])
    first = eng.prefill(prompt)
    o_first, o_logits = s.prefill(prompt)
    near = 0
    if first != o_first:
        assert decode.model.top_gap(o_logits[-1]) < NEAR_TIE
        near, s.pending = 1, first
    for cyc_i in range(8):
        int8 = cyc_i % 2 == 1
        drafts = eng.draft(cfg.skip, cfg.draft_k, act_int8=int8)
        gaps, am, rows = [], [], []
        s.draft_linear(cfg.skip, cfg.draft_k, act_int8=int8, gaps=gaps, force=drafts, argmax=am, rows=rows)
        err = float(np.max(np.abs(eng.logits(0) - rows[-1])))
        assert err < LOGIT_TOL, (cyc_i, int8, err)
        for r in range(len(drafts)):
            if am[r] != drafts[r]:  # only where the oracle's draft logits are nearly tied
                assert gaps[r] < NEAR_TIE, (cyc_i, r, drafts, am, gaps)
                near += 1
        n_acc, path, bonus = eng.verify([s.pending] + drafts)
        lo = []
        cyc = s.verify_linear(drafts, follow=(n_acc, bonus), logits_out=lo)
        for r in range(len(drafts) + 1):
            err = float(np.max(np.abs(eng.logits(r) - lo[0][r])))
            assert err < LOGIT_TOL, (cyc_i, r, err)
        if (n_acc, bonus) != (cyc.n_accepted, cyc.bonus):
            j = min(n_acc, cyc.n_accepted)  # the row whose argmax decided differently
            assert cyc.gaps[j] < NEAR_TIE, (cyc_i, n_acc, bonus, cyc)
            near += 1
        assert path == list(range(n_acc + 1))
        assert eng.position() == (s.t, s.pending)
    assert near <= 3


EXIT_SKIP = {"tiny": (0, 3), "tiny_gqa": (0, 3), "tiny_fp16": (1, 3, 4)}


@pytest.mark.parametrize("name", list(CFGS))
def test_draft_exit_matches_oracle(name, oracle_w, dev_w):
    """Draft exit: each draft's top-1 probability against the oracle's, the stop after the first
    draft below the threshold, then the verify of the shortened draft (teacher-forced cycles)."""
    cfg = CFGS[name]
    K, skip = 6, EXIT_SKIP[name]
    prompt = si.prompt(cfg)
    eng = make(name, dev_w)
    s = decode.Session(oracle_w[name])
    assert eng.prefill(prompt) == s.prefill(prompt)[0]
    near_tok = near_stop = 0
    lengths = set()
    for cyc in range(10):
        pre = []
        s.draft_linear(skip, K, probs=pre)
        q = np.sort(pre)
        thr = 1.5 if cyc == 9 else float(0.5 * (q[cyc % (K - 1)] + q[cyc % (K - 1) + 1]))
        drafts = eng.draft(skip, K, exit_thr=thr)
        n = len(drafts)
        assert 1 <= n <= K
        lengths.add(n)
        gaps, probs, am = [], [], []
        s.draft_linear(skip, n, gaps=gaps, probs=probs, force=drafts, argmax=am)
        for r in range(n):
            if am[r] != drafts[r]:
                assert gaps[r] < NEAR_TIE, (cyc, r, drafts, am, gaps)
                near_tok += 1
        conf = eng.draft_conf(n)
        for r in range(n):
            assert abs(np.log(conf[r]) - np.log(probs[r])) < 2 * LOGIT_TOL, (cyc, r, conf, probs)
        # the oracle's decision at every step the GPU took: go on before the last draft, stop at it
        for r in range(n):
            stop = probs[r] < thr
            want = r == n - 1 and n < K
            if stop != want:
                assert near_thr(probs[r], thr), (cyc, r, probs, thr, n)
                near_stop += 1
        n_acc, path, bonus = eng.verify([s.pending] + drafts)
        cyc_o = s.verify_linear(drafts, follow=(n_acc, bonus))
        if (n_acc, bonus) != (cyc_o.n_accepted, cyc_o.bonus):
            assert cyc_o.gaps[min(n_acc, cyc_o.n_accepted)] < NEAR_TIE, (cyc, n_acc, bonus, cyc_o)
            near_tok += 1
        assert eng.position() == (s.t, s.pending)
    assert near_tok + near_stop <= 3, (near_tok, near_stop)
    assert 1 in lengths and len(lengths) >= 2, lengths


def test_draft_exit_generate_matches_oracle(oracle_w, dev_w):
    """ssd_generate with a draft exit, decided on the device: lossless (equal to the GPU's own greedy
    decoding), and every cycle -- its drafts, stop point, verify rows and acceptance -- recomputed by the
    oracle on the GPU's inputs."""
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = CFGS["tiny"]
    prompt = si.prompt(cfg)
    probe = decode.Session(oracle_w["tiny"])
    probe.prefill(prompt)
    pre = []
    probe.draft_linear((0, 3), 8, probs=pre)
    thr = float(np.median(pre))
    eng = make("tiny", dev_w)
    eng.prefill(prompt)
    eng.set_option(ssd.OPT_CYCLE_LOG, 1)
    got = eng.generate(cfg.n_gen, ssd.POLICY_STATIC, skip=(0, 3), k=6, exit_thr=thr)
    assert got == gpu_ar("tiny", dev_w, prompt, cfg.n_gen)
    f = Follow(oracle_w["tiny"], prompt, got[0])
    log = eng.cycle_log()
    for e in log:
        f.linear(e, (0, 3), exit_thr=thr, k=6)
    st = eng.stats()
    assert st["cycles"] == len(log) and sum(st["accept_hist"]) == st["cycles"]
    assert st["drafted"] < 6 * st["cycles"]  # the exit cut some cycles short
    assert f.near <= 3, f.near


@pytest.mark.parametrize("impl,pdl,graphs", [(1, 1, 1), (2, 1, 1), (3, 1, 1), (0, 0, 1), (0, 1, 0), (3, 1, 0)])
def test_draft_exit_kernel_variants_agree(impl, pdl, graphs, dev_w):
    """The captured draft loop (a conditional graph node that stops launching forwards at the exit)
    and the eager path (later forwards' kernels return at a closed gate), with every GEMV variant and
    with or without programmatic dependent launch: same drafts, stop point and probabilities."""
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = CFGS["tiny_gqa"]
    prompt = si.prompt(cfg)
    ref = make("tiny_gqa", dev_w)
    e = make("tiny_gqa", dev_w, impl, graphs=graphs)
    e.set_option(ssd.OPT_PDL, pdl)
    ref.prefill(prompt)
    e.prefill(prompt)
    for cyc in range(4):
        t, p = ref.position()
        conf_all = ref.draft((0, 3), 6, exit_thr=1e-30)  # never stops: every draft's probability
        pr = np.sort(ref.draft_conf(6))
        thr = float(0.5 * (pr[cyc] + pr[cyc + 1]))
        a = ref.draft((0, 3), 6, exit_thr=thr)
        b = e.draft((0, 3), 6, exit_thr=thr)
        assert a == b and a == conf_all[: len(a)], (cyc, a, b, conf_all)
        assert np.allclose(ref.draft_conf(len(a)), e.draft_conf(len(b)), rtol=1e-3)
        na = ref.verify([p] + a)
        nb = e.verify([p] + b)
        assert na == nb


@pytest.mark.parametrize("name", list(CFGS))
def test_draft_equal_target_accepts_all(name, dev_w):
    cfg = CFGS[name]
    eng = make(name, dev_w)
    first = eng.prefill(si.prompt(cfg))
    for _ in range(4):
        t, p = eng.position()
        drafts = eng.draft((), 5)
        n_acc, _, _ = eng.verify([p] + drafts)
        assert n_acc == 5


@pytest.mark.parametrize("name", list(CFGS))
def test_spec_generate_equals_autoregressive(name, oracle_w, dev_w):
    """The speculative loop inside the library is lossless on the GPU (equal to the GPU's own greedy
    decoding), and every cycle of it is recomputed by the oracle on the GPU's inputs."""
    cfg = CFGS[name]
    import self_speculative_decoding_layer_gb300 as ssd

    prompt = si.prompt(cfg)
    b = make(name, dev_w)
    b.prefill(prompt)
    b.set_option(ssd.OPT_CYCLE_LOG, 1)
    sp = b.generate(cfg.n_gen, ssd.POLICY_STATIC)
    assert sp == gpu_ar(name, dev_w, prompt, cfg.n_gen)
    f = Follow(oracle_w[name], prompt, sp[0])
    for e in b.cycle_log():
        f.linear(e, cfg.skip)
    st = b.stats()
    assert st["cycles"] > 0 and sum(st["accept_hist"]) == st["cycles"]
    assert st["mma_fallbacks"] == 0  # every multi-row projection ran on the tensor cores
    assert f.near <= 3, f.near


def test_chain_tree_equals_linear(dev_w):
    cfg = CFGS["tiny"]
    prompt = si.prompt(cfg)
    a = make("tiny", dev_w)
    b = make("tiny", dev_w)
    pa = a.prefill(prompt)
    b.prefill(prompt)
    d = a.draft(cfg.skip, 4)
    assert d == b.draft(cfg.skip, 4)
    ra = a.verify([pa] + d)
    rb = b.verify([pa] + d, [-1, 0, 1, 2, 3])
    assert ra == rb
    assert np.array_equal(a.logits(2), b.logits(2))


@pytest.mark.parametrize("impl", [0, 4, 5])
@pytest.mark.parametrize("name", ["tiny", "tiny_gqa"])
def test_tree_verify_and_compaction_match_oracle(name, impl, oracle_w, dev_w):
    """A hand-made tree whose accepted branch is not the first one: acceptance,
    compaction and the next pass all agree with the oracle."""
    cfg = CFGS[name]
    prompt = si.prompt(cfg)
    eng = make(name, dev_w, impl)
    s = decode.Session(oracle_w[name])
    first = eng.prefill(prompt)
    s.prefill(prompt)
    ref = decode.Session(oracle_w[name])
    ref.prefill(prompt)
    a1, _ = ref.ar_step()
    a2, _ = ref.ar_step()
    wrong = (a1 + 7) % cfg.vocab
    tokens = [first, wrong, a1, (a2 + 3) % cfg.vocab, a2, 5]
    parents = [-1, 0, 0, 2, 2, 1]
    got = eng.verify(tokens, parents)
    cyc = s.verify_tree(tokens, parents)
    assert got == (cyc.n_accepted, cyc.path, cyc.bonus)
    for _ in range(3):  # continue decoding on the compacted cache
        assert eng.decode_ar(1)[0] == s.ar_step()[0]


@pytest.mark.parametrize("n", [0, 1, 2, 4])
@pytest.mark.parametrize("name", list(CFGS))
def test_dp_select_matches_oracle(name, n, oracle_w, dev_w):
    """The whole DP table, cell by cell (decision and value), against the oracle's; the mask and dp[L][n]."""
    from gpu_util import compare_dp_tables, oracle_cands

    cfg = CFGS[name]
    if n > cfg.n_layers:
        pytest.skip()
    prompt = si.prompt(cfg)
    eng = make(name, dev_w)
    s = decode.Session(oracle_w[name])
    eng.prefill(prompt)
    s.prefill(prompt)
    mask, val = eng.dp_select(n)
    o_mask, o_val, table = clasp.dp_search(s, n)
    assert len(mask) == n
    tv, tb = eng.dp_table()
    flip, _ = compare_dp_tables(tv, tb, oracle_cands(table, cfg.n_layers, n), cfg.n_layers, n)
    if flip is None:
        assert mask == o_mask and abs(val - o_val) < 2e-3
    else:  # a near-tie decided differently: the GPU's set is within 1e-3 of the oracle's optimum
        assert clasp.cosine(clasp.skipped_state(s, mask), s.target.states[cfg.n_layers]) >= o_val - 1e-3


@pytest.mark.parametrize("impl", [4, 5])
def test_dp_tables_of_both_tensor_core_distributions(impl, oracle_w, dev_w):
    """The DP pass with the split-K and the stream-K tensor-core kernels: whole table against the oracle."""
    from gpu_util import compare_dp_tables, oracle_cands

    cfg = CFGS["tiny_gqa"]
    prompt = si.prompt(cfg)
    eng = make("tiny_gqa", dev_w, impl)
    s = decode.Session(oracle_w["tiny_gqa"])
    eng.prefill(prompt)
    s.prefill(prompt)
    for n in (2, 3):
        mask, val = eng.dp_select(n)
        o_mask, o_val, table = clasp.dp_search(s, n)
        tv, tb = eng.dp_table()
        flip, _ = compare_dp_tables(tv, tb, oracle_cands(table, cfg.n_layers, n), cfg.n_layers, n)
        assert flip is not None or (mask == o_mask and abs(val - o_val) < 2e-3)


def test_dp_after_verify_uses_last_accepted_token(oracle_w, dev_w):
    cfg = CFGS["tiny"]
    prompt = si.prompt(cfg)
    eng = make("tiny", dev_w)
    s = decode.Session(oracle_w["tiny"])
    eng.prefill(prompt)
    s.prefill(prompt)
    for _ in range(3):
        d = eng.draft(cfg.skip, 4)
        eng.verify([s.pending] + d)
        s.verify_linear(s.draft_linear(cfg.skip, 4))
    mask, val = eng.dp_select(2)
    o_mask, o_val, _ = clasp.dp_search(s, 2)
    assert mask == o_mask or clasp.cosine(clasp.skipped_state(s, mask), s.target.states[4]) >= o_val - 1e-3
    assert abs(val - o_val) < 2e-3


def test_clasp_generate_equals_oracle(oracle_w, dev_w):
    """CLaSp generation: DP right after prefill and every 3 verify steps; every DP mask and every cycle
    recomputed by the oracle on the GPU's inputs, and lossless on the GPU."""
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = CFGS["tiny"]
    prompt = si.prompt(cfg)
    eng = make("tiny", dev_w)
    eng.prefill(prompt)
    eng.set_option(ssd.OPT_CYCLE_LOG, 1)
    got = eng.generate(48, ssd.POLICY_CLASP, k=3, dp_n_skip=2, dp_interval=3)
    assert got == gpu_ar("tiny", dev_w, prompt, 48)
    f = Follow(oracle_w["tiny"], prompt, got[0])
    skip, n_dp = None, 0
    for e in eng.cycle_log():
        if e["kind"] == 2:
            skip = f.dp(e, 2)
            n_dp += 1
        else:
            f.linear(e, skip)
    assert n_dp >= 2 and eng.stats()["dp_runs"] == n_dp
    assert f.near <= 3, f.near


def test_dytc_generate_matches_oracle(oracle_w, dev_w):
    """DyTC generation: every cycle's plan (from the oracle's own acceptance estimates), every expansion,
    every verify row, and the estimates after every update, recomputed by the oracle on the GPU's
    inputs; lossless on the GPU."""
    import self_speculative_decoding_layer_gb300 as ssd

    levels = (((0, 1, 2), False), ((1,), True), ((), True))
    cfg = CFGS["tiny"].replace(tree=True, levels=levels)
    prompt = si.prompt(cfg)
    eng = make("tiny", dev_w)
    eng.cfg = cfg
    eng.prefill(prompt)
    eng.set_option(ssd.OPT_CYCLE_LOG, 1)
    got = eng.generate(40, ssd.POLICY_DYTC, levels=levels)
    assert got == gpu_ar("tiny", dev_w, prompt, 40)
    f = Follow(Weights(cfg), prompt, got[0])
    dy = decode.DyTC(cfg)
    log = eng.cycle_log()
    for e in log:
        f.dytc(e, dy)
    st = eng.stats()
    assert st["cycles"] == len(log) and st["ema"][:3] == dy.a
    assert any(len(e["parents"]) > 2 for e in log)
    assert f.near <= 3, f.near


def test_early_exit_generation_matches_oracle(oracle_w, dev_w):
    """Static drafts with an early exit ([CAS-blog] §2.1 item 2): every cycle recomputed by the oracle
    (which runs the exit as a shortened layer loop) on the GPU's inputs; lossless on the GPU."""
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = CFGS["tiny_gqa"]
    prompt = si.prompt(cfg)
    eng = make("tiny_gqa", dev_w)
    eng.prefill(prompt)
    eng.set_option(ssd.OPT_CYCLE_LOG, 1)
    got = eng.generate(48, ssd.POLICY_STATIC, skip=(1,), k=4, early_exit=2)
    assert got == gpu_ar("tiny_gqa", dev_w, prompt, 48)
    f = Follow(oracle_w["tiny_gqa"], prompt, got[0])
    for e in eng.cycle_log():
        f.linear(e, (1,), exit_layers=2)
    # one draft call: the exit is the mask with the last layers set
    s = decode.Session(oracle_w["tiny_gqa"])
    s.prefill(prompt)
    e2 = make("tiny_gqa", dev_w)
    e2.prefill(prompt)
    d = e2.draft((1,), 4, early_exit=2)
    gaps, am = [], []
    s.draft_linear((1,), 4, exit_layers=2, gaps=gaps, force=d, argmax=am)
    for r in range(4):
        assert am[r] == d[r] or gaps[r] < NEAR_TIE, (r, d, am, gaps)
    assert f.near <= 3, f.near


def test_dytc_with_early_exit_level_matches_oracle(oracle_w, dev_w):
    import self_speculative_decoding_layer_gb300 as ssd

    levels = (((1,), False), ((1,), True), ((), True))
    cfg = CFGS["tiny"].replace(tree=True, levels=levels, level_exit=(2, 0, 0))
    prompt = si.prompt(cfg)
    eng = make("tiny", dev_w)
    eng.cfg = cfg
    eng.prefill(prompt)
    W = Weights(cfg)
    s = decode.Session(W)
    s.prefill(prompt)
    toks, parents = eng.draft_tree()
    plan = decode.DyTC(cfg).plan(s.t)
    assert parents == plan.parents
    assert tree_cycle_against_oracle(eng, s, toks, parents, plan.expansions, levels, cfg.level_exit) <= 2
    e2 = make("tiny", dev_w)
    e2.cfg = cfg
    e2.prefill(prompt)
    e2.set_option(ssd.OPT_CYCLE_LOG, 1)
    got = e2.generate(40, ssd.POLICY_DYTC)
    assert got == gpu_ar("tiny", dev_w, prompt, 40)
    f = Follow(W, prompt, got[0])
    dy = decode.DyTC(cfg)
    for e in e2.cycle_log():
        f.dytc(e, dy)
    assert e2.stats()["ema"][:3] == dy.a
    assert f.near <= 3, f.near


def test_dytc_tree_draft_matches_oracle(oracle_w, dev_w):
    """One DyTC tree: the same plan as the oracle's, every expansion's top-2 recomputed by the oracle on
    the GPU's tree tokens, every node's verify logits, and the acceptance."""
    levels = (((0, 1, 2), False), ((1,), True), ((), True))
    cfg = CFGS["tiny"].replace(tree=True, levels=levels)
    prompt = si.prompt(cfg)
    eng = make("tiny", dev_w)
    eng.cfg = cfg
    eng.prefill(prompt)
    toks, parents = eng.draft_tree(levels=levels)
    s = decode.Session(Weights(cfg))
    s.prefill(prompt)
    plan = decode.DyTC(cfg).plan(s.t)
    assert parents == plan.parents and toks[0] == s.pending
    assert len(plan.expansions) >= 2
    assert tree_cycle_against_oracle(eng, s, toks, parents, plan.expansions, levels) <= 2


def test_validation_errors(dev_w):
    import self_speculative_decoding_layer_gb300 as ssd

    eng = make("tiny", dev_w)
    with pytest.raises(ssd.SSDError) as e:
        eng.verify([1, 2])
    assert e.value.status == 2  # before prefill
    with pytest.raises(ssd.SSDError) as e:
        eng.dp_select(1)
    assert e.value.status == 2
    first = eng.prefill(si.prompt(CFGS["tiny"]))
    t = eng.position()
    with pytest.raises(ssd.SSDError) as e:
        eng.verify([first, 1, 2], [-1, 0, 5])  # parent not before child
    assert e.value.status == 1
    with pytest.raises(ssd.SSDError) as e:
        eng.verify([first + 1, 1])  # tokens[0] must be the pending token
    assert e.value.status == 1
    with pytest.raises(ssd.SSDError) as e:
        eng.verify([first, 5000])
    assert e.value.status == 1
    with pytest.raises(ssd.SSDError) as e:
        eng.dp_select(5)
    assert e.value.status == 1
    with pytest.raises(ssd.SSDError) as e:
        eng.draft((1,), 64)
    assert e.value.status == 1
    with pytest.raises(ssd.SSDError) as e:
        eng.rollback(t[0] + 1)
    assert e.value.status == 1
    assert eng.position() == t  # failed calls leave the context unchanged



def test_nan_logits_give_tokens_in_the_vocabulary():
    """Greedy choices count a NaN logit as -inf (the header's rule): with a NaN final RMSNorm gain every logit
    is NaN, so every choice is the lowest id, 0, on the one-row (GEMV) and the tensor-core paths alike, and the
    tokens fed back stay inside the vocabulary."""
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = CFGS["tiny"]
    w = ssd.DeviceWeights(cfg)
    w.final_norm.fill_(float("nan"))
    eng = ssd.Engine(cfg, w)
    assert eng.prefill(si.prompt(cfg)) == 0
    assert eng.decode_ar(3) == [0, 0, 0]
    drafts = eng.draft(cfg.skip, 3)
    assert drafts == [0, 0, 0]
    t, p = eng.position()
    n_acc, _, bonus = eng.verify([p] + drafts)
    assert (n_acc, bonus) == (3, 0)
    assert eng.position() == (t + 4, 0)

@pytest.mark.parametrize("name", list(CFGS))
def test_pdl_and_gemv_variants_agree(name, dev_w):
    """Programmatic dependent launch changes only when kernels start (bit-identical
    results); the two one-row GEMV kernels differ only in summation order."""
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = CFGS[name]
    prompt = si.prompt(cfg)
    outs, logits = [], []
    for pdl, impl in ((1, 0), (0, 0), (1, 2)):
        e = make(name, dev_w, impl)
        e.set_option(ssd.OPT_PDL, pdl)
        e.prefill(prompt)
        outs.append(e.generate(24, ssd.POLICY_STATIC))
        e.draft(cfg.skip, 1)
        logits.append(e.logits(0))
    assert outs[0] == outs[1]
    assert np.array_equal(logits[0], logits[1])
    assert float(np.max(np.abs(logits[0] - logits[2]))) < 1e-3


def test_calibrate_latency_fits_measured_passes(dev_w):
    """[CAS-blog] §3.2 latency model from CUDA-event timings of one-draft passes: more layers
    cost more, the fit reproduces the measured points within the pages' 15 %, the returned
    model is the library's least-squares fit of the returned times, and held-out points work."""
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = CFGS["tiny"]
    eng = make("tiny", dev_w)
    eng.prefill(si.prompt(cfg, 120))
    seqs, depths = [120, 90, 60, 30], [0, 1, 2, 3, 4]
    beta, times = eng.calibrate_latency(depths, seqs, reps=7)
    assert np.all(times > 0) and beta[2] > 0
    S = np.repeat(seqs, len(depths)).astype(float)
    D = np.tile(depths, len(seqs)).astype(float)
    pred = beta[0] + beta[1] * S + beta[2] * D
    assert np.max(np.abs(pred - times.reshape(-1)) / times.reshape(-1)) < 0.15, (beta, times)
    assert np.allclose(ssd.fit_latency(S, D, times.reshape(-1)), beta, rtol=1e-9)
    assert eng.position()[0] == 30  # rolled back to the shortest context
    # fit on two context lengths, predict the other two
    eng2 = make("tiny", dev_w)
    eng2.prefill(si.prompt(cfg, 120))
    train = np.zeros((4, 5), dtype=np.uint8)
    train[[0, 3]] = 1
    b2, t2 = eng2.calibrate_latency(depths, seqs, reps=7, train=train, act_int8=True)
    held = (b2[0] + b2[1] * S + b2[2] * D).reshape(4, 5)[1:3]
    assert np.max(np.abs(held - t2[1:3]) / t2[1:3]) < 0.15, (b2, t2)
    with pytest.raises(ssd.SSDError):  # one context length cannot determine the seq_len term
        eng2.calibrate_latency(depths, [20])


def test_dytc_latency_model_and_depth_rule_match_oracle():
    """DyTC with the latency-model costs and the cascade depth rule on a 48-layer model
    (log2(48/12) = 2 levels, one when the context passes 512): the same level costs, and every
    cycle's plan, expansions, verify rows and estimates recomputed by the oracle given the same
    latency models."""
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = si.CONFIGS["tiny"].replace(name="tiny_deep", n_layers=48, tree=True, levels=si.cascade_levels(48),
                                     prompt_len=520, n_gen=24)
    b16, b8 = (0.05, 1e-5, 0.01), (0.05, 1e-5, 0.008)
    w = ssd.DeviceWeights(cfg)
    W = Weights(cfg)
    for plen, n_active in ((32, 2), (520, 1)):
        prompt = si.prompt(cfg, plen)
        eng = ssd.Engine(cfg, w)
        eng.set_latency_model(b16, False)
        eng.set_latency_model(b8, True)
        eng.prefill(prompt)
        costs, n = eng.level_costs(cost_model=1, cascade_rules=1)
        ref = decode.DyTC(cfg, rules=True, betas=(b16, b8))
        ref.plan(plen)
        assert n == n_active
        assert costs == pytest.approx(ref.c, rel=1e-12)
        eng.set_option(ssd.OPT_CYCLE_LOG, 1)
        got = eng.generate(24, ssd.POLICY_DYTC, cost_model=1, cascade_rules=1)
        e_ar = ssd.Engine(cfg, w)
        e_ar.prefill(prompt)
        assert got == e_ar.generate(24, ssd.POLICY_AR)
        f = Follow(W, prompt, got[0])
        dy = decode.DyTC(cfg, rules=True, betas=(b16, b8))
        log = eng.cycle_log()
        for e in log:
            f.dytc(e, dy)
        assert all(len(e["parents"]) >= 1 for e in log)
        assert f.near <= 3, (plen, f.near)
        del eng, e_ar


def test_hcascade_generate_matches_oracle(oracle_w, dev_w):
    """Horizontal cascade baseline: chains drafted L3 -> L2 -> L1 by position, verified in one pass;
    every chain position and verify row recomputed by the oracle on the GPU's inputs; lossless."""
    import self_speculative_decoding_layer_gb300 as ssd

    levels = (((0, 1, 2), False), ((1,), True), ((), True))
    cfg = CFGS["tiny"].replace(tree=True, levels=levels)
    prompt = si.prompt(cfg)
    eng = make("tiny", dev_w)
    eng.cfg = cfg
    eng.prefill(prompt)
    eng.set_option(ssd.OPT_CYCLE_LOG, 1)
    got = eng.generate(40, ssd.POLICY_HCASCADE, hc_len=(2, 1, 1))
    assert got == gpu_ar("tiny", dev_w, prompt, 40)
    parents, lv = decode.hcascade_chain((2, 1, 1))
    f = Follow(Weights(cfg), prompt, got[0])
    log = eng.cycle_log()
    for e in log:
        f.tree(e, parents, [(r, l) for r, l in enumerate(lv)], levels)
    st = eng.stats()
    assert st["cycles"] == len(log) and st["drafted"] == 4 * len(log)
    assert f.near <= 3, f.near
    with pytest.raises(ssd.SSDError):
        eng.generate(8, ssd.POLICY_HCASCADE, hc_len=(0, 0, 0))


def test_vcascade_generate_matches_oracle(oracle_w, dev_w):
    """Vertical cascade baseline: L1 drafts, L2 (int8) checks them in one multi-row pass and keeps the
    prefix it agrees with plus its correction, the target verifies; every lower draft, higher check and
    verify row recomputed by the oracle on the GPU's chain.  With the target itself as the higher level
    every chain is accepted whole."""
    import self_speculative_decoding_layer_gb300 as ssd

    levels = (((0, 1, 2), False), ((1,), True), ((), False))
    cfg = CFGS["tiny"].replace(tree=True, levels=levels)
    prompt = si.prompt(cfg)
    W = Weights(cfg)
    ar = gpu_ar("tiny", dev_w, prompt, 40)
    for hi in (1, 2):
        eng = make("tiny", dev_w)
        eng.cfg = cfg
        eng.prefill(prompt)
        eng.set_option(ssd.OPT_CYCLE_LOG, 1)
        got = eng.generate(40, ssd.POLICY_VCASCADE, k=4, vc_lo=0, vc_hi=hi)
        assert got == ar
        f = Follow(W, prompt, got[0])
        log = eng.cycle_log()
        for e in log:
            f.vcascade(e, 0, hi, 4)
        st = eng.stats()
        assert st["cycles"] == len(log)
        assert st["drafted"] == sum(sum(x >= 0 for x in e["tokens"][1:]) for e in log)
        if hi == 2:
            assert st["accepted"] == st["drafted"]
        assert f.near <= 3, (hi, f.near)
    with pytest.raises(ssd.SSDError):
        eng.generate(8, ssd.POLICY_VCASCADE, k=4, vc_lo=1, vc_hi=1)
