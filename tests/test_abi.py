"""The C ABI library loads and exports every entry point its headers declare (no GPU needed)."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import self_speculative_decoding_layer_gb300 as ssd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(ssd_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    return ssd.load_library()


def test_headers_declare_the_boundary():
    names = declared_functions()
    for must in ("ssd_load_weights", "ssd_draft", "ssd_verify", "ssd_rollback", "ssd_dp_select"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_exports(lib):
    for n in ssd.EXPORTS:
        assert hasattr(lib, n)


def test_host_side_validation_without_gpu(lib):
    import ssd_inputs as si

    cfg = ssd.c_config(si.CONFIGS["tiny"])
    assert lib.ssd_workspace_bytes(ctypes.byref(cfg)) > 0
    assert lib.ssd_weight_count(ctypes.byref(cfg)) == 3 + 6 * 4
    bad = ssd.c_config(si.CONFIGS["tiny"].replace(head_dim=96))
    assert lib.ssd_workspace_bytes(ctypes.byref(bad)) == 0
    bad_rows = ssd.c_config(si.CONFIGS["tiny"], max_rows=65)
    assert lib.ssd_workspace_bytes(ctypes.byref(bad_rows)) == 0
    out = ctypes.c_void_p()
    assert lib.ssd_create(ctypes.byref(cfg), None, 0, None, ctypes.byref(out)) == 1  # null workspace
    assert lib.ssd_create(ctypes.byref(cfg), 0x1001, 1 << 40, None, ctypes.byref(out)) == 1  # misaligned
    assert lib.ssd_create(ctypes.byref(cfg), 0x10000, 16, None, ctypes.byref(out)) == 3  # too small
    assert lib.ssd_status_string(3) == b"capacity exceeded"


def test_null_context_calls_are_rejected(lib):
    assert lib.ssd_prefill(None, None, 0, None) == 1
    assert lib.ssd_verify(None, None, None, 0, None, None, None) == 1
    assert lib.ssd_rollback(None, 0, -1) == 1
    assert lib.ssd_dp_select(None, 0, None, None) == 1
    assert lib.ssd_draft(None, None, 0, 1, 0.0, None, None) == 1
    assert lib.ssd_get_draft_conf(None, 1, None) == 1
    lib.ssd_destroy(None)


def test_latency_fit_and_cascade_rule_match_the_oracle(lib):
    """Host-only parts of the DyTC scheduler: the library's least-squares latency fit and
    cascade-depth rule against the oracle's (independent code) on seeded points."""
    from oracle import latency

    rng = np.random.default_rng(11)
    for _ in range(5):
        n = int(rng.integers(3, 40))
        s = rng.uniform(1, 4096, n)
        d = rng.integers(0, 81, n).astype(float)
        if len(set(d)) < 2:
            d[0] += 1
        y = 0.3 + 2e-5 * s + 0.06 * d + rng.normal(0, 0.01, n)
        assert np.allclose(ssd.fit_latency(s, d, y), latency.fit_latency(s, d, y), rtol=1e-8, atol=1e-12)
    with pytest.raises(ssd.SSDError):
        ssd.fit_latency([64, 64, 64], [1, 2, 3], [1.0, 2.0, 3.0])
    for L in (1, 4, 11, 12, 23, 24, 32, 40, 47, 48, 80, 95, 96, 126, 200):
        for nl in (1, 2, 3):
            for sl in (0, 512, 513, 4096):
                assert ssd.cascade_depth(L, nl, sl) == latency.cascade_depth(L, nl, sl), (L, nl, sl)


def test_dytc_and_hcascade_planners_match_the_oracle(lib):
    """The library's host planners against the oracle's independent code: DyTC trees for seeded
    acceptance estimates and level costs (and budgets), horizontal-cascade chains."""
    import ssd_inputs as si
    from oracle import decode

    rng = np.random.default_rng(7)
    base = si.CONFIGS["llama2_13b_cascade"]
    for trial in range(60):
        nl = int(rng.integers(1, 4))
        ema = rng.uniform(0.05, 0.99, nl)
        cost = np.sort(rng.uniform(0.1, 1.0, nl))
        max_nodes, max_depth = int(rng.integers(1, 17)), int(rng.integers(1, 7))
        cfg = base.replace(levels=base.levels[:nl], tree_max_nodes=max_nodes, tree_max_depth=max_depth)
        d = decode.DyTC(cfg, costs=list(cost))
        d.a = list(ema)
        plan = d.plan()
        parents, exps = ssd.plan_tree(ema, cost, max_nodes, max_depth)
        assert parents == plan.parents and exps == [tuple(e) for e in plan.expansions], trial
    for lens in ([2, 1, 3], [0, 0, 1], [4, 0, 0], [1, 2]):
        parents, levels = decode.hcascade_chain(lens)
        got_parents, exps = ssd.plan_hcascade(lens)
        assert got_parents == parents and [l for _, l in exps] == levels
        assert [u for u, _ in exps] == list(range(len(levels)))
    with pytest.raises(ssd.SSDError):
        ssd.plan_hcascade([0, 0, 0])
    with pytest.raises(ssd.SSDError):
        ssd.plan_tree([0.5], [0.0], 4, 4)


def test_binding_structs_match_the_c_layout(lib):
    """Every struct the binding mirrors has the size the library was compiled with (a field added
    on one side only would shift the rest)."""
    out = (ctypes.c_size_t * 5)()
    lib.ssd_abi_sizes(out, 5)
    assert list(out) == [ctypes.sizeof(ssd.ModelConfigC), ctypes.sizeof(ssd.PolicyC), ctypes.sizeof(ssd.StatsC),
                         ctypes.sizeof(ssd.AttentionArgsC), ctypes.sizeof(ssd.CycleRecordC)]


def test_product_library_has_no_cross_check_kernels():
    """The cross-check kernels (CUDA-core rows kernel, the other batch-1 GEMVs) are built into the test
    library only: the product library refuses SSD_OPT_GEMM_IMPL != 0 before touching a context, and its
    symbol table names none of their launchers."""
    import subprocess

    prod, xcheck = ssd.LIB_PATH, ssd.XCHECK_LIB_PATH
    syms = {p: subprocess.run(["nm", "-D", "-C", p], capture_output=True, text=True).stdout +
            subprocess.run(["nm", "-C", p], capture_output=True, text=True).stdout for p in (prod, xcheck)}
    for name in ("launch_linear_rows", "launch_gemv_bulk", "k_linear_rows"):
        assert name not in syms[prod], name
        assert name in syms[xcheck], name
