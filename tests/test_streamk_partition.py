"""The stream-K work split of the tcgen05 projection (k_mma), checked on the CPU through the library's own
split rule (ssd_streamk_split runs the item_begin / item_cta the kernel uses): items (weight tile,
64-wide K stage) are cut into one contiguous run per CTA; a tile cut between CTAs is summed by the
CTA that completes it from the others' partial tiles, each stored in slot 0 (the tile is the first
of its CTA's run) or slot 1 (the last).  The model checks the index rules the kernel uses: every
item belongs to exactly one CTA, the CTA lookup inverts the run boundaries, the items counted for a
tile add up to its stage count exactly when its last contributor arrives, and the slot a reader
picks is the slot the writer used (a grid of at most one CTA per item keeps every run non-empty, so
every CTA a merge reads from wrote its partial)."""
import ctypes
import random

import pytest


@pytest.fixture(scope="module", autouse=True)
def lib():
    import __graft_entry__
    import self_speculative_decoding_layer_gb300 as ssd

    __graft_entry__.build()
    global _LIB
    _LIB = ssd.load_library()


_LIB = None


def item_begin(total, b, G):
    """The library's own rule (ssd_streamk_split, the same code the kernel runs)."""
    out = ctypes.c_int64()
    _LIB.ssd_streamk_split(total, G, b, 0, ctypes.byref(out), None)
    return out.value


def item_cta(total, i, G):
    out = ctypes.c_int()
    _LIB.ssd_streamk_split(total, G, 0, i, None, ctypes.byref(out))
    return out.value


def check(n_tiles, stages, sms):
    total = n_tiles * stages
    G = min(sms, total)  # the launcher's grid: never more CTAs than items, so no CTA's run is empty
    owner = [None] * total
    written = {}  # (cta, tile) -> slot
    for b in range(G):
        w0, w1 = item_begin(total, b, G), item_begin(total, b + 1, G)
        for i in range(w0, w1):
            assert owner[i] is None
            owner[i] = b
        assert w1 > w0
        t_first, t_last = w0 // stages, (w1 - 1) // stages
        for j, t in enumerate(range(t_first, t_last + 1)):
            s_a, s_b = max(w0, t * stages), min(w1, (t + 1) * stages)
            if s_b - s_a < stages:  # shared tile: a partial in slot 0 (first segment) or 1
                written[(b, t)] = 0 if j == 0 else 1
    assert all(o is not None for o in owner)
    for i in range(total):
        assert owner[i] == item_cta(total, i, G)
    for t in range(n_tiles):
        ta = t * stages
        c0, c1 = item_cta(total, ta, G), item_cta(total, ta + stages - 1, G)
        counted = 0
        for q in range(c0, c1 + 1):
            w0, w1 = item_begin(total, q, G), item_begin(total, q + 1, G)
            counted += min(w1, ta + stages) - max(w0, ta)
        assert counted == stages
        if c0 != c1:
            for q in range(c0, c1 + 1):
                seg = 0 if item_begin(total, q, G) // stages == t else 1
                assert written[(q, t)] == seg, (n_tiles, stages, sms, t, q)


def test_workload_shapes():
    # 8B verify: QKV 48 tiles x 64 stages, O 32 x 64, gate/up 112 x 64, down 32 x 224, lm_head 1002 x 64
    for n_tiles, stages in ((48, 64), (32, 64), (112, 64), (32, 224), (1002, 64), (40, 80), (64, 448)):
        check(n_tiles, stages, 152)


def test_seeded_shapes():
    rng = random.Random(3)
    for _ in range(300):
        check(rng.randint(1, 200), rng.randint(1, 300), rng.choice([1, 2, 7, 100, 148, 152, 160]))


def gemv_warps(nu, total):
    """The library's rule (ssd_gemv_warps)."""
    return _LIB.ssd_gemv_warps(nu, total)


def check_gemv(nu, nchunks, grid_warps):
    """Batch-1 GEMV (k_gemv_rs): nw warps split the (row pair, K chunk) steps evenly; a row pair cut
    by slice boundaries is written piece by piece (slot = the piece's first chunk) and the warp that
    completes it sums the pieces of warps g0..g1 in warp order."""
    total = nu * nchunks
    nw = min(grid_warps, gemv_warps(nu, total))
    pieces = {}  # unit -> list of (warp, c0, c1)
    for g in range(nw):
        s0, s1 = total * g // nw, total * (g + 1) // nw
        assert s1 > s0  # nw <= total: no warp without work
        s = s0
        while s < s1:
            u, c = divmod(s, nchunks)
            c1 = min(nchunks, c + (s1 - s))
            pieces.setdefault(u, []).append((g, c, c1))
            s += c1 - c
    assert sorted(pieces) == list(range(nu))
    for u, ps in pieces.items():
        assert sum(c1 - c0 for _, c0, c1 in ps) == nchunks
        assert [c0 for _, c0, _ in ps] == sorted(c0 for _, c0, _ in ps) and ps[0][1] == 0
        if len(ps) == 1:
            continue
        sa = u * nchunks
        g0 = ((sa + 1) * nw - 1) // total
        g1 = ((sa + nchunks) * nw - 1) // total
        assert [g for g, _, _ in ps] == list(range(g0, g1 + 1))
        read = [max(total * g // nw - sa, 0) for g in range(g0, g1 + 1)]
        assert read == [c0 for _, c0, _ in ps]


def test_gemv_split_rows_workload_shapes():
    # 8B: QKV 3072 row pairs x 4 chunks, O 2048 x 2 (2048-wide), gate/up 14336 x 4, down 2048 x 7, lm_head
    for nu, nch, warps in ((3072, 4, 152 * 32), (2048, 2, 152 * 16), (14336, 4, 152 * 32), (2048, 7, 152 * 16),
                           (64128, 2, 152 * 16), (128, 1, 152 * 32), (344, 1, 152 * 32)):
        check_gemv(nu, nch, warps)


def test_gemv_split_rows_seeded():
    rng = random.Random(5)
    for _ in range(300):
        check_gemv(rng.randint(1, 5000), rng.randint(1, 16), rng.choice([16, 152 * 16, 152 * 32, 1000]))
