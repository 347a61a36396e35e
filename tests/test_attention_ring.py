"""CPU model of the attention kernel's tile ring (k_attention): which warps consume which key tiles,
when slots are refilled, and what a parity wait on an mbarrier can tell apart.

A slot's mbarrier completes one phase per copy that lands in it; a wait names only the parity of the
phase it wants, so a wait for tile k + R (parity 1) on a slot that has not yet completed tile k's
phase returns at once.  The kernel therefore gives all tiles of a slot to the warps that released the
tile before it: with refills it uses a power of two R of its S slots and at most R warp sets
(R % WK == 0).  The model replays random interleavings of copies landing and warps waiting and checks
that every warp reads the tile it expects and that nothing waits forever.  The rule replayed is the
library's own (ssd_attn_ring_rule runs the functions the kernel calls); the old rule (all S slots,
kWarps / WQ sets) is shown to fail, so the model can see the hazard.  A second replay covers slots filled
before the dependency wait under a stale hint (their phases then run one ahead)."""
import ctypes
import random

import pytest

K_WARPS = 16
_LIB = None


@pytest.fixture(scope="module", autouse=True)
def lib():
    import __graft_entry__
    import self_speculative_decoding_layer_gb300 as ssd

    __graft_entry__.build()
    global _LIB
    _LIB = ssd.load_library()


def ring_rule(ntile, S, WQ, fixed=True):
    if not fixed:
        return S, K_WARPS // WQ
    R, WK = ctypes.c_int(-1), ctypes.c_int(-1)
    _LIB.ssd_attn_ring_rule(ntile, S, WQ, ctypes.byref(R), ctypes.byref(WK))
    return R.value, WK.value


def replay(ntile, S, WQ, fixed, seed):
    rnd = random.Random(seed)
    R, WK = ring_rule(ntile, S, WQ, fixed)
    completed, content, cons = [0] * R, [None] * R, [0] * R
    inflight = [(w, w) for w in range(min(R, ntile))]
    todo = [list(range(w // WQ, ntile, WK)) if w // WQ < WK else [] for w in range(K_WARPS)]
    pos = [0] * K_WARPS
    for _ in range(200000):
        busy = [w for w in range(K_WARPS) if pos[w] < len(todo[w])]
        if not busy and not inflight:
            return "ok"
        if inflight and (not busy or rnd.random() < 0.3):
            slot, tile = inflight.pop(rnd.randrange(len(inflight)))
            completed[slot] += 1
            content[slot] = tile
            continue
        w = rnd.choice(busy)
        k = todo[w][pos[w]]
        slot, parity = k % R, (k // R) & 1
        if completed[slot] % 2 != parity:  # the parity wait returns
            if content[slot] != k:
                return "wrong tile"
            pos[w] += 1
            cons[slot] += 1
            if cons[slot] == WQ:  # the last consumer refills the slot
                cons[slot] = 0
                if k + R < ntile:
                    inflight.append((slot, k + R))
    return "hang"


def replay_early(ntile, S, WQ, stale, shift, seed):
    """The ring when slots in `stale` were filled before the dependency wait under a stale prefix hint: each
    such copy lands as an extra phase, then the slot's warp issues the real first copy; consumers wait for
    parity (k // R + shift[slot]) & 1.  Slots at or past R (or with no tile) are only drained.  The slot's
    warp waits for the stale copy before the block barrier that precedes the tile loop, so no consumer
    starts before every stale copy has landed."""
    rnd = random.Random(seed)
    R, WK = ring_rule(ntile, S, WQ)
    completed, content, cons = [0] * S, [None] * S, [0] * S
    sh = [1 if shift and s in stale else 0 for s in range(S)]
    inflight = [(s, "stale") for s in stale] + [(w, w) for w in range(min(R, ntile)) if w not in stale]
    todo = [list(range(w // WQ, ntile, WK)) if w // WQ < WK else [] for w in range(K_WARPS)]
    pos = [0] * K_WARPS
    for _ in range(200000):
        busy = [w for w in range(K_WARPS) if pos[w] < len(todo[w])]
        if not busy and not inflight:
            return "ok"
        draining = any(t == "stale" for _, t in inflight)
        if inflight and (draining or not busy or rnd.random() < 0.3):
            slot, tile = inflight.pop(rnd.randrange(len(inflight)))
            completed[slot] += 1
            content[slot] = tile
            if tile == "stale" and slot < min(R, ntile):
                inflight.append((slot, slot))  # the slot's warp saw the stale copy land, then refills it
            continue
        w = rnd.choice(busy)
        k = todo[w][pos[w]]
        slot = k % R
        parity = (k // R + sh[slot]) & 1
        if completed[slot] % 2 != parity:
            if content[slot] != k:
                return "wrong tile"
            pos[w] += 1
            cons[slot] += 1
            if cons[slot] == WQ:
                cons[slot] = 0
                if k + R < ntile:
                    inflight.append((slot, k + R))
    return "hang"


def test_stale_early_copies_shift_the_slot_phase():
    """Any set of slots may hold a stale early copy (each warp decides for its own slot); with the phase
    shift every tile is still read once and in order, without it a consumer reads the stale copy."""
    rnd = random.Random(7)
    for ntile in range(1, 17):
        for S in range(1, 9):
            for WQ in (1, 2, 4, 8):
                for seed in range(4):
                    stale = {s for s in range(S) if rnd.random() < 0.5}
                    assert replay_early(ntile, S, WQ, stale, True, seed) == "ok", (ntile, S, WQ, stale, seed)
    bad = sum(replay_early(6, 4, 2, {0, 1}, False, seed) != "ok" for seed in range(20))
    assert bad > 0


@pytest.mark.parametrize("WQ", [1, 2, 4, 8])
def test_ring_rule_reads_every_tile_once_and_in_order(WQ):
    for ntile in range(1, 21):
        for S in range(1, 9):
            for seed in range(8):
                assert replay(ntile, S, WQ, True, seed) == "ok", (ntile, S, WQ, seed)


def test_model_sees_the_hazard_of_mixed_consumers():
    bad = sum(replay(10, 6, 1, False, seed) != "ok" for seed in range(20))
    assert bad > 0


def test_library_ring_rule_shapes():
    """No refill: all S slots, every warp set.  With refills: R <= S slots and WK warp sets, R % WK == 0, and no
    R' <= S with a divisor WK' <= 16 / WQ larger than WK (the rule takes the most warp sets)."""
    for S in range(1, 9):
        for WQ in (1, 2, 4, 8):
            wmax = K_WARPS // WQ
            for ntile in range(1, 24):
                R, WK = ring_rule(ntile, S, WQ)
                if ntile <= S:
                    assert (R, WK) == (S, wmax)
                    continue
                assert 1 <= R <= S and 1 <= WK <= wmax and R % WK == 0
                best = max(max(w for w in range(1, min(wmax, r) + 1) if r % w == 0) for r in range(1, S + 1))
                assert WK == best
