"""Seeded attention cases shared by the kernel-level GPU tests (not collected as tests)."""
import ctypes

import numpy as np

from oracle import model

ATTN_TOL = 1e-4  # fp32 kernel arithmetic on the same 16-bit K/V values as the oracle

# (name, rows, prefix, base, mask kind, Hq, Hkv, hd, dtype)
CASES = [
    ("decode_gqa", 1, 700, 700, "causal", 32, 8, 128, "bf16"),
    ("verify7_gqa", 7, 301, 301, "causal", 32, 8, 128, "bf16"),
    ("tree17_gqa", 17, 259, 259, "tree", 32, 8, 128, "bf16"),
    ("dp_rows", 5, 200, 413, "own", 16, 2, 128, "bf16"),
    ("prefill64", 64, 128, 128, "causal", 8, 8, 64, "bf16"),
    ("mha_fp16", 9, 77, 77, "causal", 10, 10, 128, "fp16"),
    ("empty_prefix", 3, 0, 0, "causal", 4, 4, 64, "fp16"),
    ("verify9_fp32_cache", 9, 640, 640, "causal", 64, 8, 128, "fp32"),
    # long contexts: a CTA's key tiles outnumber its ring slots, so slots are refilled
    ("decode_long_fp32", 1, 2400, 2400, "causal", 64, 8, 128, "fp32"),
    ("verify7_long_bf16", 7, 3000, 3000, "causal", 32, 8, 128, "bf16"),
    ("dp17_long_fp32", 17, 1500, 1600, "own", 32, 8, 128, "fp32"),
    # one query per warp (query blocks of at most four) with refilled rings
    ("decode_long_mqa_fp32", 1, 3000, 3000, "causal", 4, 1, 128, "fp32"),
    ("decode_long_mha_fp16", 1, 2000, 2000, "causal", 8, 8, 128, "fp16"),
    ("verify3_long_mha_bf16", 3, 2500, 2500, "causal", 6, 6, 64, "bf16"),
    # new slots continuing the prefix (tiled together with it): across a page boundary, from a tile
    # boundary, and in the last slot of a page
    ("verify7_page_cross_fp32", 7, 60, 60, "causal", 32, 8, 128, "fp32"),
    ("tree9_tile_edge_bf16", 9, 96, 96, "tree", 16, 4, 128, "bf16"),
    ("draft_page_end_fp32", 1, 63, 63, "causal", 8, 8, 128, "fp32"),
]


def masks(kind, rows, rng):
    if kind == "causal":
        return [(1 << (r + 1)) - 1 for r in range(rows)]
    if kind == "own":
        return [1 << r for r in range(rows)]
    parents = [-1] + [int(rng.integers(0, c)) for c in range(1, rows)]
    anc = []
    for c in range(rows):
        anc.append((anc[parents[c]] if c else 0) | (1 << c))
    return anc


def make_case(case, seed=0):
    """Host arrays of one case: q, K/V of every slot, paged caches, visibility matrix."""
    import torch

    name, rows, prefix, base, kind, hq, hkv, hd, dtype = case
    rng = np.random.default_rng(seed)
    n_slots = max(prefix, base + rows)
    n_pages = (n_slots + 63) // 64 + 2
    n_layers, layer = 2, 1
    tdt = {"fp16": torch.float16, "bf16": torch.bfloat16, "fp32": torch.float32}[dtype]
    k = torch.tensor(rng.standard_normal((n_slots, hkv, hd)), dtype=torch.float32).to(tdt)
    v = torch.tensor(rng.standard_normal((n_slots, hkv, hd)), dtype=torch.float32).to(tdt)
    q = (rng.standard_normal((rows, hq, hd)) * 0.5).astype(np.float32)
    perm = rng.permutation(n_pages).astype(np.int32)
    kc = torch.zeros((n_layers, n_pages, hkv, 64, hd), dtype=tdt)
    vc = torch.zeros_like(kc)
    for s in range(n_slots):
        kc[layer, perm[s // 64], :, s % 64, :] = k[s]
        vc[layer, perm[s // 64], :, s % 64, :] = v[s]
    m = masks(kind, rows, rng)
    vis = np.zeros((rows, n_slots), dtype=bool)
    for r in range(rows):
        vis[r, :prefix] = True
        for e in range(rows):
            if (m[r] >> e) & 1:
                vis[r, base + e] = True
    want = model.attention(q.astype(np.float64), k.double().numpy(), v.double().numpy(), vis)
    return dict(q=q, kc=kc, vc=vc, perm=perm, n_pages=n_pages, layer=layer, rows=rows, prefix=prefix, base=base,
                masks=m, hq=hq, hkv=hkv, hd=hd, dtype=dtype, want=want.reshape(rows, hq * hd))


def device_args(c):
    """(args struct, tensors to keep alive, output tensor) for a case on cuda."""
    import torch

    import self_speculative_decoding_layer_gb300 as ssd

    q = torch.tensor(c["q"].reshape(c["rows"], -1)).cuda()
    kc, vc = c["kc"].cuda(), c["vc"].cuda()
    bt = torch.tensor(c["perm"]).cuda()
    out = torch.full((c["rows"], c["hq"] * c["hd"]), float("nan"), dtype=torch.float32, device="cuda")
    a = ssd.AttentionArgsC()
    a.q, a.k_cache, a.v_cache, a.block_table, a.out = q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), \
        out.data_ptr()
    a.n_pages, a.layer, a.n_q_heads, a.n_kv_heads, a.head_dim = c["n_pages"], c["layer"], c["hq"], c["hkv"], c["hd"]
    a.dtype = {"bf16": 0, "fp16": 1, "fp32": 2}[c["dtype"]]
    a.rows, a.prefix, a.base = c["rows"], c["prefix"], c["base"]
    for r, mk in enumerate(c["masks"]):
        a.mask[r] = mk
    return a, (q, kc, vc, bt), out
