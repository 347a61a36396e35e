"""Decoder forward of the oracle: a Llama-style pre-norm transformer in float64.

The pages never write the model out; they say the draft is the target model
itself with some transformer layers skipped ([CAS-blog] §2.1, [CLaSp] §二)
and that verification is one full-model pass ([CLaSp] §三).  The model
family is LLaMA ([CLaSp] §四, §五).  The plain reading, per layer i:

    a   = RMSNorm(h) * g_attn             RMSNorm(x) = x / sqrt(mean(x^2) + eps)
    q,k,v = Wq a, Wk a, Wv a              RoPE (rotate-half) on q, k at the row's position
    o   = softmax(q K^T / sqrt(hd) + mask) V     per head; GQA: kv head = q head // (Hq/Hkv)
    h  += Wo o
    b   = RMSNorm(h) * g_ffn
    h  += Wd (SiLU(Wg b) * (Wu b))        SiLU(x) = x / (1 + exp(-x))

then logits = W_lm (RMSNorm(h) * g_final).  A skipped layer leaves h
unchanged and writes no KV ([CAS-blog] §2.1 item 1: whole layers skipped).
With act_int8 the inputs of the seven projections (a, o, b, SiLU*up) pass
through quant.fake_quant_rows ([CAS-blog] §2.1 item 3).

KV cache: one float64 K and V array [slots, Hkv, hd] per layer.  K is kept
after RoPE.  Visibility of slots is an explicit boolean matrix per call.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

import ssd_inputs as si

from .quant import fake_quant_rows


class Weights:
    """The seeded weight set, held as 16-bit bits and widened on use.

    compute = "f64" (default): matrices widened to float64, every product in
    float64.  compute = "f32": matrices widened to float32 (exact: every
    16-bit value is a float32) and each projection's product taken in float32
    (BLAS sgemm) then widened back; everything else (RMSNorm, RoPE, attention,
    SwiGLU, residuals, int8 codes) stays float64.  The float32 mode exists for
    the full-size workloads, whose float64 weights would not fit in memory;
    its products differ from float64 by float32 rounding of dot products
    (relative ~1e-6), far inside the GPU tolerances.
    """

    def __init__(self, cfg: si.ModelConfig, keep_bits: bool = True, cache_bytes: int = 6 << 30,
                 compute: str = "f64", evict: bool = True):
        assert compute in ("f64", "f32")
        self.cfg = cfg
        self.keep_bits = keep_bits
        self.compute = compute
        self._mat = np.float32 if compute == "f32" else np.float64
        self._bits: Dict[tuple, np.ndarray] = {}
        self._f64: Dict[int, Dict[str, np.ndarray]] = {}
        self._order: List[int] = []
        self._cache_bytes = cache_bytes
        self._evict = evict  # False: layers that do not fit are widened again on every use (no LRU thrash)
        self._lm32: Optional[np.ndarray] = None
        g = {s.name: s for s in si.global_specs(cfg)}
        self._gspec = g
        self.final_norm = self._widen(g["final_norm"])
        self._embed_bits = si.host_values(g["embed"], cfg)

    def _widen(self, spec: si.TensorSpec) -> np.ndarray:
        return si.widen(si.host_values(spec, self.cfg), self.cfg.dtype)

    def embed(self, tokens: Sequence[int]) -> np.ndarray:
        return si.widen(self._embed_bits[np.asarray(tokens, dtype=np.int64)], self.cfg.dtype)

    def layer(self, i: int) -> Dict[str, np.ndarray]:
        if i in self._f64:
            return self._f64[i]
        out = {}
        for spec in si.layer_specs(self.cfg, i):
            key = (i, spec.name)
            if self.keep_bits:
                if key not in self._bits:
                    self._bits[key] = si.host_values(spec, self.cfg)
                bits = self._bits[key]
            else:
                bits = si.host_values(spec, self.cfg)
            # gains stay float64 (RMSNorm is float64 in both modes); matrices in the compute type
            dt = np.float64 if len(spec.shape) == 1 else self._mat
            out[spec.name] = si.widen(bits, self.cfg.dtype, dt)
        nbytes = sum(v.nbytes for v in out.values())
        while self._evict and self._order and (len(self._order) + 1) * nbytes > self._cache_bytes:
            self._f64.pop(self._order.pop(0))
        if (len(self._order) + 1) * nbytes <= self._cache_bytes:
            self._f64[i] = out
            self._order.append(i)
        return out

    def logits(self, x: np.ndarray, rows_per_chunk: int = 16384) -> np.ndarray:
        """W_lm x^T for x [R, d] (already normalised), lm_head widened chunk by chunk."""
        spec = self._gspec["lm_head"]
        V, d = spec.shape
        if self.compute == "f32":  # the whole matrix widened once to float32 and kept
            if self._lm32 is None:
                self._lm32 = si.widen(si.host_values(spec, self.cfg), self.cfg.dtype, np.float32).reshape(V, d)
            return proj(x, self._lm32)
        key = ("lm_head",)
        if self.keep_bits and key not in self._bits:
            self._bits[key] = si.host_values(spec, self.cfg)
        out = np.empty((x.shape[0], V), dtype=np.float64)
        for r0 in range(0, V, rows_per_chunk):
            r1 = min(V, r0 + rows_per_chunk)
            if self.keep_bits:
                bits = self._bits[key][r0:r1]
            else:
                bits = si.host_values(spec, self.cfg, offset=r0 * d, count=(r1 - r0) * d).reshape(r1 - r0, d)
            out[:, r0:r1] = x @ si.widen(bits, self.cfg.dtype).T
        return out


class ArrayWeights:
    """A weight set given as float64 arrays (hand-built models for the oracle's own pins)."""

    def __init__(self, cfg: si.ModelConfig, embed: np.ndarray, lm_head: np.ndarray, final_norm: np.ndarray,
                 layers: List[Dict[str, np.ndarray]]):
        self.cfg = cfg
        self._embed = np.asarray(embed, dtype=np.float64)
        self._lm = np.asarray(lm_head, dtype=np.float64)
        self.final_norm = np.asarray(final_norm, dtype=np.float64)
        self._layers = layers

    def embed(self, tokens: Sequence[int]) -> np.ndarray:
        return self._embed[np.asarray(tokens, dtype=np.int64)]

    def layer(self, i: int) -> Dict[str, np.ndarray]:
        return self._layers[i]

    def logits(self, x: np.ndarray) -> np.ndarray:
        return x @ self._lm.T


class KVCache:
    """K, V float64 [max_ctx, Hkv, hd] per layer."""

    def __init__(self, cfg: si.ModelConfig, max_ctx: Optional[int] = None):
        n = cfg.max_ctx if max_ctx is None else max_ctx
        shape = (n, cfg.n_kv_heads, cfg.head_dim)
        self.k = [np.zeros(shape) for _ in range(cfg.n_layers)]
        self.v = [np.zeros(shape) for _ in range(cfg.n_layers)]

    def copy_slot(self, dst: int, src: int) -> None:
        for i in range(len(self.k)):
            self.k[i][dst] = self.k[i][src]
            self.v[i][dst] = self.v[i][src]


def proj(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """x [R, K] times w [N, K] transposed: float64, or a float32 product for float32 weights (widened back)."""
    if w.dtype == np.float32:
        return (np.asarray(x, dtype=np.float64).astype(np.float32) @ w.T).astype(np.float64)
    return x @ w.T


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * gamma


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, positions: np.ndarray, base: float) -> np.ndarray:
    """Rotate-half RoPE on x [R, H, hd]: pairs (k, k + hd/2), angle pos * base^(-2k/hd)."""
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = base ** (-(np.arange(half, dtype=np.float64) * 2.0) / hd)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos, sin = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def attention(q: np.ndarray, keys: np.ndarray, vals: np.ndarray, vis: np.ndarray) -> np.ndarray:
    """q [R, Hq, hd]; keys/vals [S, Hkv, hd]; vis bool [R, S] -> o [R, Hq, hd]."""
    R, Hq, hd = q.shape
    group = Hq // keys.shape[1]
    o = np.zeros_like(q)
    scale = 1.0 / math.sqrt(hd)
    for h in range(Hq):
        kv = h // group
        s = (q[:, h, :] @ keys[:, kv, :].T) * scale
        s = np.where(vis, s, -np.inf)
        s = s - np.max(s, axis=1, keepdims=True)
        p = np.exp(s)
        p = p / np.sum(p, axis=1, keepdims=True)
        o[:, h, :] = p @ vals[:, kv, :]
    return o


def layer_forward(cfg: si.ModelConfig, W: Dict[str, np.ndarray], K: np.ndarray, V: np.ndarray, h: np.ndarray,
                  positions: np.ndarray, slots: Optional[np.ndarray], vis: np.ndarray, act_int8: bool) -> np.ndarray:
    """One transformer block on rows h [R, d].

    slots: cache slot of each row's K/V (written before attention), or None:
    then each row's K/V stay local (never written) and are appended as extra
    key columns R..; `vis` [R, S] covers cache slots 0..S-1 (+ R local
    columns when slots is None).
    """
    R = h.shape[0]
    Hq, Hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    q8 = fake_quant_rows if act_int8 else (lambda x: x)
    a = q8(rmsnorm(h, W["g_attn"], cfg.rms_eps))
    q = proj(a, W["wq"]).reshape(R, Hq, hd)
    k = proj(a, W["wk"]).reshape(R, Hkv, hd)
    v = proj(a, W["wv"]).reshape(R, Hkv, hd)
    q = rope(q, positions, cfg.rope_base)
    k = rope(k, positions, cfg.rope_base)
    if slots is not None:
        K[slots] = k
        V[slots] = v
        S = vis.shape[1]
        keys, vals = K[:S], V[:S]
    else:
        S = vis.shape[1] - R
        keys = np.concatenate([K[:S], k], axis=0)
        vals = np.concatenate([V[:S], v], axis=0)
    o = attention(q, keys, vals, vis).reshape(R, Hq * hd)
    h = h + proj(q8(o), W["wo"])
    b = q8(rmsnorm(h, W["g_ffn"], cfg.rms_eps))
    act = silu(proj(b, W["wg"])) * proj(b, W["wu"])
    return h + proj(q8(act), W["wd"])


def forward(Wt: Weights, cache: KVCache, tokens: Sequence[int], positions: Sequence[int],
            slots: Optional[Sequence[int]], vis: np.ndarray, skip: Sequence[int] = (), act_int8: bool = False,
            with_logits: bool = True, h0: Optional[np.ndarray] = None, exit_layers: int = 0):
    """Run the decoder on rows (tokens at positions).

    exit_layers = e: early exit ([CAS-blog] §2.1 item 2, §2.2 L1): the forward
    ends after layer L - e - 1 and the final norm + lm_head read the residual
    there; the last e layers run nothing and write no KV.

    Returns (logits [R, V] or None, states) where states[i] is the residual
    stream after i layers, i = 0..L (states[0] = embedding; after an early
    exit the later entries repeat the exit residual).
    """
    cfg = Wt.cfg
    h = Wt.embed(tokens) if h0 is None else np.array(h0, dtype=np.float64)
    pos = np.asarray(positions, dtype=np.int64)
    sl = None if slots is None else np.asarray(slots, dtype=np.int64)
    skip = set(int(i) for i in skip)
    states = [h]
    for i in range(cfg.n_layers - exit_layers):
        if i not in skip:
            h = layer_forward(cfg, Wt.layer(i), cache.k[i], cache.v[i], h, pos, sl, vis, act_int8)
        states.append(h)
    states += [h] * exit_layers
    logits = Wt.logits(rmsnorm(h, Wt.final_norm, cfg.rms_eps)) if with_logits else None
    return logits, states


def causal_vis(t: int, n_new: int, width: Optional[int] = None) -> np.ndarray:
    """Rows t..t+n_new-1 in slots t..: row r sees slots [0, t + r]."""
    S = t + n_new if width is None else width
    vis = np.zeros((n_new, S), dtype=bool)
    for r in range(n_new):
        vis[r, : t + r + 1] = True
    return vis


def argmax_f32(logits: np.ndarray) -> np.ndarray:
    """Greedy token per row, decided on float32 logits; ties go to the lowest token id."""
    return np.argmax(np.asarray(logits).astype(np.float32), axis=-1)


def top2_f32(logits_row: np.ndarray):
    """(top-1 id, top-2 id) on float32 logits, ordered by value then by lower id."""
    x = np.asarray(logits_row).astype(np.float32)
    order = np.lexsort((np.arange(x.size), -x))
    return int(order[0]), int(order[1])


def top_gap(logits_row: np.ndarray) -> float:
    """top-1 minus top-2 logit (float64): the near-tie measure."""
    x = np.sort(np.asarray(logits_row, dtype=np.float64))
    return float(x[-1] - x[-2])


def top1_prob(logits_row: np.ndarray) -> float:
    """Softmax probability of the greedy token: 1 / sum_i exp(x_i - max x), float64 over the float32 logits.

    This is the draft's confidence that the draft exit threshold is compared with
    ([CLaSp] §四, the draft exit threshold, best near 0.7)."""
    x = np.asarray(logits_row).astype(np.float32).astype(np.float64)
    return float(1.0 / np.sum(np.exp(x - x.max())))
