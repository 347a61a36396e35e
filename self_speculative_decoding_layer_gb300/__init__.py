"""Python binding of libssd.so (GB300 self-speculative decoding hot path).

Argument marshalling only: every step of drafting, verification,
acceptance and the CLaSp search runs in the library's CUDA kernels.  PyTorch
provides device memory (weights, workspace) and the CUDA stream.  If the
library is not built the import of `Engine` fails loudly; there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libssd.so")
# the test library: the same code with the cross-check kernels compiled in (SSD_OPT_GEMM_IMPL 1..3)
XCHECK_LIB_PATH = os.path.join(_HERE, "lib", "libssd_xcheck.so")

SSD_OK = 0
STATUS = {0: "ok", 1: "invalid argument", 2: "call out of order", 3: "capacity exceeded", 4: "host out of memory",
          5: "CUDA error", 6: "device wait timed out"}
POLICY_STATIC, POLICY_CLASP, POLICY_DYTC, POLICY_AR, POLICY_HCASCADE, POLICY_VCASCADE = 0, 1, 2, 3, 4, 5
OPT_GEMM_IMPL, OPT_USE_GRAPHS, OPT_TIMING, OPT_PDL, OPT_L2_PREFETCH_MB, OPT_TRACE, OPT_CYCLE_LOG = 0, 1, 2, 3, 4, 5, 6

EXPORTS = ("ssd_workspace_bytes", "ssd_create", "ssd_weight_count", "ssd_load_weights", "ssd_prefill",
           "ssd_decode_ar", "ssd_draft", "ssd_verify", "ssd_rollback", "ssd_dp_select", "ssd_generate",
           "ssd_draft_tree", "ssd_get_logits", "ssd_get_hidden", "ssd_get_position", "ssd_get_stats",
           "ssd_reset_stats", "ssd_set_option", "ssd_get_pass_times", "ssd_last_error", "ssd_status_string",
           "ssd_destroy", "ssd_attention_scratch_bytes", "ssd_attention", "ssd_get_trace", "ssd_get_draft_conf",
           "ssd_calibrate_latency", "ssd_set_latency_model", "ssd_fit_latency", "ssd_get_level_costs",
           "ssd_cascade_depth", "ssd_plan_tree", "ssd_plan_hcascade", "ssd_abi_sizes", "ssd_attention_noalloc",
           "ssd_get_cycle_log", "ssd_set_ema", "ssd_get_dp_table", "ssd_streamk_split",
           "ssd_gemv_warps", "ssd_attn_ring_rule")


class ModelConfigC(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("dtype", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("rope_base", ctypes.c_float), ("max_ctx", ctypes.c_int), ("max_rows", ctypes.c_int)]


class PolicyC(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("draft_k", ctypes.c_int), ("act_int8", ctypes.c_int),
                ("skip_mask", ctypes.POINTER(ctypes.c_uint8)), ("dp_n_skip", ctypes.c_int),
                ("dp_interval", ctypes.c_int), ("dp_at_start", ctypes.c_int), ("n_levels", ctypes.c_int),
                ("level_skip", ctypes.POINTER(ctypes.c_uint8)), ("level_int8", ctypes.POINTER(ctypes.c_int32)),
                ("ema_alpha", ctypes.c_double), ("ema_init", ctypes.c_double), ("tree_max_nodes", ctypes.c_int),
                ("tree_max_depth", ctypes.c_int), ("draft_exit", ctypes.c_double), ("early_exit", ctypes.c_int),
                ("level_exit", ctypes.POINTER(ctypes.c_int32)), ("cost_model", ctypes.c_int),
                ("cascade_rules", ctypes.c_int), ("hc_len", ctypes.POINTER(ctypes.c_int32)), ("vc_lo", ctypes.c_int),
                ("vc_hi", ctypes.c_int)]


class AttentionArgsC(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("out", ctypes.c_void_p), ("n_pages", ctypes.c_int),
                ("layer", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int), ("rows", ctypes.c_int),
                ("prefix", ctypes.c_int), ("base", ctypes.c_int), ("mask", ctypes.c_uint64 * 64)]


class StatsC(ctypes.Structure):
    _fields_ = [("cycles", ctypes.c_int64), ("drafted", ctypes.c_int64), ("accepted", ctypes.c_int64),
                ("generated", ctypes.c_int64), ("dp_runs", ctypes.c_int64), ("ar_steps", ctypes.c_int64),
                ("accept_hist", ctypes.c_int64 * 65), ("ema", ctypes.c_double * 3),
                ("kernel_launches", ctypes.c_int64), ("mma_fallbacks", ctypes.c_int64)]


class CycleRecordC(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("t", ctypes.c_int32), ("n_rows", ctypes.c_int32),
                ("n_acc", ctypes.c_int32), ("bonus", ctypes.c_int32), ("tokens", ctypes.c_int32 * 64),
                ("parents", ctypes.c_int32 * 64), ("argmax", ctypes.c_int32 * 64), ("path", ctypes.c_int32 * 65),
                ("mask", ctypes.c_uint8 * 128), ("dp_value", ctypes.c_float), ("ema", ctypes.c_double * 3)]


_libs = {}


def load_library(xcheck: bool = False) -> ctypes.CDLL:
    """Load libssd.so, or with xcheck the test library libssd_xcheck.so (raises if it has not been built)."""
    if xcheck in _libs:
        return _libs[xcheck]
    path = XCHECK_LIB_PATH if xcheck else LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    P, I, U8P, I32P = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_int32)
    DP = ctypes.POINTER(ctypes.c_double)
    cfgp = ctypes.POINTER(ModelConfigC)
    sig = {
        "ssd_workspace_bytes": (ctypes.c_size_t, [cfgp]),
        "ssd_create": (I, [cfgp, P, ctypes.c_size_t, P, ctypes.POINTER(P)]),
        "ssd_weight_count": (I, [cfgp]),
        "ssd_load_weights": (I, [P, ctypes.POINTER(P), I]),
        "ssd_prefill": (I, [P, I32P, I, I32P]),
        "ssd_decode_ar": (I, [P, I, I32P]),
        "ssd_draft": (I, [P, U8P, I, I, ctypes.c_float, I32P, I32P]),
        "ssd_verify": (I, [P, I32P, I32P, I, I32P, I32P, I32P]),
        "ssd_rollback": (I, [P, I, ctypes.c_int32]),
        "ssd_dp_select": (I, [P, I, U8P, ctypes.POINTER(ctypes.c_float)]),
        "ssd_generate": (I, [P, ctypes.POINTER(PolicyC), I, I32P]),
        "ssd_draft_tree": (I, [P, ctypes.POINTER(PolicyC), I32P, I32P, ctypes.POINTER(ctypes.c_int)]),
        "ssd_get_logits": (I, [P, I, ctypes.POINTER(ctypes.c_float)]),
        "ssd_get_draft_conf": (I, [P, I, ctypes.POINTER(ctypes.c_float)]),
        "ssd_calibrate_latency": (I, [P, I, I32P, I, I32P, I, I, U8P, DP, DP]),
        "ssd_set_latency_model": (I, [P, I, DP]),
        "ssd_fit_latency": (I, [I, DP, DP, DP, DP]),
        "ssd_get_level_costs": (I, [P, ctypes.POINTER(PolicyC), DP, ctypes.POINTER(ctypes.c_int)]),
        "ssd_cascade_depth": (I, [I, I, I]),
        "ssd_abi_sizes": (None, [ctypes.POINTER(ctypes.c_size_t), I]),
        "ssd_plan_tree": (I, [I, DP, DP, I, I, I32P, ctypes.POINTER(ctypes.c_int), I32P, I32P,
                              ctypes.POINTER(ctypes.c_int)]),
        "ssd_plan_hcascade": (I, [I, I32P, I32P, ctypes.POINTER(ctypes.c_int), I32P, I32P,
                                  ctypes.POINTER(ctypes.c_int)]),
        "ssd_get_hidden": (I, [P, I, I, ctypes.POINTER(ctypes.c_float)]),
        "ssd_get_position": (I, [P, I32P, I32P]),
        "ssd_get_stats": (I, [P, ctypes.POINTER(StatsC)]),
        "ssd_reset_stats": (I, [P]),
        "ssd_set_option": (I, [P, I, I]),
        "ssd_get_pass_times": (I, [P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]),
        "ssd_last_error": (ctypes.c_char_p, [P]),
        "ssd_status_string": (ctypes.c_char_p, [I]),
        "ssd_destroy": (None, [P]),
        "ssd_attention_scratch_bytes": (ctypes.c_size_t, [I, I, I, I]),
        "ssd_attention": (I, [ctypes.POINTER(AttentionArgsC), P, ctypes.c_size_t, P]),
        "ssd_get_trace": (I, [P, ctypes.POINTER(ctypes.c_int64), I, ctypes.POINTER(ctypes.c_int)]),
        "ssd_attention_noalloc": (I, [ctypes.POINTER(AttentionArgsC), P]),
        "ssd_get_cycle_log": (I, [P, ctypes.POINTER(CycleRecordC), I, ctypes.POINTER(ctypes.c_int)]),
        "ssd_set_ema": (I, [P, DP, I]),
        "ssd_get_dp_table": (I, [P, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float), U8P]),
        "ssd_streamk_split": (None, [ctypes.c_int64, I, I, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64),
                                     ctypes.POINTER(ctypes.c_int)]),
        "ssd_gemv_warps": (ctypes.c_int64, [I, ctypes.c_int64]),
        "ssd_attn_ring_rule": (None, [I, I, I, ctypes.POINTER(I), ctypes.POINTER(I)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _libs[xcheck] = lib
    return lib


class SSDError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def fit_latency(seq_len: Sequence[float], depth: Sequence[float], ms: Sequence[float]) -> np.ndarray:
    """Least-squares latency model beta (ms = b0 + b1 * seq_len + b2 * depth), computed by the library."""
    s, d, y = (np.ascontiguousarray(np.asarray(v, dtype=np.float64)) for v in (seq_len, depth, ms))
    beta = np.zeros(3, dtype=np.float64)
    st = load_library().ssd_fit_latency(s.size, _p(s, ctypes.c_double), _p(d, ctypes.c_double),
                                        _p(y, ctypes.c_double), _p(beta, ctypes.c_double))
    if st != SSD_OK:
        raise SSDError(st, "the points do not determine the latency model")
    return beta


def cascade_depth(n_layers: int, n_levels: int, seq_len: int) -> int:
    return int(load_library().ssd_cascade_depth(n_layers, n_levels, seq_len))


def _plan_out(fn, *args):
    par, en, el = (np.zeros(64, dtype=np.int32) for _ in range(3))
    nn, ne = ctypes.c_int(), ctypes.c_int()
    st = fn(*args, _p(par, ctypes.c_int32), ctypes.byref(nn), _p(en, ctypes.c_int32), _p(el, ctypes.c_int32),
            ctypes.byref(ne))
    if st != SSD_OK:
        raise SSDError(st, "planner arguments rejected")
    return par[: nn.value].tolist(), list(zip(en[: ne.value].tolist(), el[: ne.value].tolist()))


def plan_tree(ema: Sequence[float], cost: Sequence[float], max_nodes: int, max_depth: int):
    """The library's DyTC plan: (parents, [(node, level), ...])."""
    a = np.ascontiguousarray(np.asarray(ema, dtype=np.float64))
    c = np.ascontiguousarray(np.asarray(cost, dtype=np.float64))
    return _plan_out(load_library().ssd_plan_tree, a.size, _p(a, ctypes.c_double), _p(c, ctypes.c_double),
                     max_nodes, max_depth)


def plan_hcascade(hc_len: Sequence[int]):
    """The library's horizontal-cascade chain: (parents, [(node, level), ...])."""
    h = _i32(hc_len)
    return _plan_out(load_library().ssd_plan_hcascade, h.size, _p(h, ctypes.c_int32))


def c_config(cfg, max_ctx: Optional[int] = None, max_rows: int = 64) -> ModelConfigC:
    """ssd_model_config from an ssd_inputs.ModelConfig."""
    return ModelConfigC(cfg.n_layers, cfg.d_model, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn, cfg.vocab,
                        1 if cfg.dtype == "fp16" else 0, cfg.rms_eps, cfg.rope_base,
                        cfg.max_ctx if max_ctx is None else max_ctx, max_rows)


class DeviceWeights:
    """Weights of one model in the library's fused layout, in torch device memory."""

    def __init__(self, cfg, device="cuda", fill: bool = True):
        import torch

        import ssd_inputs as si

        self.cfg = cfg
        dt = torch.float16 if cfg.dtype == "fp16" else torch.bfloat16
        d, F, hd = cfg.d_model, cfg.ffn, cfg.head_dim
        g = {s.name: s for s in si.global_specs(cfg)}
        self.tensors: List["torch.Tensor"] = []
        self.embed = torch.empty((cfg.vocab, d), dtype=dt, device=device)
        self.final_norm = torch.empty((d,), dtype=dt, device=device)
        self.lm_head = torch.empty((cfg.vocab, d), dtype=dt, device=device)
        self.tensors += [self.embed, self.final_norm, self.lm_head]
        fills = [(self.embed, 0, g["embed"]), (self.final_norm, 0, g["final_norm"]), (self.lm_head, 0, g["lm_head"])]
        for i in range(cfg.n_layers):
            s = {x.name: x for x in si.layer_specs(cfg, i)}
            qkv = torch.empty((cfg.qkv_rows, d), dtype=dt, device=device)
            wo = torch.empty((d, cfg.n_q_heads * hd), dtype=dt, device=device)
            gu = torch.empty((2 * F, d), dtype=dt, device=device)
            wd = torch.empty((d, F), dtype=dt, device=device)
            ga = torch.empty((d,), dtype=dt, device=device)
            gf = torch.empty((d,), dtype=dt, device=device)
            self.tensors += [qkv, wo, gu, wd, ga, gf]
            nq, nk = cfg.n_q_heads * hd * d, cfg.n_kv_heads * hd * d
            fills += [(qkv, 0, s["wq"]), (qkv, nq, s["wk"]), (qkv, nq + nk, s["wv"]), (wo, 0, s["wo"]),
                      (gu, 0, s["wg"]), (gu, F * d, s["wu"]), (wd, 0, s["wd"]), (ga, 0, s["g_attn"]),
                      (gf, 0, s["g_ffn"])]
        if fill:
            for t, elem_off, spec in fills:
                si.fill_device(t.data_ptr() + 2 * elem_off, spec, cfg)
            torch.cuda.synchronize()

    def pointers(self):
        return [t.data_ptr() for t in self.tensors]


class Engine:
    """One decoding context (batch 1) over the C ABI."""

    def __init__(self, cfg, weights: Optional[DeviceWeights] = None, max_ctx: Optional[int] = None,
                 max_rows: int = 64, stream=None, xcheck: bool = False):
        """xcheck: run on the test library (cross-check kernels selectable with OPT_GEMM_IMPL)."""
        import torch

        self.lib = load_library(xcheck)
        self.cfg = cfg
        self.ccfg = c_config(cfg, max_ctx, max_rows)
        nbytes = self.lib.ssd_workspace_bytes(ctypes.byref(self.ccfg))
        if nbytes == 0:
            raise SSDError(1, "invalid model config")
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda")
        ptr = (self.workspace.data_ptr() + 255) // 256 * 256
        self.ctx = ctypes.c_void_p()
        rc = self.lib.ssd_create(ctypes.byref(self.ccfg), ptr, nbytes, self.stream.cuda_stream,
                                 ctypes.byref(self.ctx))
        if rc != SSD_OK:
            raise SSDError(rc, "ssd_create failed")
        self.weights = weights
        if weights is not None:
            self.load_weights(weights)

    # -- plumbing
    def _check(self, rc: int):
        if rc != SSD_OK:
            raise SSDError(rc, self.lib.ssd_last_error(self.ctx).decode())

    def close(self):
        if getattr(self, "ctx", None) is not None and self.ctx.value:
            self.lib.ssd_destroy(self.ctx)
            self.ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- API
    def load_weights(self, w: DeviceWeights):
        ptrs = w.pointers()
        arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
        self._check(self.lib.ssd_load_weights(self.ctx, arr, len(ptrs)))
        self.weights = w

    def set_option(self, opt: int, value: int):
        self._check(self.lib.ssd_set_option(self.ctx, opt, value))

    def prefill(self, tokens: Sequence[int]) -> int:
        t = _i32(tokens)
        nxt = ctypes.c_int32()
        self._check(self.lib.ssd_prefill(self.ctx, _p(t, ctypes.c_int32), t.size, ctypes.byref(nxt)))
        return nxt.value

    def decode_ar(self, n: int) -> List[int]:
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._check(self.lib.ssd_decode_ar(self.ctx, n, _p(out, ctypes.c_int32)))
        return out[:n].tolist()

    def draft(self, skip: Sequence[int], k: int, act_int8: bool = False, exit_thr: float = 0.0,
              early_exit: int = 0) -> List[int]:
        """Up to k drafts; with exit_thr > 0 drafting ends after the first draft whose top-1
        probability is below exit_thr (that draft kept).  early_exit = e: the draft model also
        stops e layers before the end (the last e layers added to the mask)."""
        m = np.zeros(self.cfg.n_layers, dtype=np.uint8)
        m[list(skip)] = 1
        if early_exit:
            m[self.cfg.n_layers - early_exit:] = 1
        out = np.zeros(k, dtype=np.int32)
        n = ctypes.c_int32()
        self._check(self.lib.ssd_draft(self.ctx, _p(m, ctypes.c_uint8), int(act_int8), k, float(exit_thr),
                                       _p(out, ctypes.c_int32), ctypes.byref(n)))
        return out[: n.value].tolist()

    def draft_conf(self, n: int) -> List[float]:
        """Top-1 probabilities of the first n drafts of the last exit-enabled draft pass."""
        out = np.zeros(n, dtype=np.float32)
        self._check(self.lib.ssd_get_draft_conf(self.ctx, n, _p(out, ctypes.c_float)))
        return out.tolist()

    def verify(self, tokens: Sequence[int], parents: Optional[Sequence[int]] = None):
        t = _i32(tokens)
        par = None if parents is None else _i32(parents)
        n_acc, bonus = ctypes.c_int32(), ctypes.c_int32()
        path = np.zeros(t.size + 1, dtype=np.int32)
        self._check(self.lib.ssd_verify(self.ctx, _p(t, ctypes.c_int32),
                                        None if par is None else _p(par, ctypes.c_int32), t.size,
                                        ctypes.byref(n_acc), _p(path, ctypes.c_int32), ctypes.byref(bonus)))
        return n_acc.value, path[: n_acc.value + 1].tolist(), bonus.value

    def rollback(self, new_len: int, pending: int = -1):
        self._check(self.lib.ssd_rollback(self.ctx, new_len, pending))

    def dp_select(self, n_skip: int):
        m = np.zeros(self.cfg.n_layers, dtype=np.uint8)
        v = ctypes.c_float()
        self._check(self.lib.ssd_dp_select(self.ctx, n_skip, _p(m, ctypes.c_uint8), ctypes.byref(v)))
        return tuple(int(i) for i in np.nonzero(m)[0]), v.value

    def _policy(self, kind: int, **kw):
        cfg = self.cfg
        p = PolicyC()
        p.kind = kind
        p.draft_k = kw.get("k", cfg.draft_k)
        p.act_int8 = int(kw.get("act_int8", False))
        keep = []
        if kind == POLICY_STATIC:
            m = np.zeros(cfg.n_layers, dtype=np.uint8)
            m[list(kw.get("skip", cfg.skip))] = 1
            keep.append(m)
            p.skip_mask = _p(m, ctypes.c_uint8)
        p.dp_n_skip = kw.get("dp_n_skip", cfg.dp_n_skip)
        p.dp_interval = kw.get("dp_interval", cfg.dp_interval)
        p.dp_at_start = int(kw.get("dp_at_start", True))
        levels = kw.get("levels", cfg.levels)
        if kind in (POLICY_DYTC, POLICY_HCASCADE, POLICY_VCASCADE):
            ls = np.zeros((len(levels), cfg.n_layers), dtype=np.uint8)
            li = np.zeros(len(levels), dtype=np.int32)
            for l, (sk, i8) in enumerate(levels):
                ls[l, list(sk)] = 1
                li[l] = int(i8)
            keep += [ls, li]
            p.n_levels = len(levels)
            p.level_skip = _p(ls, ctypes.c_uint8)
            p.level_int8 = _p(li, ctypes.c_int32)
            lx = kw.get("level_exit", cfg.level_exit)
            if lx:
                le = np.array([int(lx[l]) if l < len(lx) else 0 for l in range(len(levels))], dtype=np.int32)
                keep.append(le)
                p.level_exit = _p(le, ctypes.c_int32)
            if kind == POLICY_VCASCADE:
                p.vc_lo, p.vc_hi = int(kw["vc_lo"]), int(kw["vc_hi"])
            if kind == POLICY_HCASCADE:
                hl = _i32(kw["hc_len"])
                keep.append(hl)
                p.hc_len = _p(hl, ctypes.c_int32)
        p.ema_alpha = kw.get("ema_alpha", cfg.ema_alpha)
        p.ema_init = kw.get("ema_init", cfg.ema_init)
        p.tree_max_nodes = kw.get("tree_max_nodes", cfg.tree_max_nodes)
        p.tree_max_depth = kw.get("tree_max_depth", cfg.tree_max_depth)
        p.draft_exit = float(kw.get("exit_thr", 0.0))
        p.early_exit = int(kw.get("early_exit", 0))
        p.cost_model = int(kw.get("cost_model", 0))
        p.cascade_rules = int(kw.get("cascade_rules", False))
        return p, keep

    def generate(self, n_gen: int, kind: int = POLICY_STATIC, **kw) -> List[int]:
        p, keep = self._policy(kind, **kw)
        out = np.zeros(n_gen, dtype=np.int32)
        self._check(self.lib.ssd_generate(self.ctx, ctypes.byref(p), n_gen, _p(out, ctypes.c_int32)))
        return out.tolist()

    def draft_tree(self, **kw):
        p, keep = self._policy(POLICY_DYTC, **kw)
        tok = np.zeros(65, dtype=np.int32)
        par = np.zeros(65, dtype=np.int32)
        n = ctypes.c_int()
        self._check(self.lib.ssd_draft_tree(self.ctx, ctypes.byref(p), _p(tok, ctypes.c_int32),
                                            _p(par, ctypes.c_int32), ctypes.byref(n)))
        return tok[: n.value].tolist(), par[: n.value].tolist()

    def calibrate_latency(self, depths: Sequence[int], seq_lens: Sequence[int], act_int8: bool = False,
                          reps: int = 5, train=None):
        """Time one-draft passes over seq_lens x depths and fit the latency model; returns
        (beta, times_ms[len(seq_lens), len(depths)]).  Rolls the committed length back to
        min(seq_lens)."""
        d, s = _i32(depths), _i32(seq_lens)
        beta = np.zeros(3, dtype=np.float64)
        times = np.zeros((s.size, d.size), dtype=np.float64)
        tr = None if train is None else np.ascontiguousarray(np.asarray(train, dtype=np.uint8).reshape(-1))
        self._check(self.lib.ssd_calibrate_latency(self.ctx, int(act_int8), _p(d, ctypes.c_int32), d.size,
                                                   _p(s, ctypes.c_int32), s.size, reps,
                                                   None if tr is None else _p(tr, ctypes.c_uint8),
                                                   _p(beta, ctypes.c_double), _p(times, ctypes.c_double)))
        return beta, times

    def set_latency_model(self, beta: Sequence[float], act_int8: bool = False):
        b = np.ascontiguousarray(np.asarray(beta, dtype=np.float64))
        self._check(self.lib.ssd_set_latency_model(self.ctx, int(act_int8), _p(b, ctypes.c_double)))

    def level_costs(self, **kw):
        """(DyTC level costs, levels in use) the planner would use now."""
        p, keep = self._policy(POLICY_DYTC, **kw)
        out = np.zeros(max(p.n_levels, 1), dtype=np.float64)
        n = ctypes.c_int()
        self._check(self.lib.ssd_get_level_costs(self.ctx, ctypes.byref(p), _p(out, ctypes.c_double),
                                                 ctypes.byref(n)))
        return out[: p.n_levels].tolist(), n.value

    def dp_table(self):
        """(val [L+1, n+1] float32, back [L+1, n+1] uint8) of the last DP search (NaN / 255 outside its range)."""
        L = self.cfg.n_layers
        n = ctypes.c_int()
        self._check(self.lib.ssd_get_dp_table(self.ctx, ctypes.byref(n), None, None))
        val = np.zeros((L + 1) * (n.value + 1), dtype=np.float32)
        back = np.zeros((L + 1) * (n.value + 1), dtype=np.uint8)
        self._check(self.lib.ssd_get_dp_table(self.ctx, ctypes.byref(n), _p(val, ctypes.c_float),
                                              _p(back, ctypes.c_uint8)))
        return val.reshape(L + 1, n.value + 1), back.reshape(L + 1, n.value + 1)

    def set_ema(self, ema: Sequence[float]):
        a = np.asarray(ema, dtype=np.float64)
        self._check(self.lib.ssd_set_ema(self.ctx, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), a.size))

    def cycle_log(self) -> List[dict]:
        """The per-cycle log (OPT_CYCLE_LOG) as dicts: kind 0 linear cycle, 1 tree cycle, 2 DP run."""
        n_max = 1 << 16
        buf = (CycleRecordC * n_max)()
        n = ctypes.c_int()
        self._check(self.lib.ssd_get_cycle_log(self.ctx, buf, n_max, ctypes.byref(n)))
        out = []
        for r in buf[: n.value]:
            rows = r.n_rows
            e = {"kind": r.kind, "t": r.t}
            if r.kind == 2:
                e.update(mask=tuple(i for i in range(self.cfg.n_layers) if r.mask[i]), dp_value=float(r.dp_value))
            else:
                e.update(tokens=list(r.tokens[:rows]), parents=list(r.parents[:rows]), argmax=list(r.argmax[:rows]),
                         n_acc=r.n_acc, bonus=r.bonus, path=list(r.path[: r.n_acc + 1]), ema=list(r.ema))
            out.append(e)
        return out

    def logits(self, row: int = 0) -> np.ndarray:
        out = np.zeros(self.cfg.vocab, dtype=np.float32)
        self._check(self.lib.ssd_get_logits(self.ctx, row, _p(out, ctypes.c_float)))
        return out

    def hidden(self, layer: int, row: int = 0) -> np.ndarray:
        out = np.zeros(self.cfg.d_model, dtype=np.float32)
        self._check(self.lib.ssd_get_hidden(self.ctx, layer, row, _p(out, ctypes.c_float)))
        return out

    def position(self):
        t, p = ctypes.c_int32(), ctypes.c_int32()
        self._check(self.lib.ssd_get_position(self.ctx, ctypes.byref(t), ctypes.byref(p)))
        return t.value, p.value

    def stats(self) -> dict:
        s = StatsC()
        self._check(self.lib.ssd_get_stats(self.ctx, ctypes.byref(s)))
        return {"cycles": s.cycles, "drafted": s.drafted, "accepted": s.accepted, "dp_runs": s.dp_runs, "ar_steps": s.ar_steps,
                "accept_hist": list(s.accept_hist), "ema": list(s.ema), "launches": s.kernel_launches, "mma_fallbacks": s.mma_fallbacks}

    def reset_stats(self):
        self._check(self.lib.ssd_reset_stats(self.ctx))

    def trace(self, max_entries: int = 8192):
        """Per-kernel device timeline of the last traced pass: list of
        (kind, resident_ns, running_ns, end_ns), times relative to the first kernel."""
        buf = np.zeros(4 * max_entries, dtype=np.int64)
        n = ctypes.c_int()
        self._check(self.lib.ssd_get_trace(self.ctx, _p(buf, ctypes.c_int64), max_entries, ctypes.byref(n)))
        rows = buf[: 4 * n.value].reshape(-1, 4)
        if len(rows):
            t0 = rows[:, 1].min()
            rows[:, 1:] -= t0
        return [tuple(int(x) for x in r) for r in rows]

    def pass_times(self):
        ms = (ctypes.c_double * 4)()
        n = (ctypes.c_int64 * 4)()
        self._check(self.lib.ssd_get_pass_times(self.ctx, ms, n))
        return {k: (ms[i], n[i]) for i, k in enumerate(("draft", "verify", "dp", "ar"))}
