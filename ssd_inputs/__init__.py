"""Seeded synthetic inputs shared by the CPU oracle and the GPU path.

This module holds no arithmetic of the decoding method.  It defines

* the model shapes and workload parameters of the five synthetic workloads
  (`CONFIGS`), including the layer-skip sets the drafts use;
* the weight recipe: which logical tensors a Llama-style decoder has, their
  shapes, their generator ids and the normal distribution each is drawn from;
* two implementations of one counter-based generator (gen_def.h):
  `libssd_inputs_host.so` (C, OpenMP; used by the oracle and tests) and
  `libssd_inputs_dev.so` (CUDA; fills device memory for the GPU path).

Random-weight recipe (the workloads' stated init rule): every matrix is
N(0, 0.02); the two output projections of each layer (attention output W_o
and FFN down W_d) are additionally scaled by 1/sqrt(2 L), so the residual
stream changes slowly across layers; RMSNorm gains are 1 (tests may draw
them from N(1, 0.1) to exercise the gain path).  Prompts are uniform random
token ids.  No trained weights or public benchmark data are used.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
from fractions import Fraction
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "lib")

# ----------------------------------------------------------------------------
# model shapes and workloads
# ----------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    dtype: str = "bf16"  # storage type of weights and KV cache: "bf16" | "fp16"
    rms_eps: float = 1e-5
    rope_base: float = 10000.0
    # workload
    prompt_len: int = 32
    n_gen: int = 64
    draft_k: int = 4
    skip: Tuple[int, ...] = ()  # static draft skip set (0-based layer indices)
    dp_n_skip: int = 0  # CLaSp: number of layers the DP selects to skip (0 = static skip)
    dp_interval: int = 0  # CLaSp: re-run the DP every this many verify steps
    tree: bool = False  # CAS-Spec cascade + DyTC tree drafts
    tree_max_nodes: int = 16
    tree_max_depth: int = 6
    levels: Tuple[Tuple[Tuple[int, ...], bool], ...] = ()  # (skip set, act_int8) per cascade level L1..L3
    level_exit: Tuple[int, ...] = ()  # per cascade level: final layers not run (early exit); () = none
    ema_alpha: float = 0.2
    ema_init: float = 0.65
    seed: int = 0
    gamma_sigma: float = 0.0  # 0 => unit RMSNorm gains (the workloads); tests may set 0.1

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def max_ctx(self) -> int:
        return self.prompt_len + self.n_gen + 2 * (self.tree_max_nodes + 2) + 64

    def replace(self, **kw) -> "ModelConfig":
        return dataclasses.replace(self, **kw)


def even_subset(pool: Sequence[int], s: int) -> Tuple[int, ...]:
    """s evenly spaced members of `pool`: pool[floor((m + 1/2) * len(pool) / s)]."""
    pool = list(pool)
    if s == 0:
        return ()
    return tuple(sorted(pool[math.floor(Fraction(2 * m + 1, 2 * s) * len(pool))] for m in range(s)))


def cascade_levels(L: int, early_exit: int = 0) -> Tuple[Tuple[Tuple[int, ...], bool], ...]:
    """The three cascade levels: L2 skips 30 % of the L layers (evenly spaced) with int8
    activations, L3 runs every layer with int8 activations, L1 skips 70 % of the layers it
    can run, nested around L2.  With early_exit = e, L1 also stops e layers before the end:
    its 70 % are taken from the first L - e layers and the last e layers are its early exit
    (returned separately by the caller as the level's exit count, not in the skip set)."""
    n = L - early_exit
    l2 = even_subset(range(L), round(0.3 * L))
    base = [i for i in l2 if i < n]
    rest = [i for i in range(n) if i not in base]
    l1 = tuple(sorted(set(base) | set(even_subset(rest, round(0.7 * n) - len(base)))))
    return ((l1, False), (l2, True), ((), True))


def _cascade_13b() -> Tuple[Tuple[Tuple[int, ...], bool], ...]:
    return cascade_levels(40)


CONFIGS: Dict[str, ModelConfig] = {
    "tiny": ModelConfig("tiny", 4, 256, 4, 4, 64, 688, 1024, prompt_len=32, n_gen=64, draft_k=4, skip=(1, 2)),
    "llama3_8b": ModelConfig("llama3_8b", 32, 4096, 32, 8, 128, 14336, 128256, prompt_len=512, n_gen=256,
                             draft_k=6, skip=even_subset(range(32), 16)),
    "llama2_13b_cascade": ModelConfig("llama2_13b_cascade", 40, 5120, 40, 40, 128, 13824, 32000, dtype="fp16",
                                      prompt_len=256, n_gen=256, tree=True, levels=_cascade_13b()),
    "llama3_8b_clasp": ModelConfig("llama3_8b_clasp", 32, 4096, 32, 8, 128, 14336, 128256, prompt_len=1024,
                                   n_gen=512, draft_k=6, dp_n_skip=16, dp_interval=32),
    "llama3_70b_clasp": ModelConfig("llama3_70b_clasp", 80, 8192, 64, 8, 128, 28672, 128256, prompt_len=2048,
                                    n_gen=256, draft_k=8, dp_n_skip=44, dp_interval=64),
}

# ----------------------------------------------------------------------------
# weight recipe
# ----------------------------------------------------------------------------

EMBED, FINAL_NORM, LM_HEAD = 0, 1, 2
WQ, WK, WV, WO, WG, WU, WD, G_ATTN, G_FFN = range(9)
LAYER_TENSORS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "g_attn", "g_ffn")


def tensor_id(kind: int, layer: Optional[int] = None) -> int:
    """Generator id of a logical tensor: globals 0..2, layer i kind k -> 16 + 16 i + k."""
    return kind if layer is None else 16 + 16 * layer + kind


@dataclasses.dataclass(frozen=True)
class TensorSpec:
    name: str
    tid: int
    shape: Tuple[int, ...]
    mean: float
    sigma: float  # 0 => constant `mean`


def layer_specs(cfg: ModelConfig, i: int) -> List[TensorSpec]:
    d, hd, F = cfg.d_model, cfg.head_dim, cfg.ffn
    s_out = 0.02 / math.sqrt(2 * cfg.n_layers)
    g_mean, g_sig = 1.0, cfg.gamma_sigma
    shapes = {
        "wq": (cfg.n_q_heads * hd, d), "wk": (cfg.n_kv_heads * hd, d), "wv": (cfg.n_kv_heads * hd, d),
        "wo": (d, cfg.n_q_heads * hd), "wg": (F, d), "wu": (F, d), "wd": (d, F), "g_attn": (d,), "g_ffn": (d,),
    }
    out = []
    for k, name in enumerate(LAYER_TENSORS):
        if name.startswith("g_"):
            mean, sig = g_mean, g_sig
        else:
            mean, sig = 0.0, (s_out if name in ("wo", "wd") else 0.02)
        out.append(TensorSpec(name, tensor_id(k, i), shapes[name], mean, sig))
    return out


def global_specs(cfg: ModelConfig) -> List[TensorSpec]:
    return [
        TensorSpec("embed", tensor_id(EMBED), (cfg.vocab, cfg.d_model), 0.0, 0.02),
        TensorSpec("final_norm", tensor_id(FINAL_NORM), (cfg.d_model,), 1.0, cfg.gamma_sigma),
        TensorSpec("lm_head", tensor_id(LM_HEAD), (cfg.vocab, cfg.d_model), 0.0, 0.02),
    ]


# ----------------------------------------------------------------------------
# host generator (C)
# ----------------------------------------------------------------------------

_host = None


def _build(cmd: List[str]) -> None:
    os.makedirs(_LIBDIR, exist_ok=True)
    subprocess.run(cmd, check=True, cwd=_HERE)


def build_host(force: bool = False) -> str:
    out = os.path.join(_LIBDIR, "libssd_inputs_host.so")
    if force or not os.path.exists(out):
        _build(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC", "-o", out, "gen_host.c", "-lm"])
    return out


def build_dev(force: bool = False, nvcc: str = "nvcc") -> str:
    out = os.path.join(_LIBDIR, "libssd_inputs_dev.so")
    if force or not os.path.exists(out):
        _build([nvcc, "-O3", "-fmad=false", "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-Xcompiler", "-fPIC",
                "-cudart", "shared", "-o", out, "gen_dev.cu"])
    return out


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host())
        lib.ssd_inputs_fill_host.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                             ctypes.c_uint64, ctypes.c_double, ctypes.c_double, ctypes.c_int]
        lib.ssd_inputs_fill_host.restype = None
        lib.ssd_inputs_fill_const_host.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_float, ctypes.c_int]
        lib.ssd_inputs_prompt_host.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_int]
        lib.ssd_inputs_mix_host.argtypes = [ctypes.c_uint64]
        lib.ssd_inputs_mix_host.restype = ctypes.c_uint64
        _host = lib
    return _host


def host_values(spec: TensorSpec, cfg: ModelConfig, offset: int = 0, count: Optional[int] = None) -> np.ndarray:
    """16-bit storage bits (np.uint16) of a logical tensor, or a slice of its flat elements."""
    n = int(np.prod(spec.shape)) if count is None else count
    out = np.empty(n, dtype=np.uint16)
    fp16 = 1 if cfg.dtype == "fp16" else 0
    lib = _host_lib()
    if spec.sigma == 0.0:
        lib.ssd_inputs_fill_const_host(out.ctypes.data, n, spec.mean, fp16)
    else:
        lib.ssd_inputs_fill_host(out.ctypes.data, n, offset, cfg.seed, spec.tid, spec.mean, spec.sigma, fp16)
    if count is None:
        out = out.reshape(spec.shape)
    return out


def mix(x: int) -> int:
    """The generator's counter hash (SplitMix64 output function), from the C library."""
    return int(_host_lib().ssd_inputs_mix_host(x & ((1 << 64) - 1)))


def const_bits(c: float, dtype: str) -> int:
    """16-bit storage bits of the constant c, from the C library's rounding."""
    out = np.empty(1, dtype=np.uint16)
    _host_lib().ssd_inputs_fill_const_host(out.ctypes.data, 1, c, 1 if dtype == "fp16" else 0)
    return int(out[0])


def widen(bits: np.ndarray, dtype: str, out=np.float64) -> np.ndarray:
    """16-bit storage bits -> their exact values as float64 (or float32: every bf16/fp16 value is one)."""
    if dtype == "fp16":
        return bits.view(np.float16).astype(out)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    return f if out == np.float32 else f.astype(out)


def prompt(cfg: ModelConfig, n: Optional[int] = None, seed: Optional[int] = None) -> np.ndarray:
    n = cfg.prompt_len if n is None else n
    out = np.empty(n, dtype=np.int32)
    _host_lib().ssd_inputs_prompt_host(out.ctypes.data, n, cfg.seed if seed is None else seed, cfg.vocab)
    return out


# ----------------------------------------------------------------------------
# device generator (CUDA), for the GPU path
# ----------------------------------------------------------------------------

_dev = None


def _dev_lib():
    global _dev
    if _dev is None:
        path = os.path.join(_LIBDIR, "libssd_inputs_dev.so")
        if not os.path.exists(path):
            raise RuntimeError("libssd_inputs_dev.so is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        lib.ssd_inputs_fill_dev.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                            ctypes.c_uint64, ctypes.c_double, ctypes.c_double, ctypes.c_int,
                                            ctypes.c_void_p]
        lib.ssd_inputs_fill_dev.restype = ctypes.c_int
        lib.ssd_inputs_fill_const_dev.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_float, ctypes.c_int,
                                                  ctypes.c_void_p]
        lib.ssd_inputs_fill_const_dev.restype = ctypes.c_int
        _dev = lib
    return _dev


def fill_device(ptr: int, spec: TensorSpec, cfg: ModelConfig, offset: int = 0, count: Optional[int] = None,
                stream: int = 0) -> None:
    """Write the 16-bit values of a logical tensor (or a flat slice of it) to device address `ptr`."""
    n = int(np.prod(spec.shape)) if count is None else count
    fp16 = 1 if cfg.dtype == "fp16" else 0
    lib = _dev_lib()
    if spec.sigma == 0.0:
        rc = lib.ssd_inputs_fill_const_dev(ptr, n, spec.mean, fp16, stream)
    else:
        rc = lib.ssd_inputs_fill_dev(ptr, n, offset, cfg.seed, spec.tid, spec.mean, spec.sigma, fp16, stream)
    if rc != 0:
        raise RuntimeError(f"device input fill failed (code {rc})")
