"""Seeded synthetic inputs for the MoE routing workloads.

This package only produces input tensors (scores, bias, expert outputs) with
the shapes and value distributions of the five routing workloads. It holds
none of the routing, index-building or combine arithmetic, and it is the only
code shared by the oracle's tests, the GPU parity tests and the benchmark.

The generator itself is the C file ``synth.c`` next to this module (counter
based SplitMix64 + Box-Muller, multi-threaded); ``build()`` compiles it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")

# Independent generator streams, one per input tensor, keyed (seed, tensor id).
TENSOR_SCORES = 1
TENSOR_BIAS = 2
TENSOR_DOWN = 3
TENSOR_INPUT = 4


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` (host code, no GPU needed)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u64, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                  ctypes.c_void_p)
        lib.synth_normal_f32.argtypes = [u64, u64, dbl, dbl, vp, i64, i64, i32]
        lib.synth_sigmoid_normal_f32.argtypes = [u64, u64, vp, i64, i64, i32]
        lib.synth_softmax_normal_f32.argtypes = [u64, u64, vp, i64, i64, i64, i32]
        lib.synth_normal_bf16.argtypes = [u64, u64, vp, i64, i64, i32]
        for f in (lib.synth_normal_f32, lib.synth_sigmoid_normal_f32,
                  lib.synth_softmax_normal_f32, lib.synth_normal_bf16):
            f.restype = None
        _lib = lib
    return _lib


def normal_f32(seed: int, tensor: int, n: int, mean: float = 0.0, std: float = 1.0,
               first: int = 0, threads: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    if n:
        _load().synth_normal_f32(seed, tensor, mean, std, out.ctypes.data, first, n, threads)
    return out


def sigmoid_normal_f32(seed: int, tensor: int, n: int, first: int = 0,
                       threads: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    if n:
        _load().synth_sigmoid_normal_f32(seed, tensor, out.ctypes.data, first, n, threads)
    return out


def softmax_normal_f32(seed: int, tensor: int, rows: int, cols: int, first_row: int = 0,
                       threads: int = 0) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.float32)
    if rows and cols:
        _load().synth_softmax_normal_f32(seed, tensor, out.ctypes.data, first_row, rows, cols,
                                         threads)
    return out


def normal_bf16_into(ptr: int, seed: int, tensor: int, n: int, first: int = 0,
                     threads: int = 0) -> None:
    """Write n bf16 N(0,1) values (raw uint16 bit patterns) to host address ``ptr``."""
    if n:
        _load().synth_normal_bf16(seed, tensor, ctypes.c_void_p(ptr), first, n, threads)


def normal_bf16(seed: int, tensor: int, n: int, first: int = 0, threads: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    normal_bf16_into(out.ctypes.data, seed, tensor, n, first, threads)
    return out


@dataclass(frozen=True)
class MoeConfig:
    """One routing workload: sizes, score/bias recipe and router options.

    T tokens, E routed experts in G groups (topk_group M kept), K experts per
    token, hidden size H of the expert outputs combined by finalize.
    """
    name: str
    T: int
    E: int
    G: int
    M: int
    K: int
    H: int
    scores: str            # "sigmoid": sigmoid(N(0,1)); "softmax": row softmax of N(0,1) logits
    bias: str              # "normal": N(0, bias_std); "hot": hot_bias for e < hot_experts; "zero"
    norm_weights: bool
    scale: float
    bias_std: float = 0.0
    hot_experts: int = 0
    hot_bias: float = 0.0
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def N(self) -> int:
        return self.T * self.K

    def replace(self, **kw) -> "MoeConfig":
        d = dict(self.__dict__)
        d.update(kw)
        return MoeConfig(**d)


CONFIGS = [
    MoeConfig("tiny", T=64, E=16, G=4, M=2, K=4, H=256, scores="sigmoid", bias="normal",
              bias_std=0.1, norm_weights=True, scale=1.0),
    MoeConfig("dsv3_decode", T=128, E=256, G=8, M=4, K=8, H=7168, scores="sigmoid",
              bias="normal", bias_std=0.05, norm_weights=True, scale=2.5),
    MoeConfig("dsv3_prefill", T=16384, E=256, G=8, M=4, K=8, H=7168, scores="sigmoid",
              bias="normal", bias_std=0.05, norm_weights=True, scale=2.5),
    MoeConfig("skewed_ungrouped", T=8192, E=128, G=1, M=1, K=8, H=4096, scores="softmax",
              bias="hot", hot_experts=8, hot_bias=2.0, norm_weights=True, scale=1.0),
    MoeConfig("few_expert_large_batch", T=131072, E=8, G=1, M=1, K=2, H=4096, scores="softmax",
              bias="zero", norm_weights=False, scale=1.0),
]
CONFIG_BY_NAME = {c.name: c for c in CONFIGS}


def get_config(name_or_index) -> MoeConfig:
    if isinstance(name_or_index, int):
        return CONFIGS[name_or_index]
    return CONFIG_BY_NAME[name_or_index]


def make_scores(cfg: MoeConfig, first_token: int = 0, n_tokens: int | None = None,
                threads: int = 0) -> np.ndarray:
    """fp32 routing scores [n_tokens, E] (tokens first_token .. first_token+n_tokens-1)."""
    n = cfg.T - first_token if n_tokens is None else n_tokens
    if cfg.scores == "sigmoid":
        flat = sigmoid_normal_f32(cfg.seed, TENSOR_SCORES, n * cfg.E, first=first_token * cfg.E,
                                  threads=threads)
        return flat.reshape(n, cfg.E)
    if cfg.scores == "softmax":
        return softmax_normal_f32(cfg.seed, TENSOR_SCORES, n, cfg.E, first_row=first_token,
                                  threads=threads)
    raise ValueError(cfg.scores)


def make_bias(cfg: MoeConfig) -> np.ndarray:
    """fp32 per-expert bias [E]."""
    if cfg.bias == "normal":
        return normal_f32(cfg.seed, TENSOR_BIAS, cfg.E, std=cfg.bias_std)
    if cfg.bias == "hot":
        b = np.zeros(cfg.E, dtype=np.float32)
        b[:cfg.hot_experts] = np.float32(cfg.hot_bias)
        return b
    if cfg.bias == "zero":
        return np.zeros(cfg.E, dtype=np.float32)
    raise ValueError(cfg.bias)


def make_down(cfg: MoeConfig, first_row: int = 0, n_rows: int | None = None,
              out_ptr: int | None = None, threads: int = 0):
    """bf16 N(0,1) expert outputs [n_rows, H] as uint16 bit patterns.

    Row r of the full tensor is elements r*H .. r*H+H-1 of the stream, so any
    row range can be regenerated on its own. With ``out_ptr`` the values are
    written to that host address (e.g. a pinned buffer) and None is returned.
    """
    n = cfg.N - first_row if n_rows is None else n_rows
    if out_ptr is not None:
        normal_bf16_into(out_ptr, cfg.seed, TENSOR_DOWN, n * cfg.H, first=first_row * cfg.H,
                         threads=threads)
        return None
    return normal_bf16(cfg.seed, TENSOR_DOWN, n * cfg.H, first=first_row * cfg.H,
                       threads=threads).reshape(n, cfg.H)


def make_input(cfg: MoeConfig, first_row: int = 0, n_rows: int | None = None,
               out_ptr: int | None = None, threads: int = 0):
    """bf16 N(0,1) token rows [n_rows, H] (the permute's input) as uint16 bit patterns."""
    n = cfg.T - first_row if n_rows is None else n_rows
    if out_ptr is not None:
        normal_bf16_into(out_ptr, cfg.seed, TENSOR_INPUT, n * cfg.H, first=first_row * cfg.H,
                         threads=threads)
        return None
    return normal_bf16(cfg.seed, TENSOR_INPUT, n * cfg.H, first=first_row * cfg.H,
                       threads=threads).reshape(n, cfg.H)
