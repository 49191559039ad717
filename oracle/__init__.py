"""Python access to the CPU oracle (``moe_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the product package. The oracle shares
no code with the CUDA path; ``build()`` compiles it with the host compiler
(no fast-math, no floating-point contraction, so it computes the same bits on
x86-64 and aarch64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "moe_oracle.cpp"), os.path.join(_HERE, "moe_oracle.h")]
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

OK, ERR_ARG, ERR_NAN, ERR_DATA = 0, -1, -2, -3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(s) for s in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRCS[0]]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _open(path: str):
    lib = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    lib.oracle_route.argtypes = [vp, vp, i64, i32, i32, i32, i32, i32, f32, vp, vp]
    lib.oracle_create_indices.argtypes = [vp, i64, i32, vp, vp, vp, vp, vp]
    lib.oracle_finalize.argtypes = [vp, vp, vp, i64, i32, i64, vp]
    lib.oracle_finalize_tokens.argtypes = [vp, vp, vp, i64, i32, i64, vp, i64, vp]
    lib.oracle_finalize_f64.argtypes = [vp, vp, vp, i64, i32, i64, vp]
    lib.oracle_permute.argtypes = [vp, vp, i64, i32, i64, vp]
    lib.oracle_scales_offsets.argtypes = [vp, i64, i32, ctypes.c_uint32, vp]
    lib.oracle_exp.argtypes = [vp, i64, vp]
    lib.oracle_sigmoid.argtypes = [vp, i64, vp]
    lib.oracle_softmax.argtypes = [vp, i64, i32, vp]
    for f in (lib.oracle_route, lib.oracle_create_indices, lib.oracle_finalize,
              lib.oracle_finalize_tokens, lib.oracle_finalize_f64, lib.oracle_permute,
              lib.oracle_scales_offsets, lib.oracle_exp, lib.oracle_sigmoid,
              lib.oracle_softmax):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _open(build())
    return _lib


class using_library:
    """Temporarily route every oracle call through another build of the oracle
    (the tests that plant a mistake in a copy of the oracle source use it)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self._saved = _lib
        _lib = _open(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def _check(rc, what):
    if rc != OK:
        raise OracleError(f"{what} returned {rc}")


def route(scores, bias, K: int, n_groups: int, topk_group: int, norm_weights: bool,
          scale: float):
    """Returns (expert_indices int32 [T,K], expert_weights float32 [T,K])."""
    s, sp = _c(scores, np.float32)
    b, bp = _c(bias, np.float32)
    T, E = s.shape
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float32)
    rc = _load().oracle_route(sp, bp, T, E, K, n_groups, topk_group, int(bool(norm_weights)),
                              float(scale), ids.ctypes.data, w.ctypes.data)
    _check(rc, "oracle_route")
    return ids, w


def create_indices(topk_ids, E: int):
    """Returns dict of token_expert_order, expert_start_indices, restore_token_order,
    expert_ids, expert_usage_stats."""
    ids, ip = _c(np.asarray(topk_ids).reshape(-1), np.int32)
    N = ids.size
    teo = np.empty(N, dtype=np.uint32)
    start = np.empty(E + 1, dtype=np.uint32)
    restore = np.empty(N, dtype=np.uint32)
    eids = np.empty(E, dtype=np.int32)
    stats = np.empty(2, dtype=np.uint32)
    rc = _load().oracle_create_indices(ip, N, E, teo.ctypes.data, start.ctypes.data,
                                       restore.ctypes.data, eids.ctypes.data, stats.ctypes.data)
    _check(rc, "oracle_create_indices")
    return {"token_expert_order": teo, "expert_start_indices": start,
            "restore_token_order": restore, "expert_ids": eids, "expert_usage_stats": stats}


def finalize(down_bf16_bits, restore, w, T: int, K: int, H: int, tokens=None):
    """fp32 result [T,H] (or [len(tokens),H]) before bf16 rounding.

    ``down_bf16_bits`` holds raw bf16 bit patterns (uint16) [T*K, H]."""
    d, dp = _c(down_bf16_bits, np.uint16)
    r, rp = _c(restore, np.uint32)
    ww, wp = _c(w, np.float32)
    assert d.size == T * K * H and r.size == T * K and ww.size == T * K
    if tokens is None:
        out = np.empty((T, H), dtype=np.float32)
        rc = _load().oracle_finalize(dp, rp, wp, T, K, H, out.ctypes.data)
    else:
        tk, tp = _c(tokens, np.int64)
        out = np.empty((tk.size, H), dtype=np.float32)
        rc = _load().oracle_finalize_tokens(dp, rp, wp, T, K, H, tp, tk.size, out.ctypes.data)
    _check(rc, "oracle_finalize")
    return out


def finalize_f64(down_bf16_bits, restore, w, T: int, K: int, H: int):
    d, dp = _c(down_bf16_bits, np.uint16)
    r, rp = _c(restore, np.uint32)
    ww, wp = _c(w, np.float32)
    out = np.empty((T, H), dtype=np.float64)
    rc = _load().oracle_finalize_f64(dp, rp, wp, T, K, H, out.ctypes.data)
    _check(rc, "oracle_finalize_f64")
    return out


def permute(input_bf16_bits, token_expert_order, K: int):
    """Expert-contiguous token rows [T*K, H] (bf16 bit patterns)."""
    x, xp = _c(input_bf16_bits, np.uint16)
    teo, tp = _c(token_expert_order, np.uint32)
    T, H = x.shape
    out = np.empty((T * K, H), dtype=np.uint16)
    rc = _load().oracle_permute(xp, tp, T, K, H, out.ctypes.data)
    _check(rc, "oracle_permute")
    return out


def scales_offsets(topk_ids, E: int, row_align: int = 128):
    """Aligned per-expert scale offsets [E+1] (see moe_oracle.h)."""
    ids, ip = _c(np.asarray(topk_ids).reshape(-1), np.int32)
    out = np.empty(E + 1, dtype=np.uint32)
    rc = _load().oracle_scales_offsets(ip, ids.size, E, row_align, out.ctypes.data)
    _check(rc, "oracle_scales_offsets")
    return out


def exp_f32(x):
    """fp32 exp of the score loaders (argument clamped to [-87, 88])."""
    a, ap = _c(x, np.float32)
    out = np.empty_like(a)
    _check(_load().oracle_exp(ap, a.size, out.ctypes.data), "oracle_exp")
    return out


def sigmoid(x):
    """fp32 sigmoid score loader (same shape as x)."""
    a, ap = _c(x, np.float32)
    out = np.empty_like(a)
    _check(_load().oracle_sigmoid(ap, a.size, out.ctypes.data), "oracle_sigmoid")
    return out


def softmax(x):
    """fp32 softmax score loader over the last axis of a [rows, E] array."""
    a, ap = _c(x, np.float32)
    a2 = a.reshape(-1, a.shape[-1])
    out = np.empty_like(a2)
    _check(_load().oracle_softmax(ap, a2.shape[0], a2.shape[1], out.ctypes.data),
           "oracle_softmax")
    return out.reshape(a.shape)
