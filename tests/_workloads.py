"""Shared helpers of the test suite: seeded workload inputs, the oracle's
expected results for them (cached per process), and host/device conversions."""
from __future__ import annotations

import functools

import numpy as np

import oracle
import synth


def bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (numpy, no NaN inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def finalize_tolerance_ok(got_bf16_bits, ref_f32):
    """|gpu - ref| <= 1e-2 + 8e-3 |ref| against the fp32 oracle before rounding."""
    got = bits_to_f32(got_bf16_bits)
    return np.abs(got - ref_f32) <= 1e-2 + 8e-3 * np.abs(ref_f32)


@functools.lru_cache(maxsize=2)
def workload(name: str):
    cfg = synth.get_config(name)
    scores = synth.make_scores(cfg)
    bias = synth.make_bias(cfg)
    ids, w = oracle.route(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    idx = oracle.create_indices(ids, cfg.E)
    return cfg, scores, bias, ids, w, idx


@functools.lru_cache(maxsize=1)
def workload_down(name: str):
    cfg = synth.get_config(name)
    return synth.make_down(cfg)


@functools.lru_cache(maxsize=1)
def workload_finalize_ref(name: str):
    cfg, _, _, _, w, idx = workload(name)
    down = workload_down(name)
    return oracle.finalize(down, idx["restore_token_order"], w, cfg.T, cfg.K, cfg.H)
