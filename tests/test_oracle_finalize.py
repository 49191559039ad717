"""Pins for the oracle's combine (moe_finalize page).

Checked against closed forms (a permutation copy, constant rows), a library
gather-and-weighted-sum in fp64, the oracle's own fp64 variant within the
fp32 rounding bound, and a hand-derived fixture.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import GOLDEN


def bf16_bits(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _random_case(T, K, H, seed):
    rng = np.random.default_rng(seed)
    N = T * K
    down = synth.normal_bf16(seed, 3, N * H).reshape(N, H)
    restore = rng.permutation(N).astype(np.uint32)
    w = rng.random((T, K), dtype=np.float32) * 2 - 0.5
    return down, restore, w


def fp32_sum_bound(down, restore, w, T, K, H):
    """|fp32 result - exact| <= K * 2^-24 * sum_k |w_k x_k| (sequential FMA chain)."""
    x = bits_to_f32(down)[restore.astype(np.int64)].reshape(T, K, H).astype(np.float64)
    mag = (np.abs(w.astype(np.float64))[:, :, None] * np.abs(x)).sum(axis=1)
    return K * 2.0 ** -24 * mag + 1e-30


def test_golden_fixture():
    with open(os.path.join(GOLDEN, "finalize_small.json")) as fh:
        fx = json.load(fh)
    T, K, H = fx["T"], fx["K"], fx["H"]
    out = oracle.finalize(bf16_bits(fx["down"]), np.array(fx["restore_order"]),
                          np.array(fx["router_weight"], dtype=np.float32), T, K, H)
    assert out.tolist() == fx["expected"]


def test_permutation_copy_closed_form():
    """K = 1 and weight 1: output row t is exactly down[restore[t]]."""
    T, H = 37, 24
    down, restore, _ = _random_case(T, 1, H, 1)
    w = np.ones((T, 1), dtype=np.float32)
    out = oracle.finalize(down, restore, w, T, 1, H)
    assert np.array_equal(out, bits_to_f32(down)[restore.astype(np.int64)])


def test_constant_rows_closed_form():
    """All rows equal to c = 0.5 (exact in bf16): output = c * sum_k w_k."""
    T, K, H = 20, 6, 16
    N = T * K
    down = bf16_bits(np.full((N, H), 0.5))
    rng = np.random.default_rng(2)
    restore = rng.permutation(N).astype(np.uint32)
    w = rng.random((T, K), dtype=np.float32)
    out = oracle.finalize(down, restore, w, T, K, H)
    ref = 0.5 * w.astype(np.float64).sum(axis=1)
    np.testing.assert_allclose(out, np.broadcast_to(ref[:, None], (T, H)), rtol=K * 2 ** -24)


@pytest.mark.parametrize("T,K,H", [(1, 1, 8), (5, 2, 40), (33, 8, 256), (64, 4, 256),
                                   (17, 3, 72)])
def test_library_gather_weighted_sum(T, K, H):
    """torch CPU index_select + weighted sum in fp64 vs the oracle's fp32 sum."""
    down, restore, w = _random_case(T, K, H, T * 100 + K * 10 + H)
    out = oracle.finalize(down, restore, w, T, K, H)
    d = torch.from_numpy(bits_to_f32(down).reshape(T * K, H)).double()
    rows = torch.index_select(d, 0, torch.from_numpy(restore.astype(np.int64)))
    ref = (torch.from_numpy(w).double()[:, :, None] * rows.view(T, K, H)).sum(dim=1).numpy()
    bound = fp32_sum_bound(down, restore, w, T, K, H)
    assert (np.abs(out - ref) <= bound).all()
    # a wrong row, a dropped term or a swapped weight would move far past the bound
    assert np.abs(out - ref).max() < 1e-3


def test_fp64_variant_bounds_fp32():
    T, K, H = 48, 8, 128
    down, restore, w = _random_case(T, K, H, 5)
    out32 = oracle.finalize(down, restore, w, T, K, H)
    out64 = oracle.finalize_f64(down, restore, w, T, K, H)
    assert (np.abs(out32 - out64) <= fp32_sum_bound(down, restore, w, T, K, H)).all()


def test_selected_tokens_match_full():
    T, K, H = 40, 3, 64
    down, restore, w = _random_case(T, K, H, 9)
    full = oracle.finalize(down, restore, w, T, K, H)
    toks = np.array([0, 39, 7, 7, 21])
    part = oracle.finalize(down, restore, w, T, K, H, tokens=toks)
    assert np.array_equal(part, full[toks])


def test_tiny_workload_chain():
    """Route -> index -> finalize on the 64-token workload, checked in fp64
    against a direct per-(token, k) lookup of each chosen expert's row."""
    cfg = synth.get_config("tiny")
    scores = synth.make_scores(cfg)
    ids, w = oracle.route(scores, synth.make_bias(cfg), cfg.K, cfg.G, cfg.M, cfg.norm_weights,
                          cfg.scale)
    idx = oracle.create_indices(ids, cfg.E)
    down = synth.make_down(cfg)
    out = oracle.finalize(down, idx["restore_token_order"], w, cfg.T, cfg.K, cfg.H)
    x = bits_to_f32(down).astype(np.float64)
    teo = idx["token_expert_order"]
    ref = np.zeros((cfg.T, cfg.H))
    for p in range(cfg.N):  # row p of down belongs to slot teo[p] = t*K + k
        t, k = divmod(int(teo[p]), cfg.K)
        ref[t] += float(w[t, k]) * x[p]
    bound = fp32_sum_bound(down, idx["restore_token_order"], w, cfg.T, cfg.K, cfg.H)
    assert (np.abs(out - ref) <= bound).all()


def test_out_of_range_row_rejected():
    down = bf16_bits(np.zeros((4, 8)))
    with pytest.raises(oracle.OracleError):
        oracle.finalize(down, np.array([0, 1, 2, 4]), np.ones((2, 2), np.float32), 2, 2, 8)
