"""Pins for the oracle's expert-contiguous token rows (the grouped matmul's
input, moe_create_indices page): a hand-derived fixture, a library gather,
the multiset property and a closed-form round trip through finalize."""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from conftest import GOLDEN
from test_oracle_finalize import bf16_bits, bits_to_f32


def test_golden_fixture():
    with open(os.path.join(GOLDEN, "permute_small.json")) as fh:
        fx = json.load(fh)
    out = oracle.permute(bf16_bits(fx["input"]), np.array(fx["token_expert_order"]), fx["K"])
    assert bits_to_f32(out).tolist() == fx["expected"]


@pytest.mark.parametrize("T,K,H", [(1, 1, 8), (7, 3, 16), (64, 4, 24), (200, 8, 40)])
def test_library_gather(T, K, H):
    rng = np.random.default_rng(T + K + H)
    x = synth.normal_bf16(1, 4, T * H).reshape(T, H)
    teo = rng.permutation(T * K).astype(np.uint32)
    out = oracle.permute(x, teo, K)
    assert np.array_equal(out, np.take(x, teo.astype(np.int64) // K, axis=0))
    # every token row appears exactly K times
    rows, counts = np.unique(out.view(np.dtype((np.void, 2 * H))), return_counts=True)
    assert (counts % K == 0).all()


@pytest.mark.parametrize("K", [1, 2, 4, 8])
def test_round_trip_through_finalize(K):
    """finalize(permute(x)) with every weight 1/K (a power of two) gives back x
    exactly: the K gathered copies of each row sum to K * (x/K)."""
    T, H = 33, 16
    cfg = synth.get_config("tiny")
    scores = synth.make_scores(cfg.replace(T=T))
    E = cfg.E
    ids = np.argsort(-scores, axis=1, kind="stable")[:, :K].astype(np.int32)
    idx = oracle.create_indices(ids, E)
    x = synth.normal_bf16(2, 4, T * H).reshape(T, H)
    down = oracle.permute(x, idx["token_expert_order"], K)
    w = np.full((T, K), 1.0 / K, dtype=np.float32)
    out = oracle.finalize(down, idx["restore_token_order"], w, T, K, H)
    assert np.array_equal(out, bits_to_f32(x))


def test_out_of_range_slot_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.permute(np.zeros((2, 8), np.uint16), np.array([0, 1, 2, 4]), 2)
