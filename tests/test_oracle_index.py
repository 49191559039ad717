"""Pins for the oracle's index builder (moe_create_indices page).

Checked against a library stable sort, bincount-derived CSR, the inverse
permutation relation, hand-derived fixtures and the special cases the
method has (one expert, all experts, empty input, experts far past any
per-expert cache size).
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from conftest import GOLDEN


def check_index_outputs(ids_flat, E, out):
    """Everything the pages and the readings fix, derived without the oracle."""
    ids_flat = np.asarray(ids_flat, dtype=np.int64).reshape(-1)
    N = ids_flat.size
    teo = out["token_expert_order"].astype(np.int64)
    start = out["expert_start_indices"].astype(np.int64)
    restore = out["restore_token_order"].astype(np.int64)
    eids = out["expert_ids"].astype(np.int64)
    stats = out["expert_usage_stats"].astype(np.int64)
    # token_expert_order is the stable argsort of the flat expert ids
    assert np.array_equal(teo, np.argsort(ids_flat, kind="stable"))
    # restore is its inverse permutation
    assert np.array_equal(restore[teo], np.arange(N))
    assert np.array_equal(teo[restore], np.arange(N))
    # compact CSR over active experts in ascending id
    counts = np.bincount(ids_flat, minlength=E)
    active = np.nonzero(counts)[0]
    A = active.size
    assert np.array_equal(eids[:A], active)
    assert (eids[A:] == -1).all()
    expected_start = np.concatenate([[0], np.cumsum(counts[active])])
    assert np.array_equal(start[:A + 1], expected_start)
    assert (start[A:] == N).all()
    assert start[A] == N
    # each active expert's segment holds exactly its slots
    for j in range(A):
        seg = teo[start[j]:start[j + 1]]
        assert (ids_flat[seg] == active[j]).all()
    # stats = [max tokens per expert, active experts]
    assert stats.tolist() == [int(counts.max()) if N else 0, A]


def test_golden_fixture():
    with open(os.path.join(GOLDEN, "create_indices_small.json")) as fh:
        fx = json.load(fh)
    out = oracle.create_indices(np.array(fx["topk_ids"]), fx["E"])
    for key in ("token_expert_order", "expert_start_indices", "restore_token_order",
                "expert_ids", "expert_usage_stats"):
        assert out[key].tolist() == fx[key], key
    check_index_outputs(np.array(fx["topk_ids"]), fx["E"], out)


@pytest.mark.parametrize("N,E", [(1, 1), (7, 3), (256, 16), (1000, 64), (4096, 256),
                                 (20000, 1024)])
def test_random_ids(N, E):
    rng = np.random.default_rng(N + E)
    ids = rng.integers(0, E, size=N).astype(np.int32)
    check_index_outputs(ids, E, oracle.create_indices(ids, E))


def test_all_slots_on_one_expert():
    N, E = 5000, 32
    ids = np.full(N, 17, dtype=np.int32)
    out = oracle.create_indices(ids, E)
    check_index_outputs(ids, E, out)
    assert out["expert_usage_stats"].tolist() == [N, 1]
    assert out["expert_ids"][0] == 17
    assert np.array_equal(out["token_expert_order"], np.arange(N))


def test_every_expert_active():
    E = 64
    ids = np.tile(np.arange(E, dtype=np.int32)[::-1], 9)
    out = oracle.create_indices(ids, E)
    check_index_outputs(ids, E, out)
    assert out["expert_usage_stats"].tolist() == [9, E]


def test_empty():
    E = 8
    out = oracle.create_indices(np.zeros(0, dtype=np.int32), E)
    check_index_outputs(np.zeros(0), E, out)
    assert out["expert_start_indices"].tolist() == [0] * (E + 1)
    assert out["expert_usage_stats"].tolist() == [0, 0]


def test_far_past_shared_memory_cache():
    """moe_create_indices, Parameters expected_count: more than 8192 slots on one
    expert must still be placed correctly (here ~32768 per expert)."""
    rng = np.random.default_rng(3)
    ids = rng.integers(0, 8, size=262144).astype(np.int32)
    out = oracle.create_indices(ids, 8)
    check_index_outputs(ids, 8, out)
    assert out["expert_usage_stats"][0] > 8192 * 3


@pytest.mark.parametrize("cfg_name", ["tiny", "dsv3_decode", "skewed_ungrouped"])
def test_on_router_output(cfg_name):
    cfg = synth.get_config(cfg_name)
    scores = synth.make_scores(cfg)
    ids, _ = oracle.route(scores, synth.make_bias(cfg), cfg.K, cfg.G, cfg.M, cfg.norm_weights,
                          cfg.scale)
    out = oracle.create_indices(ids, cfg.E)
    check_index_outputs(ids, cfg.E, out)
    if cfg_name == "skewed_ungrouped":
        # bias 2.0 > any softmax value: every token picks experts 0..7, exactly T each
        assert out["expert_usage_stats"].tolist() == [cfg.T, 8]
        assert out["expert_ids"][:8].tolist() == list(range(8))


def test_out_of_range_id_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.create_indices(np.array([0, 3, 8], dtype=np.int32), 8)
    with pytest.raises(oracle.OracleError):
        oracle.create_indices(np.array([0, -1], dtype=np.int32), 8)
