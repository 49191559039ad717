"""Pins for the oracle's router (group_limited_router_kernel page).

The oracle is checked against things other than itself: brute-force subset
enumeration on tiny inputs, a library top-k where the router reduces to one,
hand-derived fixtures, tie-stress inputs and invariants on every workload.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import GOLDEN

f32 = np.float32


def _beats(va, ia, vb, ib):
    """a ranks ahead of b: larger value, ties to the lower index (IEEE compare)."""
    return va > vb or (va == vb and ia < ib)


def brute_force_route(s, bias, K, G, M, norm, scale):
    """Enumerate every group subset and expert subset; keep the unique one whose
    members all rank ahead of all non-members. Group score = the largest sum of
    two distinct biased scores in the group (checks the top-2 reading without
    sorting)."""
    E = s.shape[0]
    S = E // G
    b = [f32(s[e]) + f32(bias[e]) for e in range(E)]
    g = []
    for j in range(G):
        members = range(j * S, (j + 1) * S)
        if S == 1:
            g.append(b[j * S])
        else:
            g.append(max(f32(b[p] + b[q]) for p, q in itertools.combinations(members, 2)))
    kept = None
    for sub in itertools.combinations(range(G), M):
        rest = [j for j in range(G) if j not in sub]
        if all(_beats(g[a], a, g[c], c) for a in sub for c in rest):
            assert kept is None
            kept = sub
    assert kept is not None
    allowed = [e for j in kept for e in range(j * S, (j + 1) * S)]
    chosen = None
    for sub in itertools.combinations(allowed, K):
        rest = [e for e in allowed if e not in sub]
        if all(_beats(b[a], a, b[c], c) for a in sub for c in rest):
            assert chosen is None
            chosen = sub
    assert chosen is not None
    # the chosen set also maximises the summed biased score among allowed K-subsets
    best = max(sum(float(b[e]) for e in sub) for sub in itertools.combinations(allowed, K))
    assert sum(float(b[e]) for e in chosen) == pytest.approx(best, rel=0, abs=1e-12)
    # selection order: rank order among the chosen
    order = sorted(chosen, key=lambda e: (-float(b[e]), e))
    w = np.array([float(s[e]) for e in order], dtype=np.float64)
    if norm:
        w = w / w.sum()
    return order, w * scale, kept


def _check_against_brute(scores, bias, K, G, M, norm, scale):
    ids, w = oracle.route(scores, bias, K, G, M, norm, scale)
    for t in range(scores.shape[0]):
        order, w_ref, _ = brute_force_route(scores[t], bias, K, G, M, norm, scale)
        assert list(ids[t]) == order, (t, list(ids[t]), order)
        np.testing.assert_allclose(w[t], w_ref, rtol=1e-6, atol=0)


@pytest.mark.parametrize("golden", ["route_group_limited.json", "route_ungrouped_no_norm.json"])
def test_golden_fixtures(golden):
    with open(os.path.join(GOLDEN, golden)) as fh:
        fx = json.load(fh)
    scores = np.array(fx["scores"], dtype=np.float32)
    bias = np.array(fx["bias"], dtype=np.float32)
    ids, w = oracle.route(scores, bias, fx["K"], fx["n_groups"], fx["topk_group"],
                          fx["norm_weights"], fx["scale"])
    assert ids.tolist() == fx["expected_ids"]
    np.testing.assert_allclose(w, np.array(fx["expected_weights"]), rtol=max(fx["rtol"], 1e-7),
                               atol=0)


def test_brute_force_tiny_workload():
    """The whole 64-token, 16-expert workload against subset enumeration."""
    cfg = synth.get_config("tiny")
    scores = synth.make_scores(cfg)
    bias = synth.make_bias(cfg)
    _check_against_brute(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)


@pytest.mark.parametrize("E,G,M,K", [(8, 4, 2, 3), (12, 3, 2, 4), (16, 8, 3, 4), (8, 1, 1, 2),
                                     (9, 3, 1, 3), (6, 6, 4, 3), (16, 2, 1, 8), (10, 5, 5, 10)])
@pytest.mark.parametrize("norm", [True, False])
def test_brute_force_random(E, G, M, K, norm):
    rng = np.random.default_rng(E * 1000 + G * 100 + M * 10 + K + norm)
    scores = rng.random((24, E), dtype=np.float32)
    bias = (rng.standard_normal(E) * 0.2).astype(np.float32)
    _check_against_brute(scores, bias, K, G, M, norm, 1.75)


@pytest.mark.parametrize("bias_kind", ["zero", "equal", "quantised"])
def test_tie_stress_brute_force(bias_kind):
    """Scores on a grid of 1/8 so that biased, group and expert ties are frequent."""
    rng = np.random.default_rng(7)
    E, G, M, K = 16, 4, 2, 4
    scores = (rng.integers(0, 9, size=(64, E)) / 8).astype(np.float32)
    if bias_kind == "zero":
        bias = np.zeros(E, dtype=np.float32)
    elif bias_kind == "equal":
        bias = np.full(E, 0.25, dtype=np.float32)
    else:
        bias = (rng.integers(-2, 3, size=E) / 8).astype(np.float32)
    _check_against_brute(scores, bias, K, G, M, True, 1.0)


def test_all_equal_scores_pick_lowest_indices():
    E, G, M, K = 16, 4, 2, 5
    scores = np.full((3, E), 0.5, dtype=np.float32)
    bias = np.zeros(E, dtype=np.float32)
    ids, w = oracle.route(scores, bias, K, G, M, True, 1.0)
    assert ids.tolist() == [[0, 1, 2, 3, 4]] * 3
    np.testing.assert_allclose(w, 0.2, rtol=1e-6)


@pytest.mark.parametrize("cfg_name", ["skewed_ungrouped", "few_expert_large_batch"])
def test_ungrouped_matches_library_topk(cfg_name):
    """With one group the router is a plain top-K of the biased scores: compare
    with torch.topk on the workload (tie-free: checked below)."""
    cfg = synth.get_config(cfg_name)
    T = min(cfg.T, 4096)
    scores = synth.make_scores(cfg, n_tokens=T)
    bias = synth.make_bias(cfg)
    b = torch.from_numpy(scores) + torch.from_numpy(bias)
    vals, idx = torch.topk(b, cfg.K, dim=1, largest=True, sorted=True)
    # tie-free at the K boundary and within the chosen set
    full = torch.sort(b, dim=1, descending=True).values
    if cfg.K < cfg.E:
        assert bool((full[:, cfg.K - 1] > full[:, cfg.K]).all())
    assert bool((vals[:, :-1] > vals[:, 1:]).all())
    ids, w = oracle.route(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    assert np.array_equal(ids, idx.numpy().astype(np.int32))
    s_sel = np.take_along_axis(scores.astype(np.float64), ids.astype(np.int64), axis=1)
    if cfg.norm_weights:
        s_sel = s_sel / s_sel.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w, s_sel * cfg.scale, rtol=1e-6, atol=0)


def _group_scores_f32(b, G):
    """Top-1 + top-2 of each group via a library sort (independent of the oracle)."""
    T, E = b.shape
    S = E // G
    gs = np.sort(b.reshape(T, G, S), axis=2)[:, :, ::-1]
    return gs[:, :, 0] if S == 1 else (gs[:, :, 0] + gs[:, :, 1]).astype(np.float32)


@pytest.mark.parametrize("cfg_name", ["tiny", "dsv3_decode", "dsv3_prefill", "skewed_ungrouped",
                                      "few_expert_large_batch"])
def test_invariants_on_workloads(cfg_name):
    cfg = synth.get_config(cfg_name)
    T = min(cfg.T, 8192)
    scores = synth.make_scores(cfg, n_tokens=T)
    bias = synth.make_bias(cfg)
    ids, w = oracle.route(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    S = cfg.E // cfg.G
    b = (scores + bias).astype(np.float32)
    # distinct ids in range
    assert ids.min() >= 0 and ids.max() < cfg.E
    srt = np.sort(ids, axis=1)
    assert (srt[:, 1:] != srt[:, :-1]).all()
    # ids lie only in the kept groups (kept = top-M by group score, ties to lower index)
    g = _group_scores_f32(b, cfg.G)
    order = np.lexsort((np.broadcast_to(np.arange(cfg.G), g.shape), -g.astype(np.float64)), axis=1)
    kept = order[:, :cfg.M]
    grp = ids // S
    assert all(set(grp[t]).issubset(set(kept[t])) for t in range(T))
    # selection order: biased score non-increasing along each row
    bsel = np.take_along_axis(b, ids.astype(np.int64), axis=1)
    assert (bsel[:, :-1] >= bsel[:, 1:]).all()
    # every allowed, unchosen expert ranks behind the K-th choice
    kth_v, kth_i = bsel[:, -1], ids[:, -1]
    for t in range(0, T, max(1, T // 64)):
        allowed = [e for j in kept[t] for e in range(j * S, (j + 1) * S) if e not in ids[t]]
        for e in allowed:
            assert b[t, e] < kth_v[t] or (b[t, e] == kth_v[t] and e > kth_i[t])
    # weights: unbiased scores, normalised to sum to the factor
    s_sel = np.take_along_axis(scores, ids.astype(np.int64), axis=1).astype(np.float64)
    if cfg.norm_weights:
        np.testing.assert_allclose(w.astype(np.float64).sum(axis=1), cfg.scale, rtol=1e-6)
        np.testing.assert_allclose(w, s_sel / s_sel.sum(axis=1, keepdims=True) * cfg.scale,
                                   rtol=1e-6)
    else:
        np.testing.assert_array_equal(w, (s_sel * cfg.scale).astype(np.float32))


def test_bias_changes_selection_but_not_weights():
    """Bias used for selection only: a large bias forces an expert in, and its
    weight is still its unbiased score."""
    E, G, M, K = 8, 1, 1, 2
    scores = np.array([[0.9, 0.8, 0.1, 0.7, 0.6, 0.5, 0.4, 0.3]], dtype=np.float32)
    bias = np.zeros(E, dtype=np.float32)
    bias[2] = 1.0
    ids, w = oracle.route(scores, bias, K, G, M, False, 1.0)
    assert ids.tolist() == [[2, 0]]
    assert w.tolist() == [[np.float32(0.1), np.float32(0.9)]]


@pytest.mark.parametrize("bad", [dict(G=3), dict(M=5), dict(K=9), dict(K=0), dict(M=0)])
def test_invalid_arguments_rejected(bad):
    E = 8
    p = dict(G=4, M=2, K=2)
    p.update(bad)
    scores = np.zeros((1, E), dtype=np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.route(scores, np.zeros(E, np.float32), p["K"], p["G"], p["M"], True, 1.0)
