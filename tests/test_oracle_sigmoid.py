"""Pins for the oracle's sigmoid score loader (group_limited_router_kernel
page, Parameters scores_input_fn): error bound against float64, exact special
values, symmetry and monotonicity."""
import numpy as np
import pytest

import oracle
import synth


def _ulp_err(got, x):
    ref = 1.0 / (1.0 + np.exp(-x.astype(np.float64)))
    spacing = np.spacing(ref.astype(np.float32)).astype(np.float64)
    return np.abs(got.astype(np.float64) - ref) / spacing


def test_error_bound_on_normal_logits():
    x = synth.normal_f32(0, 1, 1 << 20, std=3.0)
    assert _ulp_err(oracle.sigmoid(x), x).max() <= 4.0


def test_error_bound_on_a_grid():
    x = np.linspace(-30, 30, 600001, dtype=np.float32)
    assert _ulp_err(oracle.sigmoid(x), x).max() <= 4.0


def test_special_values():
    x = np.array([0.0, -0.0, 200.0, -200.0, 87.0, -88.0], dtype=np.float32)
    y = oracle.sigmoid(x)
    assert y[0] == 0.5 and y[1] == 0.5
    assert y[2] == 1.0 and y[4] == 1.0
    # exp's argument is clamped to [-87, 88]: below -88 the score stays at sigmoid(-88)
    assert y[3] == y[5] and 6.0e-39 < y[5] < 6.1e-39


def test_monotone_and_symmetric():
    x = np.sort(synth.normal_f32(1, 1, 200000, std=4.0))
    y = oracle.sigmoid(x)
    assert (np.diff(y) >= 0).all()
    z = oracle.sigmoid(-x)
    assert np.abs((y.astype(np.float64) + z) - 1.0).max() < 3e-7


def test_router_on_sigmoid_scores_matches_precomputed():
    """Routing the sigmoid of the logits equals routing precomputed scores."""
    cfg = synth.get_config("dsv3_decode")
    logits = synth.normal_f32(0, synth.TENSOR_SCORES, cfg.T * cfg.E).reshape(cfg.T, cfg.E)
    scores = oracle.sigmoid(logits)
    bias = synth.make_bias(cfg)
    ids, w = oracle.route(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    assert ids.shape == (cfg.T, cfg.K)
    np.testing.assert_allclose(w.sum(1), cfg.scale, rtol=1e-6)
