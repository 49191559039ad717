"""Pins for the oracle's softmax score loader (group_limited_router_kernel
page, Parameters scores_input_fn): error bound against float64 derived from
the arithmetic, exact special cases, shift invariance and row sums."""
import numpy as np
import pytest

import oracle
import synth


def _ref64(x):
    x = x.astype(np.float64)
    z = np.exp(x - x.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def _bound(E):
    """Relative error bound: exp within 4 ulp (the sigmoid pins), the
    sequential fp32 sum of E positive terms within (E-1) half-ulps, and one
    rounded division."""
    u = 2.0 ** -24
    return 8 * u + (E - 1) * u + u


@pytest.mark.parametrize("E", [8, 64, 256, 1024])
def test_error_bound_against_float64(E):
    x = synth.normal_f32(3, 1, 512 * E, std=2.5).reshape(512, E)
    got = oracle.softmax(x).astype(np.float64)
    ref = _ref64(x)
    rel = np.abs(got - ref) / ref
    assert rel.max() <= _bound(E)


def test_large_logits_need_the_max_shift():
    """Logits near 100: exp(x) itself would saturate, exp(x - max) does not."""
    x = (100.0 + synth.normal_f32(4, 1, 64 * 256, std=1.0)).astype(np.float32).reshape(64, 256)
    got = oracle.softmax(x).astype(np.float64)
    assert (np.abs(got - _ref64(x)) / _ref64(x)).max() <= _bound(256)


def test_all_equal_row_is_exactly_uniform():
    for v in (0.0, -3.5, 77.0):
        x = np.full((3, 256), v, dtype=np.float32)
        assert (oracle.softmax(x) == np.float32(1.0 / 256)).all()


def test_one_dominant_logit():
    x = np.full((1, 256), -200.0, dtype=np.float32)
    x[0, 17] = 0.0
    y = oracle.softmax(x)[0]
    assert y[17] == 1.0
    # exp's argument is clamped at -87
    assert (np.delete(y, 17) == y[0]).all() and 1.6e-38 < y[0] < 1.7e-38


def test_shift_invariance_on_integer_logits():
    rng = np.random.default_rng(7)
    x = rng.integers(-20, 20, size=(50, 128)).astype(np.float32)
    assert np.array_equal(oracle.softmax(x), oracle.softmax(x + np.float32(64.0)))


def test_rows_sum_to_one():
    x = synth.normal_f32(5, 1, 300 * 256, std=3.0).reshape(300, 256)
    s = oracle.softmax(x).astype(np.float64).sum(axis=1)
    assert np.abs(s - 1.0).max() <= 256 * _bound(256)


def test_router_on_softmax_scores():
    """Routing the softmax of the logits: weights renormalise to the scale."""
    cfg = synth.get_config("dsv3_decode")
    logits = synth.normal_f32(0, synth.TENSOR_SCORES, cfg.T * cfg.E).reshape(cfg.T, cfg.E)
    ids, w = oracle.route(oracle.softmax(logits), synth.make_bias(cfg), cfg.K, cfg.G, cfg.M,
                          cfg.norm_weights, cfg.scale)
    assert ids.shape == (cfg.T, cfg.K)
    np.testing.assert_allclose(w.sum(1), cfg.scale, rtol=1e-6)
