"""The seeded generators: determinism, random access and the distributions the
workloads ask for."""
import numpy as np
import pytest

import synth


def test_deterministic_and_seekable():
    a = synth.normal_f32(0, 5, 10001)
    b = synth.normal_f32(0, 5, 10001, threads=1)
    assert np.array_equal(a, b)
    c = synth.normal_f32(0, 5, 501, first=4321)
    assert np.array_equal(c, a[4321:4822])
    assert not np.array_equal(a, synth.normal_f32(1, 5, 10001))
    assert not np.array_equal(a, synth.normal_f32(0, 6, 10001))


def test_bf16_rows_regenerate():
    cfg = synth.get_config("tiny")
    full = synth.make_down(cfg)
    part = synth.make_down(cfg, first_row=17, n_rows=9)
    assert np.array_equal(part, full[17:26])


def test_normal_moments():
    x = synth.normal_f32(3, 1, 1 << 20).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    y = synth.normal_f32(3, 2, 1 << 20, std=0.05).astype(np.float64)
    assert abs(y.std() - 0.05) < 5e-4


@pytest.mark.parametrize("cfg", synth.CONFIGS, ids=lambda c: c.name)
def test_workload_recipes(cfg):
    T = min(cfg.T, 2048)
    s = synth.make_scores(cfg, n_tokens=T)
    assert s.shape == (T, cfg.E) and s.dtype == np.float32
    assert (s > 0).all() and (s < 1).all()
    if cfg.scores == "softmax":
        np.testing.assert_allclose(s.astype(np.float64).sum(1), 1.0, rtol=1e-5)
    b = synth.make_bias(cfg)
    assert b.shape == (cfg.E,)
    if cfg.bias == "hot":
        assert (b[:cfg.hot_experts] == cfg.hot_bias).all() and (b[cfg.hot_experts:] == 0).all()
    d = synth.make_down(cfg, n_rows=4)
    assert d.shape == (4, cfg.H) and d.dtype == np.uint16


def test_config_table():
    names = [c.name for c in synth.CONFIGS]
    assert names == ["tiny", "dsv3_decode", "dsv3_prefill", "skewed_ungrouped",
                     "few_expert_large_batch"]
    c2 = synth.get_config("dsv3_prefill")
    assert (c2.T, c2.E, c2.G, c2.M, c2.K, c2.H, c2.scale) == (16384, 256, 8, 4, 8, 7168, 2.5)
    assert c2.N * c2.H * 2 == 1879048192
