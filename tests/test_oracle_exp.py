"""Independent pin of the exp inside the oracle's score loaders
(group_limited_router_kernel page, Parameters scores_input_fn): the oracle's
fp32 exp against double-precision exp at every float32 binade endpoint of
the clamp range [-87, 88], their neighbours, and a dense sample.

Bound, from the arithmetic: n * ln2_head is exact (the head has 12 trailing
zero bits and |n| <= 127); the tail step adds at most half an ulp of r,
|r| <= ln2/2, so below 0.35 ulp of exp(r); Horner's rule with seven fused
multiply-adds adds at most about one ulp; the degree-8 truncation term
(ln2/2)^8 / 8! is below 0.05 ulp; scaling by 2^n is exact for the normal
results of the clamp range. Hence 2 ulp.
"""
import numpy as np

import oracle

BOUND_ULP = 2.0


def _ulp_err(x):
    got = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(np.clip(x.astype(np.float64), -87.0, 88.0))
    spacing = np.spacing(ref.astype(np.float32)).astype(np.float64)
    return np.abs(got - ref) / spacing


def _binade_endpoints():
    xs = []
    for k in range(-149, 7):
        for s in (1.0, -1.0):
            lo = np.float32(s * 2.0 ** k)                                  # first of the binade
            hi = np.nextafter(np.float32(s * 2.0 ** (k + 1)), np.float32(0))  # last of the binade
            for v in (lo, hi, np.nextafter(lo, np.float32(0)), np.nextafter(hi, np.float32(s * 1e30))):
                if -87.0 <= v <= 88.0:
                    xs.append(v)
    xs += [np.float32(-87.0), np.float32(88.0), np.float32(0.0), np.float32(-0.0)]
    return np.array(xs, dtype=np.float32)


def test_binade_endpoints_within_bound():
    x = _binade_endpoints()
    assert x.size > 1000
    assert _ulp_err(x).max() <= BOUND_ULP


def test_dense_sample_within_bound():
    x = np.random.default_rng(11).uniform(-87.0, 88.0, 1 << 20).astype(np.float32)
    assert _ulp_err(x).max() <= BOUND_ULP


def test_exact_points_and_clamp():
    e = oracle.exp_f32(np.array([0.0, -0.0, -87.0, -1000.0, 88.0, 1000.0], dtype=np.float32))
    assert e[0] == 1.0 and e[1] == 1.0
    assert e[3] == e[2] and e[5] == e[4]       # the argument is clamped to [-87, 88]
    assert np.isfinite(e).all() and e[2] > np.finfo(np.float32).tiny


def test_monotone_on_a_fine_grid():
    x = np.linspace(-87.0, 88.0, 1_000_001, dtype=np.float32)
    assert (np.diff(oracle.exp_f32(x)) >= 0).all()
