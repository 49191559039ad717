"""Pins for the oracle's aligned scale offsets (moe_create_indices page, Args
scales_offset_p; the 128-row alignment is the library's reading of the page)."""
import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def test_golden_fixture():
    with open(os.path.join(GOLDEN, "scales_offsets_small.json")) as fh:
        fx = json.load(fh)
    ids = np.repeat(np.arange(fx["E"]), fx["counts"]).astype(np.int32)
    np.random.default_rng(0).shuffle(ids)
    out = oracle.scales_offsets(ids, fx["E"], fx["row_align"])
    assert out.tolist() == fx["expected"]


@pytest.mark.parametrize("N,E,align", [(0, 5, 128), (1, 1, 128), (5000, 64, 128), (777, 9, 32),
                                       (300000, 256, 128)])
def test_properties(N, E, align):
    rng = np.random.default_rng(N + E)
    ids = rng.integers(0, E, size=N).astype(np.int32)
    out = oracle.scales_offsets(ids, E, align).astype(np.int64)
    counts = np.bincount(ids, minlength=E)
    active = counts[counts > 0]
    A = active.size
    padded = -(-active // align) * align
    assert np.array_equal(out[:A], np.concatenate([[0], np.cumsum(padded)[:-1]]) if A else [])
    assert (out[A:] == padded.sum()).all()
    assert (out % align == 0).all()
    assert (np.diff(out[:A + 1]) >= active).all()
    # same segment order as the CSR of create_indices
    idx = oracle.create_indices(ids, E)
    assert idx["expert_usage_stats"][1] == A
