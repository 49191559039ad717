"""moe_create_indices_no_alloc: the index build for callers that cannot
allocate device memory (for example an operator that a framework hands only
its declared input and output tensors). Its scratch is a static array inside
the library instead of a caller-provided workspace.

Checked through the C ABI against moe_create_indices on two calls in a row
with different sizes, so that the second call also shows that what the
first one left in the shared scratch does not leak into its result; against
the CPU oracle element by element (the prefill workload's router output, a
single-CTA case and the largest request the 1 MiB scratch accepts); and for
the first request it refuses.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from _guard import check_all, guarded

pytestmark = pytest.mark.gpu

MAX_SCRATCH = 1 << 20  # MOE_NO_ALLOC_SCRATCH_BYTES


def _lib():
    import moe_token_routing_gb300 as moe
    lib = moe.load_library()
    f = lib.moe_create_indices_no_alloc
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int32, vp, vp]
    f.restype = ctypes.c_int
    return moe, lib


def _outputs(N, E):
    shapes = ((N,), (E + 1,), (N,), (E,), (2,))
    names = ("token_expert_order", "expert_start_indices", "restore_token_order", "expert_ids",
             "expert_usage_stats")
    pairs = [guarded(sh, torch.int32, fill=-5, name=n) for sh, n in zip(shapes, names)]
    return [p[0] for p in pairs], [p[1] for p in pairs]


def _no_alloc(lib, ids, E, status):
    outs, guards = _outputs(ids.numel(), E)
    rc = lib.moe_create_indices_no_alloc(*[t.data_ptr() for t in outs], ids.data_ptr(),
                                         ids.numel(), E, status.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    check_all(guards)
    return outs


def _with_workspace(moe, ids, E):
    b = moe.create_indices(ids, E)
    return [b.token_expert_order, b.expert_start_indices, b.restore_token_order, b.expert_ids,
            b.expert_usage_stats]


def test_matches_workspace_entry_point_on_two_calls_in_a_row():
    moe, lib = _lib()
    rng = np.random.default_rng(2024)
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    cases = [(131072, 256), (50000, 64)]  # multi-CTA path both times, different layouts
    for N, E in cases:
        assert moe.moe_create_indices_workspace_size(N, E) <= MAX_SCRATCH
        ids = torch.from_numpy(rng.integers(0, E, size=N).astype(np.int32)).cuda()
        got = _no_alloc(lib, ids, E, status)
        ref = _with_workspace(moe, ids, E)
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            assert torch.equal(g, r)
        assert int(status.item()) == 0


def test_small_case_and_bad_id_status():
    moe, lib = _lib()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids = torch.tensor([3, 1, 3, 0, 9], dtype=torch.int32, device="cuda")  # 9 >= E
    _no_alloc(lib, ids, 8, status)
    torch.cuda.synchronize()
    assert int(status.item()) & moe.DEVICE_STATUS_BAD_EXPERT_ID
    ok = torch.tensor([3, 1, 3, 0, 2], dtype=torch.int32, device="cuda")
    got = _no_alloc(lib, ok, 8, status)
    ref = _with_workspace(moe, ok, 8)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for g, r in zip(got, ref):
        assert torch.equal(g, r)


def test_rejects_requests_beyond_the_scratch_size():
    moe, lib = _lib()
    N, E = 8_000_000, 1024
    assert moe.moe_create_indices_workspace_size(N, E) > MAX_SCRATCH
    fake = 0x7f0000001000  # never dereferenced: the call fails before enqueueing
    rc = lib.moe_create_indices_no_alloc(fake, fake, fake, fake, fake, fake, N, E, None, None)
    assert rc == 6  # MOE_ERR_WORKSPACE


INDEX_KEYS = ("token_expert_order", "expert_start_indices", "restore_token_order", "expert_ids",
              "expert_usage_stats")


def _assert_matches_oracle(got, ids_np, E):
    ref = oracle.create_indices(ids_np, E)
    for k, g in zip(INDEX_KEYS, got):
        r = ref[k]
        g = g.cpu().numpy()
        g = g if k == "expert_ids" else g.view(np.uint32)
        assert np.array_equal(g, r), k


@pytest.mark.parametrize("case", ["prefill_router_ids", "single_cta", "largest_accepted"])
def test_matches_oracle(case):
    """Element by element against the oracle's bucket sort (page
    moe_create_indices: every output), twice in a row on the shared scratch."""
    moe, lib = _lib()
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    if case == "prefill_router_ids":
        from _workloads import workload
        cfg, _, _, ids_ref, _, _ = workload("dsv3_prefill")
        ids_np, E = ids_ref.reshape(-1).astype(np.int32), cfg.E
    elif case == "single_cta":
        ids_np, E = np.random.default_rng(5).integers(0, 16, size=1000).astype(np.int32), 16
    else:
        E = 256
        N = 1_040_384  # the largest num_slots over 256 experts that fits 1 MiB
        assert moe.moe_create_indices_workspace_size(N, E) <= MAX_SCRATCH
        assert moe.moe_create_indices_workspace_size(N + 1, E) > MAX_SCRATCH
        ids_np = np.random.default_rng(6).integers(0, E, size=N).astype(np.int32)
    ids = torch.from_numpy(ids_np).cuda()
    for _ in range(2):
        got = _no_alloc(lib, ids, E, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _assert_matches_oracle(got, ids_np, E)


def test_rejects_the_first_request_over_the_limit():
    moe, lib = _lib()
    for N, E in ((1_040_385, 256), (1 << 20, 256), (2_076_673, 128)):
        assert moe.moe_create_indices_workspace_size(N, E) > MAX_SCRATCH
        fake = 0x7f0000001000  # never dereferenced: the call fails before enqueueing
        rc = lib.moe_create_indices_no_alloc(fake, fake, fake, fake, fake, fake, N, E, None, None)
        assert rc == 6  # MOE_ERR_WORKSPACE
