"""moe_create_indices_no_alloc: the index build for callers that cannot
allocate device memory (for example an operator that a framework hands only
its declared input and output tensors). Its scratch is a static array inside
the library instead of a caller-provided workspace.

Checked through the C ABI against moe_create_indices on two calls in a row
with different sizes, so that the second call also shows that what the
first one left in the shared scratch does not leak into its result.
"""
import ctypes

import numpy as np
import pytest
import torch

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
    z = dict(dtype=torch.int32, device="cuda")
    return [torch.full((N,), -5, **z), torch.full((E + 1,), -5, **z), torch.full((N,), -5, **z),
            torch.full((E,), -5, **z), torch.full((2,), -5, **z)]


def _no_alloc(lib, ids, E, status):
    outs = _outputs(ids.numel(), E)
    rc = lib.moe_create_indices_no_alloc(*[t.data_ptr() for t in outs], ids.data_ptr(),
                                         ids.numel(), E, status.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == 0
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
