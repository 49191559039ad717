"""GPU parity of moe_create_indices (moe_create_indices page) against the oracle.

Every output is integer data and must be bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _guard import check_all, guard_attrs
from _workloads import workload
from test_oracle_index import check_index_outputs

pytestmark = pytest.mark.gpu

KEYS = ("token_expert_order", "expert_start_indices", "restore_token_order", "expert_ids",
        "expert_usage_stats")


def gpu_index(ids, E):
    import moe_token_routing_gb300 as moe
    t = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)).cuda()
    bufs = moe.IndexBuffers(t.numel(), E, "cuda")
    guards = guard_attrs(bufs, KEYS + ("workspace",))
    bufs.run(t)
    check_all(guards)
    out = {k: getattr(bufs, k).cpu().numpy() for k in KEYS}
    for k in ("token_expert_order", "expert_start_indices", "restore_token_order",
              "expert_usage_stats"):
        out[k] = out[k].view(np.uint32)
    return out, bufs.device_status()


def assert_index_parity(ids, E):
    ref = oracle.create_indices(ids, E)
    got, status = gpu_index(ids, E)
    assert status == 0
    for k in KEYS:
        assert np.array_equal(got[k], ref[k]), k
    return got


@pytest.mark.parametrize("name", [c.name for c in synth.CONFIGS])
def test_parity_on_workloads(name):
    cfg, _, _, ids, _, ref = workload(name)
    got, status = gpu_index(ids, cfg.E)
    assert status == 0
    for k in KEYS:
        assert np.array_equal(got[k], ref[k]), k


@pytest.mark.parametrize("N", [0, 1, 31, 1023, 1024, 1025, 2047, 2048, 2049, 4113, 100003])
@pytest.mark.parametrize("E", [1, 3, 8, 64, 256, 1000, 1024])
def test_random_ids(N, E):
    rng = np.random.default_rng(N * 31 + E)
    ids = rng.integers(0, E, size=N).astype(np.int32)
    got = assert_index_parity(ids, E)
    check_index_outputs(ids, E, got)


def test_all_slots_on_one_expert_past_any_cache():
    ids = np.full(300001, 5, dtype=np.int32)
    got = assert_index_parity(ids, 64)
    assert got["expert_usage_stats"].tolist() == [300001, 1]


def test_hot_experts_and_idle_experts():
    """Eight hot experts far past 8192 slots each, most experts idle."""
    rng = np.random.default_rng(4)
    ids = rng.integers(0, 8, size=262144).astype(np.int32)
    ids[::97] = 100
    assert_index_parity(ids, 128)


def test_every_expert_active_descending():
    E = 1024
    ids = np.tile(np.arange(E, dtype=np.int32)[::-1], 37)
    assert_index_parity(ids, E)


def test_bad_expert_id_flagged():
    import moe_token_routing_gb300 as moe
    for N in (100, 10000):
        ids = np.zeros(N, dtype=np.int32)
        ids[N // 2] = 64  # out of range for E = 64
        ids[N // 3] = -3
        t = torch.from_numpy(ids).cuda()
        bufs = moe.create_indices(t, 64)
        assert bufs.device_status() & moe.DEVICE_STATUS_BAD_EXPERT_ID
        # a clean call on the same workspace clears the flag
        bufs.run(torch.zeros(N, dtype=torch.int32, device="cuda"))
        assert bufs.device_status() == 0


def test_workspace_checks():
    import moe_token_routing_gb300 as moe
    N, E = 10000, 64
    need = moe.moe_create_indices_workspace_size(N, E)
    assert need >= 256
    bufs = moe.IndexBuffers(N, E, "cuda")
    bufs.workspace = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    ids = torch.zeros(N, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        bufs.run(ids)
    assert ei.value.status == 6


def test_deterministic():
    cfg, _, _, ids, _, _ = workload("dsv3_prefill")
    a, _ = gpu_index(ids, cfg.E)
    b, _ = gpu_index(ids, cfg.E)
    for k in KEYS:
        assert np.array_equal(a[k], b[k])


@pytest.mark.parametrize("N,E", [(1000, 16), (2048, 256), (131072, 256), (100003, 1000), (0, 8)])
def test_scales_offsets(N, E):
    """moe_create_indices page, Args scales_offset_p: 128-row aligned offsets
    of the active experts (the alignment is the library's reading of the page)."""
    import moe_token_routing_gb300 as moe
    rng = np.random.default_rng(N + E)
    ids = rng.integers(0, E, size=N).astype(np.int32)
    ids[: N // 3] = 0  # one heavy expert
    t = torch.from_numpy(ids).cuda()
    bufs = moe.IndexBuffers(N, E, "cuda")
    scales = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    lib = moe.load_library()
    rc = lib.moe_create_indices(bufs.token_expert_order.data_ptr() if N else None,
                                bufs.expert_start_indices.data_ptr(),
                                bufs.restore_token_order.data_ptr() if N else None,
                                bufs.expert_ids.data_ptr(), bufs.expert_usage_stats.data_ptr(),
                                t.data_ptr() if N else None, N, E, bufs.workspace.data_ptr(),
                                bufs.workspace.numel(), scales.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), oracle.scales_offsets(ids, E))
    ref = oracle.create_indices(ids, E)
    for k in KEYS:
        got = getattr(bufs, k).cpu().numpy()
        if k != "expert_ids":
            got = got.view(np.uint32)
        assert np.array_equal(got, ref[k]), k


def test_one_workspace_across_sizes_and_done_counter_left_zero():
    """A workspace sized for the largest call serves smaller ones in any order:
    every call leaves the count CTAs' done counter (header word 1) at zero."""
    import moe_token_routing_gb300 as moe
    E = 256
    bufs = moe.IndexBuffers(300_000, E, "cuda")
    for N in (300_000, 1025, 5_000, 1024, 131_072, 2):
        rng = np.random.default_rng(N)
        ids = rng.integers(0, E, size=N).astype(np.int32)
        ref = oracle.create_indices(ids, E)
        t = torch.from_numpy(ids).cuda()
        lib = moe.load_library()
        rc = lib.moe_create_indices(bufs.token_expert_order.data_ptr(),
                                    bufs.expert_start_indices.data_ptr(),
                                    bufs.restore_token_order.data_ptr(), bufs.expert_ids.data_ptr(),
                                    bufs.expert_usage_stats.data_ptr(), t.data_ptr(), N, E,
                                    bufs.workspace.data_ptr(), bufs.workspace.numel(), None,
                                    torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert bufs.device_status() == 0
        assert bufs.workspace[:8].view(torch.int32)[1].item() == 0
        assert np.array_equal(bufs.token_expert_order[:N].cpu().numpy().view(np.uint32),
                              ref["token_expert_order"])
        assert np.array_equal(bufs.restore_token_order[:N].cpu().numpy().view(np.uint32),
                              ref["restore_token_order"])
        assert np.array_equal(bufs.expert_start_indices.cpu().numpy().view(np.uint32),
                              ref["expert_start_indices"])


@pytest.mark.parametrize("N,E", [(3_000_001, 64), (600_000, 1024)])
def test_long_count_rows(N, E):
    """Count rows longer than one 128-count pass of the row-prefix kernel (2930
    and 586 CTAs), with a skewed expert mix."""
    rng = np.random.default_rng(N + E)
    ids = rng.integers(0, E, size=N).astype(np.int32)
    ids[::3] = rng.integers(0, 4, size=ids[::3].size)
    assert_index_parity(ids, E)
