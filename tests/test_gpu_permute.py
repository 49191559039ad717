"""GPU parity of moe_permute (expert-contiguous token rows for the grouped
matmul, moe_create_indices page) against the oracle: a pure copy, so
bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _guard import check_all, guarded
from _workloads import bits_to_f32, workload

pytestmark = pytest.mark.gpu


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def gpu_permute(x_bits, restore):
    import moe_token_routing_gb300 as moe
    r = torch.from_numpy(np.ascontiguousarray(restore, dtype=np.uint32).view(np.int32)).cuda()
    x = to_dev_bf16(x_bits)
    out, g = guarded((r.numel(), x.shape[1]), torch.bfloat16, name="permuted")
    moe.moe_permute(out, x, r)
    check_all([g])
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name", [c.name for c in synth.CONFIGS])
def test_parity_on_workloads(name):
    cfg, _, _, _, _, idx = workload(name)
    x = synth.make_input(cfg)
    got = gpu_permute(x, idx["restore_token_order"])
    ref = oracle.permute(x, idx["token_expert_order"], cfg.K)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 6, 8, 16])
@pytest.mark.parametrize("H", [8, 24, 2056])
def test_parity_shapes(K, H):
    T = 97
    rng = np.random.default_rng(K * 100 + H)
    x = synth.normal_bf16(K, 4, T * H).reshape(T, H)
    teo = rng.permutation(T * K).astype(np.uint32)
    restore = np.empty_like(teo)
    restore[teo] = np.arange(T * K, dtype=np.uint32)
    assert np.array_equal(gpu_permute(x, restore), oracle.permute(x, teo, K))


def test_round_trip_with_finalize():
    """finalize(permute(x)) with weights 1/K reproduces x bit for bit on the
    skewed workload's real index."""
    import moe_token_routing_gb300 as moe
    cfg, _, _, _, _, idx = workload("skewed_ungrouped")
    x = synth.make_input(cfg)
    r = torch.from_numpy(idx["restore_token_order"].view(np.int32)).cuda()
    down = moe.permute(to_dev_bf16(x), r)
    w = torch.full((cfg.T, cfg.K), 1.0 / cfg.K, dtype=torch.float32, device="cuda")
    out = moe.finalize(down, r, w)
    torch.cuda.synchronize()
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), x)


def test_out_of_range_entries_skipped_and_errors():
    import moe_token_routing_gb300 as moe
    T, K, H = 6, 2, 16
    x = synth.normal_bf16(9, 4, T * H).reshape(T, H)
    restore = np.arange(T * K, dtype=np.uint32)
    restore[3] = 0xFFFFFFFF
    out = torch.zeros((T * K, H), dtype=torch.bfloat16, device="cuda")
    r = torch.from_numpy(restore.view(np.int32)).cuda()
    moe.moe_permute(out, to_dev_bf16(x), r)
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    keep = np.ones(T * K, bool)
    keep[3] = False
    assert np.array_equal(got[keep], x[np.arange(T * K)[keep] // K])
    assert (got[3] == 0).all()
    lib = moe.load_library()
    st = torch.cuda.current_stream().cuda_stream
    assert lib.moe_permute(out.data_ptr(), out.data_ptr(), r.data_ptr(), T, K, H, None,
                           st) == 2


@pytest.mark.parametrize("K", [2, 5])  # the specialised kernel and the any-K kernel
def test_out_of_range_entry_sets_status(K):
    """An entry >= T*K is skipped (its slot is never written) and, with a
    status word, sets MOE_DEVICE_STATUS_BAD_RESTORE_ORDER; no fault."""
    import moe_token_routing_gb300 as moe
    T, H = 40, 72
    x = synth.normal_bf16(9, 4, T * H).reshape(T, H)
    restore = np.random.default_rng(K).permutation(T * K).astype(np.uint32)
    slot = int(restore[7])
    restore[7] = np.uint32(T * K + 3)
    r = torch.from_numpy(restore.view(np.int32)).cuda()
    out, g = guarded((T * K, H), torch.bfloat16, fill=0.0, name="permuted")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_permute(out, to_dev_bf16(x), r, device_status=status)
    check_all([g])
    assert moe.moe_read_device_status(status) == moe.DEVICE_STATUS_BAD_RESTORE_ORDER
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (got[slot] == 0).all()          # the slot the bad entry named stays unwritten
    written = np.delete(np.arange(T * K), slot)
    src = np.empty(T * K, np.int64)
    src[restore[restore < T * K]] = np.nonzero(restore < T * K)[0] // K
    assert np.array_equal(got[written], x[src[written]])
