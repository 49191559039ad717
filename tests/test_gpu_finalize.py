"""GPU parity of moe_finalize (moe_finalize page) against the fp32 oracle.

Gate: |gpu - ref| <= 1e-2 + 8e-3 |ref| with ref the oracle's fp32 sum before
bf16 rounding. The kernel also uses the oracle's accumulation order (k
ascending, fp32 FMA from 0), so its output is expected to equal the
round-to-nearest-even bf16 of the oracle value exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _guard import check_all, guarded
from _workloads import (bits_to_f32, f32_to_bf16_bits, finalize_tolerance_ok, workload,
                        workload_down, workload_finalize_ref)

pytestmark = pytest.mark.gpu


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def gpu_finalize(down_bits, restore, w):
    import moe_token_routing_gb300 as moe
    d = to_dev_bf16(down_bits)
    r = torch.from_numpy(np.ascontiguousarray(restore, dtype=np.uint32).view(np.int32)).cuda()
    ww = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()
    T, K = ww.shape
    out, g = guarded((T, d.shape[1]), torch.bfloat16, name="output")
    moe.moe_finalize(out, d, r, ww)
    check_all([g])
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_finalize_parity(down_bits, restore, w, T, K, H, exact=True):
    ref = oracle.finalize(down_bits, restore, w, T, K, H)
    got = gpu_finalize(down_bits, restore, w)
    ok = finalize_tolerance_ok(got, ref)
    assert ok.all(), f"{(~ok).sum()} elements outside 1e-2 + 8e-3|ref|"
    if exact:
        assert np.array_equal(got, f32_to_bf16_bits(ref))
    return got, ref


@pytest.mark.parametrize("name", [c.name for c in synth.CONFIGS])
def test_parity_on_workloads(name):
    cfg, _, _, _, w, idx = workload(name)
    down = workload_down(name)
    ref = workload_finalize_ref(name)
    got = gpu_finalize(down, idx["restore_token_order"], w)
    ok = finalize_tolerance_ok(got, ref)
    assert ok.all(), f"{(~ok).sum()} elements outside tolerance"
    assert np.array_equal(got, f32_to_bf16_bits(ref))


def _case(T, K, H, seed):
    rng = np.random.default_rng(seed)
    down = synth.normal_bf16(seed, 3, T * K * H).reshape(T * K, H)
    restore = rng.permutation(T * K).astype(np.uint32)
    w = (rng.random((T, K), dtype=np.float32) * 2 - 0.5).astype(np.float32)
    return down, restore, w


@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 6, 7, 8, 16, 32])
@pytest.mark.parametrize("H", [8, 24, 2056, 7168])
def test_parity_shapes(K, H):
    T = 37 if H >= 2048 else 129
    down, restore, w = _case(T, K, H, K * 10000 + H)
    assert_finalize_parity(down, restore, w, T, K, H)


@pytest.mark.parametrize("K", [2, 8, 3])
@pytest.mark.parametrize("T", [1, 150, 160, 300, 310, 600, 620])
def test_parity_across_launch_shapes(T, K):
    """Token counts on both sides of the launch shape's thresholds (512, 256
    and 128 threads per token at one, two and more tokens per SM; a fully
    ordered launch under four tokens per SM), with a ragged last pass of the
    row (H = 7168 is 896 chunks of 8)."""
    H = 7168
    down, restore, w = _case(T, K, H, T * 100 + K)
    assert_finalize_parity(down, restore, w, T, K, H)


def test_permutation_copy():
    """K = 1, weight 1: the output is the unpermuted rows, bit for bit."""
    T, H = 1000, 512
    down, restore, _ = _case(T, 1, H, 3)
    got = gpu_finalize(down, restore, np.ones((T, 1), np.float32))
    assert np.array_equal(got, down[restore.astype(np.int64)])


def test_zero_tokens_and_zero_hidden():
    import moe_token_routing_gb300 as moe
    for T, H in ((0, 64), (5, 0)):
        K = 2
        out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        d = torch.empty((T * K, H), dtype=torch.bfloat16, device="cuda")
        r = torch.zeros(T * K, dtype=torch.int32, device="cuda")
        w = torch.zeros((T, K), dtype=torch.float32, device="cuda")
        moe.moe_finalize(out, d, r, w)
    torch.cuda.synchronize()


def test_out_of_range_rows_are_skipped():
    T, K, H = 50, 4, 64
    down, restore, w = _case(T, K, H, 8)
    bad = restore.copy()
    bad[[3, 77, 150]] = [T * K, 0xFFFFFFFF, T * K + 5]
    got = gpu_finalize(down, bad, w)
    w2 = w.copy().reshape(-1)
    w2[[3, 77, 150]] = 0.0
    ref = oracle.finalize(down, np.where(bad < T * K, bad, 0).astype(np.uint32),
                          w2.reshape(T, K), T, K, H)
    assert finalize_tolerance_ok(got, ref).all()


def test_argument_errors():
    import moe_token_routing_gb300 as moe
    lib = moe.load_library()
    st = torch.cuda.current_stream().cuda_stream
    T, K, H = 4, 2, 64
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    d = torch.empty((T * K + 1, H), dtype=torch.bfloat16, device="cuda")
    r = torch.zeros(T * K, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, K), dtype=torch.float32, device="cuda")
    p = (out.data_ptr(), d.data_ptr(), r.data_ptr(), w.data_ptr())
    assert lib.moe_finalize(*p, T, K, 60, st) == 4          # H % 8
    assert lib.moe_finalize(*p, T, 33, H, st) == 4          # K > 32
    assert lib.moe_finalize(*p, T, 0, H, st) == 2           # K < 1
    assert lib.moe_finalize(p[0] + 2, *p[1:], T, K, H, st) == 3   # output not 16-byte aligned
    assert lib.moe_finalize(p[0], p[1] + 8, *p[2:], T, K, H, st) == 3
    assert lib.moe_finalize(None, *p[1:], T, K, H, st) == 1
    assert lib.moe_finalize(p[1], p[1], p[2], p[3], T, K, H, st) == 2   # output overlaps down


def test_deterministic():
    cfg, _, _, _, w, idx = workload("skewed_ungrouped")
    down = workload_down("skewed_ungrouped")
    a = gpu_finalize(down, idx["restore_token_order"], w)
    b = gpu_finalize(down, idx["restore_token_order"], w)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("w_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [2, 3, 8])
def test_finalize_ex_dtypes(w_dtype, out_dtype, K):
    """moe_finalize page, Parameters weight_type / out_type: bf16 weights widen
    exactly to fp32; an fp32 output is the oracle's fp32 sum bit for bit."""
    import moe_token_routing_gb300 as moe
    T, H = 211, 1032
    down, restore, w = _case(T, K, H, K + 77)
    if w_dtype == "bf16":
        w_bits = f32_to_bf16_bits(w)
        w_ref = bits_to_f32(w_bits).reshape(T, K)
        w_dev = torch.from_numpy(w_bits.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        w_ref = w
        w_dev = torch.from_numpy(w).cuda()
    ref = oracle.finalize(down, restore, w_ref, T, K, H)
    tdt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out = torch.empty((T, H), dtype=tdt, device="cuda")
    r = torch.from_numpy(restore.view(np.int32)).cuda()
    moe.moe_finalize_ex(out, to_dev_bf16(down), r, w_dev)
    torch.cuda.synchronize()
    if out_dtype == "f32":
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    else:
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert finalize_tolerance_ok(got, ref).all()
        assert np.array_equal(got, f32_to_bf16_bits(ref))


def test_finalize_ex_default_types_match_finalize():
    import moe_token_routing_gb300 as moe
    cfg, _, _, _, w, idx = workload("tiny")
    down = workload_down("tiny")
    r = torch.from_numpy(idx["restore_token_order"].view(np.int32)).cuda()
    d = to_dev_bf16(down)
    wd = torch.from_numpy(w).cuda()
    a = moe.finalize(d, r, wd)
    b = torch.empty_like(a)
    moe.moe_finalize_ex(b, d, r, wd)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("K", [8, 3])  # the specialised kernel and the any-K kernel
def test_out_of_range_restore_entry_sets_status(K):
    """Page moe_finalize, Args restore_order: an entry >= T*K (corrupt index
    data) is skipped and never read; with a status word moe_finalize_ex
    records MOE_DEVICE_STATUS_BAD_RESTORE_ORDER instead of faulting or
    trapping. Every other token's row is the oracle's, bit for bit, and the
    bad token's row is the oracle's with that term left out."""
    import moe_token_routing_gb300 as moe
    T, H = 97, 520
    down, restore, w = _case(T, K, H, 1000 + K)
    bad = restore.copy()
    bad[5 * K + 1] = T * K          # first value past the end
    bad[(T - 1) * K] = 0xFFFFFFFF   # the largest value
    d, wd = to_dev_bf16(down), torch.from_numpy(w).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # a clean call leaves the word at zero
    out, g = guarded((T, H), torch.bfloat16, name="output")
    moe.moe_finalize_ex(out, d, torch.from_numpy(restore.view(np.int32)).cuda(), wd,
                        device_status=status)
    check_all([g])
    assert moe.moe_read_device_status(status) == 0
    out, g = guarded((T, H), torch.bfloat16, name="output")
    moe.moe_finalize_ex(out, d, torch.from_numpy(bad.view(np.int32)).cuda(), wd,
                        device_status=status)
    check_all([g])
    assert moe.moe_read_device_status(status) == moe.DEVICE_STATUS_BAD_RESTORE_ORDER
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    # the reference with the two bad terms dropped: weight 0 on a valid row
    w_drop = w.copy()
    w_drop[5, 1] = 0.0
    w_drop[T - 1, 0] = 0.0
    ref = oracle.finalize(down, restore, w_drop, T, K, H)
    assert finalize_tolerance_ok(got, ref).all()
    good = np.ones(T, bool)
    good[[5, T - 1]] = False
    assert np.array_equal(got[good], f32_to_bf16_bits(ref)[good])
