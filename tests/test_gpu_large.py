"""Parity past 2^31 elements: the router on a score matrix, finalize on a
`down` matrix and permute on an output of more than 2^31 elements, so that
every offset into them needs 64-bit arithmetic. The oracle checks sampled
rows (the first ones, those on both sides of element 2^31, the last ones and
random ones) one by one; the index build on the router's slots (up to 135
million) is checked against the definitions of its outputs (inverse permutation, stable
order within each expert, counts, compact CSR, stats) on the whole arrays.

Inputs come from torch's seeded generator on the device (uniform scores,
normal `down`, a random permutation as the restore order); the sampled rows
are copied to the host for the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from _guard import check_all, guarded
from _workloads import f32_to_bf16_bits, finalize_tolerance_ok

pytestmark = pytest.mark.gpu

TWO31 = 1 << 31


def _moe():
    import moe_token_routing_gb300 as moe
    moe.load_library()
    return moe


def _sample_rows(n_rows, boundary_row, seed, k=300, n_random=1000):
    rng = np.random.default_rng(seed)
    parts = [np.arange(0, k), np.arange(boundary_row - k, boundary_row + k),
             np.arange(n_rows - k, n_rows), rng.integers(0, n_rows, n_random)]
    return np.unique(np.concatenate(parts).clip(0, n_rows - 1))


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("E,G,M,K", [(256, 8, 4, 8), (1024, 32, 4, 8), (200, 8, 4, 6),
                                     (32, 4, 2, 2)],
                         ids=["staged", "segment", "warp", "thread"])
def test_router_and_index_past_2_31_score_elements(E, G, M, K):
    """More than 2^31 scores (about 8.9 GB) in each router layout: the
    DeepSeek-V3 shape (256 experts in 8 groups, top-4 groups, K = 8; 8.65
    million tokens, a ragged last chunk, thousands of ring buffer turns per
    warp), 1024 experts in 32 groups (segment layout), 200 experts in 8
    groups of 25 (warp layout) and 32 experts in 4 groups (thread layout, 67
    million tokens)."""
    moe = _moe()
    boundary = TWO31 // E
    T = boundary + 262144 + 3
    gen = torch.Generator(device="cuda").manual_seed(20231 + E)
    s = torch.rand((T, E), generator=gen, device="cuda", dtype=torch.float32)
    bias = torch.randn(E, generator=gen, device="cuda", dtype=torch.float32) * 0.05
    ids, gi = guarded((T, K), torch.int32, name="expert_indices")
    w, gw = guarded((T, K), torch.float32, name="expert_weights")
    moe.moe_route(ids, w, s, bias, G, M, True, 2.5)
    check_all([gi, gw])

    rows = _sample_rows(T, boundary, E)
    sel = torch.from_numpy(rows).cuda()
    ids_ref, w_ref = oracle.route(s.index_select(0, sel).cpu().numpy(), bias.cpu().numpy(),
                                  K, G, M, True, 2.5)
    got_ids = ids.index_select(0, sel).cpu().numpy()
    bad = np.nonzero((got_ids != ids_ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} sampled rows differ, first token {rows[bad[:1]]}"
    assert np.array_equal(w.index_select(0, sel).cpu().numpy().view(np.uint32),
                          w_ref.view(np.uint32))

    # the same router counting its own output, then the index build over
    # N = T*K slots (17 to 135 million)
    bufs = moe.RouteIndexBuffers(T, E, K, "cuda")
    bufs.run(s, bias, G, M, True, 2.5)
    del s
    _free()
    assert bufs.device_status() == 0
    assert torch.equal(bufs.expert_indices, ids)
    assert torch.equal(bufs.expert_weights.view(torch.int32), w.view(torch.int32))
    flat = ids.reshape(-1).long()
    del ids, w, gi, gw
    _free()
    _check_index(bufs, flat, E)
    del bufs, flat
    _free()


def _check_index(bufs, flat, E):
    """The index outputs in `bufs` against their definitions for the flat
    expert ids `flat` (int64 on the device), on the whole arrays."""
    N = flat.numel()
    order = bufs.token_expert_order.long()
    restore = bufs.restore_token_order.long()
    # restore_token_order is the inverse permutation of token_expert_order
    assert torch.equal(order[restore], torch.arange(N, device="cuda"))
    del restore
    _free()
    # experts ascend along the order, and slots ascend within each expert
    e_sorted = flat[order]
    assert bool((e_sorted[1:] >= e_sorted[:-1]).all())
    same = e_sorted[1:] == e_sorted[:-1]
    assert bool((order[1:] > order[:-1])[same].all())
    del order, same
    _free()
    # the order's experts are the sorted ids
    assert torch.equal(e_sorted, torch.sort(flat).values)
    del e_sorted
    _free()
    # compact CSR over the active experts, expert_ids, stats
    counts = torch.bincount(flat, minlength=E)
    active = torch.nonzero(counts).reshape(-1)
    A = active.numel()
    starts = torch.cat([torch.zeros(1, dtype=torch.long, device="cuda"),
                        torch.cumsum(counts[active], 0)])
    csr = bufs.expert_start_indices.long()
    assert torch.equal(csr[:A + 1], starts)
    assert bool((csr[A + 1:] == N).all())
    eids = bufs.expert_ids.long()
    assert torch.equal(eids[:A], active)
    assert bool((eids[A:] == -1).all())
    assert bufs.expert_usage_stats.cpu().tolist() == [int(counts.max()), A]


def test_create_indices_on_134_million_slots():
    """The separate index build (count, rows and scatter kernels) on 2^27 + 5
    slots over 256 experts, ids from a skewed draw (expert e with weight
    proportional to e + 1), against the definitions of its outputs."""
    moe = _moe()
    E, N = 256, (1 << 27) + 5
    gen = torch.Generator(device="cuda").manual_seed(20234)
    p = torch.arange(1, E + 1, dtype=torch.float32, device="cuda")
    ids = torch.multinomial(p, 1 << 20, replacement=True, generator=gen).to(torch.int32)
    reps = -(-N // ids.numel())
    perm = torch.randperm(ids.numel() * reps, generator=gen, device="cuda")
    flat_ids = ids.repeat(reps)[perm][:N].contiguous()
    del perm
    bufs = moe.create_indices(flat_ids, E)
    assert bufs.device_status() == 0
    _check_index(bufs, flat_ids.long(), E)
    del bufs, flat_ids, ids
    _free()


def test_single_launch_route_index_past_2_31_score_elements():
    """The cooperative single-launch router + index on the DeepSeek-V3 shape
    over 8.65 million tokens (more than 2^31 scores): the same ids and weights
    as moe_route on sampled rows' oracle results, and index outputs that meet
    their definitions."""
    moe = _moe()
    E, G, M, K = 256, 8, 4, 8
    boundary = TWO31 // E
    T = boundary + 262144 + 3
    gen = torch.Generator(device="cuda").manual_seed(20235)
    s = torch.rand((T, E), generator=gen, device="cuda", dtype=torch.float32)
    bias = torch.randn(E, generator=gen, device="cuda", dtype=torch.float32) * 0.05
    bufs = moe.RouteIndexBuffers(T, E, K, "cuda", single_launch=True)
    bufs.run(s, bias, G, M, True, 2.5)
    assert bufs.device_status() == 0
    rows = _sample_rows(T, boundary, 3)
    sel = torch.from_numpy(rows).cuda()
    ids_ref, w_ref = oracle.route(s.index_select(0, sel).cpu().numpy(), bias.cpu().numpy(),
                                  K, G, M, True, 2.5)
    del s
    _free()
    assert np.array_equal(bufs.expert_indices.index_select(0, sel).cpu().numpy(), ids_ref)
    assert np.array_equal(bufs.expert_weights.index_select(0, sel).cpu().numpy().view(np.uint32),
                          w_ref.view(np.uint32))
    _check_index(bufs, bufs.expert_indices.reshape(-1).long(), E)
    del bufs
    _free()


@pytest.mark.parametrize("fn", ["sigmoid", "softmax"])
def test_score_loaders_past_2_31_logits(fn):
    """The fused sigmoid and softmax loaders on the DeepSeek-V3 router shape
    over 8.65 million tokens of gate logits (more than 2^31 of them), sampled
    rows against the oracle's loader followed by its router."""
    moe = _moe()
    E, G, M, K = 256, 8, 4, 8
    boundary = TWO31 // E
    T = boundary + 262144 + 3
    gen = torch.Generator(device="cuda").manual_seed(20236 + len(fn))
    x = torch.randn((T, E), generator=gen, device="cuda", dtype=torch.float32)
    bias = torch.randn(E, generator=gen, device="cuda", dtype=torch.float32) * 0.05
    ids, gi = guarded((T, K), torch.int32, name="expert_indices")
    w, gw = guarded((T, K), torch.float32, name="expert_weights")
    code = moe.SCORES_SIGMOID if fn == "sigmoid" else moe.SCORES_SOFTMAX
    moe.moe_route_ex(ids, w, x, bias, G, M, True, 2.5, code)
    check_all([gi, gw])
    rows = _sample_rows(T, boundary, 4 + len(fn))
    sel = torch.from_numpy(rows).cuda()
    load = oracle.sigmoid if fn == "sigmoid" else oracle.softmax
    ids_ref, w_ref = oracle.route(load(x.index_select(0, sel).cpu().numpy()), bias.cpu().numpy(),
                                  K, G, M, True, 2.5)
    assert np.array_equal(ids.index_select(0, sel).cpu().numpy(), ids_ref)
    assert np.array_equal(w.index_select(0, sel).cpu().numpy().view(np.uint32),
                          w_ref.view(np.uint32))
    del x, ids, w, gi, gw
    _free()


@pytest.mark.parametrize("K", [8, 16])
def test_finalize_past_2_31_down_elements(K):
    """The prefill row width (H = 7168) over 320 000 slots (40 000 tokens of
    K = 8, or 20 000 of K = 16, the kernel for any K): `down` holds 2.29
    billion bf16 values (4.6 GB), and the restore order is a random
    permutation, so sampled tokens gather rows on both sides of element 2^31."""
    moe = _moe()
    T, H = 320000 // K, 7168
    N = T * K
    assert N * H > TWO31
    gen = torch.Generator(device="cuda").manual_seed(20232)
    down = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, N, 32768):
        r1 = min(N, r0 + 32768)
        down[r0:r1] = torch.randn((r1 - r0, H), generator=gen, device="cuda").to(torch.bfloat16)
    restore = torch.randperm(N, generator=gen, device="cuda").to(torch.int32)
    w = torch.rand((T, K), generator=gen, device="cuda", dtype=torch.float32) * 2 - 0.5
    out, g = guarded((T, H), torch.bfloat16, name="output")
    moe.moe_finalize(out, down, restore, w)
    check_all([g])

    # tokens whose rows lie past element 2^31 among the sampled ones
    far_row = TWO31 // H
    tok = _sample_rows(T, T // 2, 2)
    r_s = restore.reshape(T, K)[torch.from_numpy(tok).cuda()].long()
    assert int((r_s >= far_row).sum()) > 0
    # the oracle on the sampled tokens: their K rows gathered in order, so
    # that token j of the sample reads rows j*K .. j*K+K-1
    rows_c = down.index_select(0, r_s.reshape(-1)).view(torch.int16).cpu().numpy().view(np.uint16)
    S = tok.size
    w_c = w[torch.from_numpy(tok).cuda()].cpu().numpy()
    ref = oracle.finalize(rows_c, np.arange(S * K, dtype=np.uint32), w_c, S, K, H)
    got = out[torch.from_numpy(tok).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    ok = finalize_tolerance_ok(got, ref)
    assert ok.all(), f"{(~ok).sum()} elements outside 1e-2 + 8e-3|ref|"
    assert np.array_equal(got, f32_to_bf16_bits(ref))
    del down, restore, w, out, g
    _free()


def test_permute_past_2_31_output_elements():
    """permuted[restore[t*K + k]] = input[t] with T*K*H above 2^31 (the prefill
    row width, K = 8, 40 000 tokens), checked on every slot."""
    moe = _moe()
    T, K, H = 40000, 8, 7168
    N = T * K
    gen = torch.Generator(device="cuda").manual_seed(20233)
    x = torch.randn((T, H), generator=gen, device="cuda").to(torch.bfloat16)
    restore = torch.randperm(N, generator=gen, device="cuda").to(torch.int32)
    out, g = guarded((N, H), torch.bfloat16, name="permuted")
    moe.moe_permute(out, x, restore)
    check_all([g])
    src = torch.arange(N, device="cuda") // K
    r = restore.long()
    for i0 in range(0, N, 65536):
        i1 = min(N, i0 + 65536)
        assert torch.equal(out[r[i0:i1]].view(torch.int16), x[src[i0:i1]].view(torch.int16)), i0
    del x, restore, out, g, src, r
    _free()
