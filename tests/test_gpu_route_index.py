"""GPU parity of moe_route_index and moe_route_index_single_launch: the
group-limited router (page "group_limited_router_kernel") and the index build
(page "moe_create_indices"), with the router counting its own output or in one
cooperative launch, against the oracle's route followed by its create_indices.

Ids and every index output are bit-exact; the weights are the router's fp32
arithmetic and are compared bit for bit as well (the same device code makes
them). The bounded wait of the cross-CTA hand-off is driven by a small
harness (tests/cuda) on a word that nothing tags: it must give up within its
one-second bound and leave the GPU usable.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _guard import check_all, guard_attrs, guarded
from _workloads import workload

pytestmark = pytest.mark.gpu

INDEX_KEYS = ("token_expert_order", "expert_start_indices", "restore_token_order", "expert_ids",
              "expert_usage_stats")


def _moe():
    import moe_token_routing_gb300 as moe
    moe.load_library()
    return moe


def gpu_route_index(scores, bias, K, G, M, norm, scale, score_fn=0, scales=False, bufs=None,
                    single=False):
    moe = _moe()
    s = torch.from_numpy(np.ascontiguousarray(scores)).cuda()
    b = torch.from_numpy(np.ascontiguousarray(bias)).cuda()
    T, E = scores.shape
    if bufs is None:
        bufs = moe.RouteIndexBuffers(T, E, K, "cuda", single_launch=single)
    if not hasattr(bufs, "_guards"):
        bufs._guards = guard_attrs(bufs, ("expert_indices", "expert_weights") + INDEX_KEYS
                                   + ("workspace",))
    so = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda") if scales else None
    bufs.run(s, b, G, M, norm, scale, score_fn, scales_offset=so)
    check_all(bufs._guards)
    out = {k: getattr(bufs, k).cpu().numpy() for k in INDEX_KEYS}
    for k in INDEX_KEYS:
        if k != "expert_ids":
            out[k] = out[k].view(np.uint32)
    out["ids"] = bufs.expert_indices.cpu().numpy()
    out["weights"] = bufs.expert_weights.cpu().numpy()
    if scales:
        out["scales"] = so.cpu().numpy().view(np.uint32)
    return out, bufs


def assert_parity(got, ids_ref, w_ref, idx_ref, E):
    bad = np.nonzero((got["ids"] != ids_ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} token rows differ, first {bad[:1]}"
    assert np.array_equal(got["weights"].view(np.uint32), w_ref.view(np.uint32))
    for k in INDEX_KEYS:
        assert np.array_equal(got[k], idx_ref[k]), k


def check(scores, bias, K, G, M, norm, scale, **kw):
    ids_ref, w_ref = oracle.route(scores, bias, K, G, M, norm, scale)
    idx_ref = oracle.create_indices(ids_ref, scores.shape[1])
    got, bufs = gpu_route_index(scores, bias, K, G, M, norm, scale, **kw)
    assert_parity(got, ids_ref, w_ref, idx_ref, scores.shape[1])
    assert bufs.device_status() == 0
    return got, bufs, ids_ref


BOTH = pytest.mark.parametrize("single", [False, True], ids=["counting", "single_launch"])


@BOTH
@pytest.mark.parametrize("name", [c.name for c in synth.CONFIGS])
def test_parity_on_workloads(name, single):
    cfg, scores, bias, ids_ref, w_ref, idx_ref = workload(name)
    got, bufs = gpu_route_index(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale,
                                single=single)
    assert_parity(got, ids_ref, w_ref, idx_ref, cfg.E)
    assert bufs.device_status() == 0


# (E, G, M, K): thread path (E <= 32), warp path with every group layout
# (all kept, power-of-two lane segments, shared-memory groups), and C = 2 .. 32.
SHAPES = [(8, 1, 1, 2), (8, 4, 2, 3), (12, 3, 2, 4), (16, 4, 2, 4), (32, 4, 2, 8),
          (48, 4, 2, 6), (64, 8, 4, 8), (96, 4, 2, 8), (120, 5, 2, 8), (128, 1, 1, 8),
          (160, 8, 3, 6), (256, 8, 4, 8), (256, 1, 1, 32), (384, 12, 4, 8), (512, 8, 2, 16),
          (1024, 32, 4, 8)]


@BOTH
@pytest.mark.parametrize("E,G,M,K", SHAPES)
@pytest.mark.parametrize("T", [1, 333, 5000])
def test_parity_shapes(E, G, M, K, T, single):
    rng = np.random.default_rng(E * 7919 + G * 31 + M * 7 + K + T)
    scores = rng.random((T, E), dtype=np.float32)
    bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
    check(scores, bias, K, G, M, True, 1.5, single=single)


@BOTH
@pytest.mark.parametrize("T", [0, 1, 7, 8, 9, 128, 129, 255, 257, 4097, 100003])
def test_token_counts_prefill_shape(T, single):
    cfg = synth.get_config("dsv3_prefill")
    scores = synth.make_scores(cfg, n_tokens=T) if T else np.zeros((0, cfg.E), np.float32)
    bias = synth.make_bias(cfg)
    got, _, _ = check(scores, bias, cfg.K, cfg.G, cfg.M, True, 2.5, single=single)
    if T == 0:
        assert (got["expert_ids"] == -1).all() and (got["expert_start_indices"] == 0).all()
        assert got["expert_usage_stats"].tolist() == [0, 0]


@BOTH
@pytest.mark.parametrize("E,G,M,K,T", [(8, 1, 1, 2, 2_000_000), (64, 8, 4, 8, 200_000)])
def test_large_token_counts(E, G, M, K, T, single):
    """Large batches: for the single launch, many more slots per warp than one
    placement round holds; for the counting path, count rows longer than one
    pass of the row-prefix kernel (thread path and warp path)."""
    rng = np.random.default_rng(T)
    scores = rng.random((T, E), dtype=np.float32)
    bias = np.zeros(E, np.float32)
    check(scores, bias, K, G, M, False, 1.0, single=single)


@BOTH
def test_hot_experts_and_ties(single):
    """Scores on a 1/8 grid plus a large bias on four experts: many equal keys
    and a few experts holding most slots."""
    rng = np.random.default_rng(5)
    T, E = 20000, 128
    scores = (rng.integers(0, 9, size=(T, E)) / 8).astype(np.float32)
    bias = np.zeros(E, np.float32)
    bias[[3, 17, 64, 100]] = 2.0
    got, _, _ = check(scores, bias, 8, 8, 4, True, 1.0, single=single)
    assert got["expert_usage_stats"][0] >= T // 2


@BOTH
@pytest.mark.parametrize("name", ["dsv3_decode", "dsv3_prefill", "few_expert_large_batch"])
def test_sigmoid_loader(name, single):
    cfg = synth.get_config(name)
    logits = synth.normal_f32(cfg.seed, synth.TENSOR_SCORES, cfg.T * cfg.E).reshape(cfg.T, cfg.E)
    bias = synth.make_bias(cfg)
    ids_ref, w_ref = oracle.route(oracle.sigmoid(logits), bias, cfg.K, cfg.G, cfg.M,
                                  cfg.norm_weights, cfg.scale)
    idx_ref = oracle.create_indices(ids_ref, cfg.E)
    moe = _moe()
    got, _ = gpu_route_index(logits, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale,
                             score_fn=moe.SCORES_SIGMOID, single=single)
    assert_parity(got, ids_ref, w_ref, idx_ref, cfg.E)


@BOTH
@pytest.mark.parametrize("name", ["tiny", "dsv3_prefill", "skewed_ungrouped"])
def test_scales_offsets(name, single):
    cfg, scores, bias, ids_ref, w_ref, idx_ref = workload(name)
    got, _ = gpu_route_index(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale,
                             scales=True, single=single)
    assert_parity(got, ids_ref, w_ref, idx_ref, cfg.E)
    assert np.array_equal(got["scales"], oracle.scales_offsets(ids_ref, cfg.E))


def test_counts_left_zero_and_calls_repeat():
    """The counting path leaves its whole count matrix zero after each call
    (the prefixes live elsewhere, at the workspace's end), so repeated calls on
    one workspace need no clearing."""
    cfg, scores, bias, ids_ref, w_ref, idx_ref = workload("dsv3_prefill")
    bufs = None
    for _ in range(3):
        got, bufs = gpu_route_index(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights,
                                    cfg.scale, bufs=bufs)
        assert_parity(got, ids_ref, w_ref, idx_ref, cfg.E)
        # header (256 B) | totals (1024 words) | counts [E][row] | ... prefixes at the end
        row = (-(-cfg.T * cfg.K // 1024) + 3) // 4 * 4
        matrix = -(-4 * cfg.E * row // 256) * 256
        counts = bufs.workspace[256 + 4 * 1024:256 + 4 * 1024 + matrix].view(torch.int32)
        assert int(counts.abs().sum().item()) == 0
        assert bufs.device_status() == 0


def test_call_counter_advances_and_calls_repeat():
    """Single launch: header word 1 counts the calls; nothing is cleared
    between calls."""
    cfg, scores, bias, ids_ref, w_ref, idx_ref = workload("dsv3_prefill")
    bufs = None
    for n in range(1, 4):
        got, bufs = gpu_route_index(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights,
                                    cfg.scale, bufs=bufs, single=True)
        assert_parity(got, ids_ref, w_ref, idx_ref, cfg.E)
        header = bufs.workspace[:8].view(torch.int32).cpu().numpy()
        assert header.tolist() == [0, n]


@pytest.mark.parametrize("name", ["dsv3_prefill", "skewed_ungrouped"])
def test_unzeroed_workspace_is_reported(name):
    """A workspace that was not zero-filled (every word 1, so each count of
    this shape is one too high and the totals exceed T*K) sets
    MOE_DEVICE_STATUS_SYNC_STATE; the guard regions around every output and
    the workspace stay intact (no position at or past T*K is written), and
    the call leaves the counts it used zero, so the next call is exact."""
    moe = _moe()
    cfg, scores, bias, ids_ref, w_ref, idx_ref = workload(name)
    bufs = moe.RouteIndexBuffers(cfg.T, cfg.E, cfg.K, "cuda")
    ws, gws = guarded((bufs.workspace.numel(),), torch.uint8, fill=0, name="workspace")
    ws.view(torch.int32).fill_(1)
    bufs.workspace = ws
    bufs._guards = guard_attrs(bufs, ("expert_indices", "expert_weights") + INDEX_KEYS) + [gws]
    got, bufs = gpu_route_index(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale,
                                bufs=bufs)
    # the routing itself does not read the workspace
    assert np.array_equal(got["ids"], ids_ref)
    assert bufs.device_status() & moe.DEVICE_STATUS_SYNC_STATE
    got, bufs = gpu_route_index(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale,
                                bufs=bufs)
    assert_parity(got, ids_ref, w_ref, idx_ref, cfg.E)
    assert bufs.device_status() == 0


@BOTH
def test_workspace_reused_across_shapes(single):
    """One workspace, sized for the largest call, serves calls of other shapes
    in any order: stale tagged words never pass for a later call's (single
    launch), and the count matrix of any layout starts zero (counting)."""
    moe = _moe()
    big = synth.get_config("dsv3_prefill")
    nbytes = (moe.moe_route_index_single_launch_workspace_size(big.T, big.E) if single
              else moe.moe_route_index_workspace_size(big.T, big.E, big.K))
    ws, gws = guarded((nbytes,), torch.uint8, fill=0, name="workspace")
    for name in ("dsv3_prefill", "dsv3_decode", "tiny", "skewed_ungrouped", "dsv3_prefill"):
        cfg, scores, bias, ids_ref, w_ref, idx_ref = workload(name)
        bufs = moe.RouteIndexBuffers(cfg.T, cfg.E, cfg.K, "cuda", single_launch=single)
        bufs.workspace = ws  # the same (guarded) workspace for every call
        bufs._guards = guard_attrs(bufs, ("expert_indices", "expert_weights") + INDEX_KEYS) + [gws]
        got, bufs = gpu_route_index(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights,
                                    cfg.scale, bufs=bufs)
        assert_parity(got, ids_ref, w_ref, idx_ref, cfg.E)
        assert bufs.device_status() == 0


def test_call_counter_wraps_past_zero():
    """After call number 0xFFFFFFFF the next is 2: 0 is never a number (a
    zero-filled word never looks current) and the parity of consecutive
    numbers, which picks the progress-counter slot, keeps alternating. The
    workspace is left as call 0xFFFFFFFF would leave it: its counter slot
    (odd) still holds its final counts, the other slot zeroed."""
    moe = _moe()
    cfg, scores, bias, ids_ref, w_ref, idx_ref = workload("skewed_ungrouped")
    bufs = moe.RouteIndexBuffers(cfg.T, cfg.E, cfg.K, "cuda", single_launch=True)
    words = bufs.workspace.view(torch.int32)
    words[1] = -1                    # the last call's number: 0xFFFFFFFF
    words[(256 + 256) // 4] = 0x7fff  # CTAs-counted slot 1: that call's count
    words[(768 + 256) // 4] = 0x7fff  # rows-scanned slot 1: that call's count
    got, bufs = gpu_route_index(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale,
                                bufs=bufs)
    assert_parity(got, ids_ref, w_ref, idx_ref, cfg.E)
    assert bufs.device_status() == 0
    assert bufs.workspace.view(torch.int32)[1].item() == 2
    # the next call (number 3, odd) uses slot 1, which call 2 zeroed
    got, bufs = gpu_route_index(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale,
                                bufs=bufs)
    assert_parity(got, ids_ref, w_ref, idx_ref, cfg.E)
    assert bufs.workspace.view(torch.int32)[1].item() == 3


def _selftest_lib():
    """The bounded-wait harness of tests/cuda, built with nvcc for sm_103a."""
    import ctypes
    import os
    import subprocess
    from moe_token_routing_gb300 import build
    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(here, "cuda", "tagged_sync_selftest.cu")
    so = os.path.join(here, "cuda", "libtagged_sync_selftest.so")
    hdr = os.path.join(os.path.dirname(os.path.abspath(build.__file__)), "csrc")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.run([build.nvcc()] + build.ARCH_FLAGS + ["-O2", "-std=c++17", "-Xcompiler",
                        "-fPIC", "-shared", "-I", hdr, "-I", os.path.join(build.ROOT, "include"),
                        src, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    vp = ctypes.c_void_p
    lib.tagged_sync_selftest.argtypes = [vp, ctypes.c_uint32, ctypes.c_int, vp, vp]
    lib.tagged_sync_selftest.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("publish", [True, False])
def test_bounded_wait(publish):
    """The wait of the cross-CTA hand-off: with a producer it returns the
    value; with none (a word that nothing tags) it gives up after its one
    second limit and reports failure, and the GPU stays usable."""
    lib = _selftest_lib()
    word = torch.zeros(1, dtype=torch.int64, device="cuda")
    out = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    rc = lib.tagged_sync_selftest(word.data_ptr(), 5, int(publish), out.data_ptr(),
                                  elapsed.data_ptr())
    assert rc == 0
    ok, value = out.cpu().tolist()
    seconds = elapsed.item() * 1e-9
    if publish:
        assert ok == 1 and value == 1234 and seconds < 0.5
    else:
        assert ok == 0 and 0.9 < seconds < 5.0
    # the context is still healthy
    assert torch.ones(4, device="cuda").sum().item() == 4.0


def test_fused_pipeline_matches_separate_launches():
    moe = _moe()
    cfg, scores, bias, *_ = workload("skewed_ungrouped")
    s = torch.from_numpy(scores).cuda()
    b = torch.from_numpy(bias).cuda()
    down = torch.from_numpy(synth.make_down(cfg).view(np.int16)).cuda().view(torch.bfloat16)
    outs = []
    for fused in (False, True):
        pipe = moe.RoutingPipeline(cfg.T, cfg.E, cfg.K, cfg.H, cfg.G, cfg.M, cfg.norm_weights,
                                   cfg.scale, fused=fused)
        out = pipe(s, b, down).clone()
        torch.cuda.synchronize()
        assert pipe.device_status() == 0
        outs.append((out, pipe.index.restore_token_order.clone(), pipe.expert_weights.clone()))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][2].view(torch.int32), outs[1][2].view(torch.int32))


@pytest.mark.parametrize("fn", ["sigmoid", "softmax"])
@pytest.mark.parametrize("E,G,M", [(256, 8, 4), (128, 1, 1)])
def test_loader_tie_stress(fn, E, G, M):
    """Gate logits on a grid of five values (dozens of equal scores per row)
    through the counting router's loaders: the tokens that the tie ranking
    or the exact path settle are counted like the others."""
    rng = np.random.default_rng(E + len(fn))
    T, K = 515, 8
    logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    bias = np.zeros(E, np.float32)
    load = oracle.sigmoid if fn == "sigmoid" else oracle.softmax
    ids_ref, w_ref = oracle.route(load(logits), bias, K, G, M, True, 2.5)
    idx_ref = oracle.create_indices(ids_ref, E)
    moe = _moe()
    code = moe.SCORES_SIGMOID if fn == "sigmoid" else moe.SCORES_SOFTMAX
    got, bufs = gpu_route_index(logits, bias, K, G, M, True, 2.5, score_fn=code)
    assert_parity(got, ids_ref, w_ref, idx_ref, E)
    assert bufs.device_status() == 0


@BOTH
@pytest.mark.parametrize("name", ["dsv3_decode", "skewed_ungrouped", "few_expert_large_batch"])
def test_softmax_loader(name, single):
    cfg = synth.get_config(name)
    logits = synth.normal_f32(cfg.seed, synth.TENSOR_SCORES, cfg.T * cfg.E).reshape(cfg.T, cfg.E)
    bias = synth.make_bias(cfg)
    ids_ref, w_ref = oracle.route(oracle.softmax(logits), bias, cfg.K, cfg.G, cfg.M,
                                  cfg.norm_weights, cfg.scale)
    idx_ref = oracle.create_indices(ids_ref, cfg.E)
    moe = _moe()
    got, _ = gpu_route_index(logits, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale,
                             score_fn=moe.SCORES_SOFTMAX, single=single)
    assert_parity(got, ids_ref, w_ref, idx_ref, cfg.E)
