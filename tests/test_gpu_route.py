"""GPU parity of moe_route (group_limited_router_kernel page) against the oracle.

Expert ids must be bit-exact; weights within 1e-6 relative error (fp32).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _guard import check_all, guarded
from _workloads import workload

pytestmark = pytest.mark.gpu

CONFIG_NAMES = [c.name for c in synth.CONFIGS]


def _moe():
    import moe_token_routing_gb300 as moe
    moe.load_library()
    return moe


def gpu_route(scores, bias, K, G, M, norm, scale, scores_offset=0):
    moe = _moe()
    s = torch.from_numpy(np.ascontiguousarray(scores)).cuda()
    if scores_offset:
        # same values at a pointer that is only 4-byte aligned (scalar-load path)
        buf = torch.empty(s.numel() + scores_offset, dtype=torch.float32, device="cuda")
        buf[scores_offset:] = s.reshape(-1)
        s = buf[scores_offset:].view(s.shape)
    b = torch.from_numpy(np.ascontiguousarray(bias)).cuda()
    T = s.shape[0]
    ids, gi = guarded((T, K), torch.int32, name="expert_indices")
    w, gw = guarded((T, K), torch.float32, name="expert_weights")
    moe.moe_route(ids, w, s, b, G, M, norm, scale)
    check_all([gi, gw])
    return ids.cpu().numpy(), w.cpu().numpy()


def assert_route_parity(scores, bias, K, G, M, norm, scale, **kw):
    ids_ref, w_ref = oracle.route(scores, bias, K, G, M, norm, scale)
    ids, w = gpu_route(scores, bias, K, G, M, norm, scale, **kw)
    bad = np.nonzero((ids != ids_ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first token {bad[:1]}: {ids[bad[:1]]} vs {ids_ref[bad[:1]]}"
    np.testing.assert_allclose(w, w_ref, rtol=1e-6, atol=0)
    return ids, w


@pytest.mark.parametrize("name", CONFIG_NAMES)
def test_parity_on_workloads(name):
    cfg, scores, bias, ids_ref, w_ref, _ = workload(name)
    ids, w = gpu_route(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    assert np.array_equal(ids, ids_ref)
    np.testing.assert_allclose(w, w_ref, rtol=1e-6, atol=0)
    # same arithmetic in the same order: expected bit-identical
    assert np.array_equal(w.view(np.uint32), w_ref.view(np.uint32))


# (E, G, M, K): thread-per-token path (E <= 32) and the warp path's group layouts
SHAPES = [
    (8, 1, 1, 2), (8, 4, 2, 3), (12, 3, 2, 4), (16, 4, 2, 4), (16, 16, 5, 5), (24, 8, 3, 6),
    (32, 4, 2, 8), (32, 32, 7, 7),
    (48, 4, 2, 6), (64, 8, 4, 8), (64, 32, 8, 8), (64, 1, 1, 6), (96, 4, 2, 8),
    (128, 8, 4, 8), (128, 32, 4, 8), (128, 1, 1, 8), (160, 8, 3, 6), (192, 6, 3, 8),
    (256, 8, 4, 8), (256, 16, 4, 8), (256, 32, 8, 16), (256, 2, 1, 8), (256, 4, 1, 8),
    (256, 1, 1, 32), (384, 1, 1, 8), (384, 12, 4, 8), (512, 8, 2, 16), (1024, 32, 4, 8),
]


@pytest.mark.parametrize("E,G,M,K", SHAPES)
@pytest.mark.parametrize("norm", [True, False])
def test_parity_shapes(E, G, M, K, norm):
    rng = np.random.default_rng(E * 7919 + G * 31 + M * 7 + K)
    T = 333
    scores = rng.random((T, E), dtype=np.float32)
    bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
    assert_route_parity(scores, bias, K, G, M, norm, 1.5)


@pytest.mark.parametrize("E,G,M,K", [(16, 4, 2, 4), (128, 8, 4, 8), (256, 8, 4, 8),
                                     (160, 8, 3, 6), (64, 32, 8, 8)])
def test_tie_stress(E, G, M, K):
    """Scores on a 1/8 grid: many equal biased scores, group scores and ranks."""
    rng = np.random.default_rng(E + K)
    T = 512
    scores = (rng.integers(0, 9, size=(T, E)) / 8).astype(np.float32)
    for bias in (np.zeros(E, np.float32), np.full(E, 0.125, np.float32),
                 (rng.integers(-1, 2, size=E) / 8).astype(np.float32)):
        assert_route_parity(scores, bias, K, G, M, True, 1.0)


def test_all_equal_and_signed_zero():
    E, G, M, K = 256, 8, 4, 8
    scores = np.zeros((64, E), dtype=np.float32)
    scores[1::2] = -0.0
    bias = np.zeros(E, np.float32)
    bias[::3] = -0.0
    ids, _ = assert_route_parity(scores, bias, K, G, M, False, 1.0)
    assert (ids == np.arange(K)).all()


@pytest.mark.parametrize("E", [16, 256])
def test_unaligned_scores_use_scalar_loads(E):
    rng = np.random.default_rng(11)
    scores = rng.random((77, E), dtype=np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    G = 4 if E == 16 else 8
    assert_route_parity(scores, bias, 4, G, 2, True, 2.0, scores_offset=1)


@pytest.mark.parametrize("T", [1, 7, 8, 9, 255, 257, 4097, 100000])
def test_token_counts(T):
    E, G, M, K = 256, 8, 4, 8
    cfg = synth.get_config("dsv3_prefill")
    scores = synth.make_scores(cfg, n_tokens=T)
    bias = synth.make_bias(cfg)
    assert_route_parity(scores, bias, K, G, M, True, 2.5)


def test_zero_tokens_is_noop():
    moe = _moe()
    ids = torch.full((0, 8), -7, dtype=torch.int32, device="cuda")
    w = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    s = torch.empty((0, 256), dtype=torch.float32, device="cuda")
    b = torch.zeros(256, dtype=torch.float32, device="cuda")
    moe.moe_route(ids, w, s, b, 8, 4, True, 1.0)
    torch.cuda.synchronize()


@pytest.mark.parametrize("E,G,M,K,status", [(256, 7, 4, 8, 2), (256, 8, 9, 8, 2),
                                            (256, 8, 1, 33, 2), (256, 8, 4, 0, 2),
                                            (2048, 8, 4, 8, 4), (256, 8, 4, 33, 4),
                                            (32, 32, 1, 2, 2)])
def test_invalid_arguments(E, G, M, K, status):
    moe = _moe()
    T = 4
    s = torch.rand((T, E), device="cuda")
    b = torch.zeros(E, device="cuda")
    ids = torch.empty((T, max(K, 1)), dtype=torch.int32, device="cuda")
    w = torch.empty((T, max(K, 1)), dtype=torch.float32, device="cuda")
    lib = moe.load_library()
    rc = lib.moe_route(ids.data_ptr(), w.data_ptr(), s.data_ptr(), b.data_ptr(), T, E, K, G, M, 1,
                       1.0, torch.cuda.current_stream().cuda_stream)
    assert rc == status


def test_deterministic():
    cfg, scores, bias, *_ = workload("dsv3_prefill")
    a = gpu_route(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    b = gpu_route(scores, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))


# Segment layout (E = 32 * L, K <= 8, groups of whole lanes): list lengths K < 8,
# groups spanning several lanes, one group per lane, all groups kept, L = 2 .. 32.
# The shapes here with every group kept and E = 128 or 256 run on the
# staged layout instead (units of 32 experts), and so do the near-equal, tie
# and one-lane cases below for those shapes: both layouts are held to the
# same exact result.
SEG_SHAPES = [
    (64, 1, 1, 8), (64, 2, 1, 4), (128, 1, 1, 1), (128, 4, 2, 8), (128, 2, 2, 7),
    (256, 8, 4, 1), (256, 8, 4, 2), (256, 8, 4, 5), (256, 8, 4, 7), (256, 8, 8, 8),
    (256, 8, 1, 8), (256, 8, 2, 3), (512, 16, 4, 8), (512, 8, 3, 6), (512, 1, 1, 8),
    (1024, 32, 4, 8), (1024, 4, 2, 8), (1024, 1, 1, 3),
]


@pytest.mark.parametrize("E,G,M,K", SEG_SHAPES)
@pytest.mark.parametrize("norm", [True, False])
def test_segment_layout_shapes(E, G, M, K, norm):
    rng = np.random.default_rng(E * 131 + G * 17 + M * 5 + K)
    T = 1003  # not a multiple of the tokens per warp or per CTA
    scores = rng.random((T, E), dtype=np.float32)
    bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
    assert_route_parity(scores, bias, K, G, M, norm, 2.5)


@pytest.mark.parametrize("E,G,M", [(256, 8, 4), (256, 8, 1), (128, 1, 1), (512, 16, 2)])
def test_segment_one_lane_takes_all(E, G, M):
    """Every pick comes from one lane's 32 experts, so the (K+1)-th key is
    that lane's ninth best, found by rescanning its scores."""
    rng = np.random.default_rng(E + G + M)
    T, K = 700, 8
    scores = rng.random((T, E), dtype=np.float32)
    bias = np.zeros(E, np.float32)
    bias[40:48] = 1.0          # inside expert block 1 (experts 32 .. 63)
    bias[40:48] += rng.random(8, dtype=np.float32) * 0.01
    ids, _ = assert_route_parity(scores, bias, K, G, M, True, 1.0)
    assert ((ids >= 40) & (ids < 48)).all()


@pytest.mark.parametrize("E,G,M,K", [(256, 8, 4, 8), (128, 1, 1, 8), (512, 16, 4, 6),
                                     (1024, 32, 8, 8)])
def test_segment_near_equal_scores(E, G, M, K):
    """Clusters of scores a few ULPs apart, in an order that disagrees with
    the expert order: the selection keys agree above their index bits, so the
    tokens take the exact fallback; ids and weights must still be exact."""
    rng = np.random.default_rng(E * 3 + K)
    T = 640
    scores = (rng.random((T, E), dtype=np.float32) * 0.8).astype(np.float32)
    for t in range(T):
        members = rng.choice(E, size=12, replace=False)
        base = np.float32(0.85 + 0.1 * rng.random())
        steps = rng.permutation(12) * int(rng.integers(1, 20))
        vals = base.view(np.uint32) + steps.astype(np.uint32)
        scores[t, members] = vals.view(np.float32)
    bias = np.zeros(E, np.float32)
    assert_route_parity(scores, bias, K, G, M, True, 1.0)
    bias = (rng.integers(-2, 3, size=E) * np.float32(2.0 ** -22)).astype(np.float32)
    assert_route_parity(scores, bias, K, G, M, False, 1.0)


@pytest.mark.parametrize("E,G,M,K", [(128, 1, 1, 8), (256, 8, 4, 8), (512, 16, 4, 8),
                                     (1024, 32, 4, 8)])
def test_segment_tie_stress(E, G, M, K):
    """Scores on a 1/8 grid: nearly every token falls back to the exact path."""
    rng = np.random.default_rng(E + 5 * K)
    T = 300
    scores = (rng.integers(0, 9, size=(T, E)) / 8).astype(np.float32)
    for bias in (np.zeros(E, np.float32), (rng.integers(-1, 2, size=E) / 8).astype(np.float32)):
        assert_route_parity(scores, bias, K, G, M, True, 1.0)


def gpu_route_sigmoid(logits, bias, K, G, M, norm, scale):
    import moe_token_routing_gb300 as moe
    s = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    b = torch.from_numpy(np.ascontiguousarray(bias)).cuda()
    T = logits.shape[0]
    ids, gi = guarded((T, K), torch.int32, name="expert_indices")
    w, gw = guarded((T, K), torch.float32, name="expert_weights")
    moe.moe_route_ex(ids, w, s, b, G, M, norm, scale, moe.SCORES_SIGMOID)
    check_all([gi, gw])
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("name", CONFIG_NAMES)
def test_sigmoid_loader_on_workloads(name):
    """Parameters scores_input_fn: routing gate logits with the fused sigmoid
    equals routing the oracle's sigmoid of the same logits, bit for bit."""
    cfg = synth.get_config(name)
    logits = synth.normal_f32(cfg.seed, synth.TENSOR_SCORES, cfg.T * cfg.E).reshape(cfg.T, cfg.E)
    bias = synth.make_bias(cfg)
    ids_ref, w_ref = oracle.route(oracle.sigmoid(logits), bias, cfg.K, cfg.G, cfg.M,
                                  cfg.norm_weights, cfg.scale)
    ids, w = gpu_route_sigmoid(logits, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    assert np.array_equal(ids, ids_ref)
    assert np.array_equal(w.view(np.uint32), w_ref.view(np.uint32))


@pytest.mark.parametrize("E,G,M,K", [(8, 4, 2, 3), (16, 4, 2, 4), (96, 4, 2, 8), (256, 8, 4, 8),
                                     (384, 1, 1, 8), (128, 1, 1, 8), (512, 16, 4, 8),
                                     (1024, 32, 4, 5)])
def test_sigmoid_loader_shapes_and_extremes(E, G, M, K):
    rng = np.random.default_rng(E + K)
    logits = (rng.standard_normal((300, E)) * 6).astype(np.float32)
    logits[::7, ::3] = 120.0
    logits[1::7, ::5] = -120.0
    bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
    ids_ref, w_ref = oracle.route(oracle.sigmoid(logits), bias, K, G, M, True, 2.5)
    ids, w = gpu_route_sigmoid(logits, bias, K, G, M, True, 2.5)
    assert np.array_equal(ids, ids_ref)
    assert np.array_equal(w.view(np.uint32), w_ref.view(np.uint32))


def gpu_route_softmax(logits, bias, K, G, M, norm, scale):
    import moe_token_routing_gb300 as moe
    s = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    b = torch.from_numpy(np.ascontiguousarray(bias)).cuda()
    T = logits.shape[0]
    ids, gi = guarded((T, K), torch.int32, name="expert_indices")
    w, gw = guarded((T, K), torch.float32, name="expert_weights")
    moe.moe_route_ex(ids, w, s, b, G, M, norm, scale, moe.SCORES_SOFTMAX)
    check_all([gi, gw])
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("name", CONFIG_NAMES)
def test_softmax_loader_on_workloads(name):
    """Parameters scores_input_fn: routing gate logits with the fused softmax
    equals routing the oracle's softmax of the same logits, bit for bit (the
    sum over experts in ascending order on both sides)."""
    cfg = synth.get_config(name)
    logits = synth.normal_f32(cfg.seed, synth.TENSOR_SCORES, cfg.T * cfg.E).reshape(cfg.T, cfg.E)
    bias = synth.make_bias(cfg)
    ids_ref, w_ref = oracle.route(oracle.softmax(logits), bias, cfg.K, cfg.G, cfg.M,
                                  cfg.norm_weights, cfg.scale)
    ids, w = gpu_route_softmax(logits, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    assert np.array_equal(ids, ids_ref)
    assert np.array_equal(w.view(np.uint32), w_ref.view(np.uint32))


@pytest.mark.parametrize("E,G,M,K", [(8, 4, 2, 3), (12, 3, 2, 4), (32, 4, 2, 8), (48, 4, 2, 6),
                                     (96, 4, 2, 8), (120, 5, 2, 8), (256, 8, 4, 8),
                                     (384, 1, 1, 8), (1024, 32, 4, 8),
                                     # segment layout: L = 2, 4, 8, 16 lanes per token, K < 8;
                                     # (256, 8, 4, 8) and (128, 1, 1, 8) take the staged one
                                     (64, 2, 1, 4), (128, 1, 1, 8), (256, 8, 4, 3),
                                     (512, 16, 4, 8)])
@pytest.mark.parametrize("norm", [True, False])
def test_softmax_loader_shapes_and_extremes(E, G, M, K, norm):
    rng = np.random.default_rng(E + K + norm)
    logits = (rng.standard_normal((300, E)) * 4).astype(np.float32)
    logits[::7, ::3] = 90.0      # very large logits (exp needs the max shift)
    logits[1::7, :] = -5.0       # all-equal rows
    logits[2::7, ::5] = -150.0   # exp underflow clamp
    bias = (rng.standard_normal(E) * 0.01).astype(np.float32)
    ids_ref, w_ref = oracle.route(oracle.softmax(logits), bias, K, G, M, norm, 2.5)
    ids, w = gpu_route_softmax(logits, bias, K, G, M, norm, 2.5)
    assert np.array_equal(ids, ids_ref)
    assert np.array_equal(w.view(np.uint32), w_ref.view(np.uint32))


@pytest.mark.parametrize("fn", ["sigmoid", "softmax"])
@pytest.mark.parametrize("E,G,M,K", [(128, 4, 2, 8), (256, 8, 4, 8), (512, 16, 4, 8),
                                     (128, 1, 1, 8), (256, 1, 1, 8), (256, 8, 4, 6)])
def test_loader_tie_stress(fn, E, G, M, K):
    """Gate logits on a grid of five values, so that dozens of a row's loaded
    scores are equal: ties in the biased scores, the group scores and the
    group ranks. The staged layout (groups or units of 32 experts; softmax
    with K = 8 and at most 256 experts) ranks them by exact keys or hands
    the token to the exact path, which for softmax rebuilds the row; the
    result must still be the oracle's, bit for bit."""
    rng = np.random.default_rng(E + 10 * K + len(fn))
    T = 515
    logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    load = oracle.sigmoid if fn == "sigmoid" else oracle.softmax
    run = gpu_route_sigmoid if fn == "sigmoid" else gpu_route_softmax
    for bias in (np.zeros(E, np.float32), (rng.integers(-1, 2, size=E) / 8).astype(np.float32)):
        ids_ref, w_ref = oracle.route(load(logits), bias, K, G, M, True, 2.5)
        ids, w = run(logits, bias, K, G, M, True, 2.5)
        bad = np.nonzero((ids != ids_ref).any(axis=1))[0]
        assert bad.size == 0, f"{bad.size} rows differ, first token {bad[:1]}"
        assert np.array_equal(w.view(np.uint32), w_ref.view(np.uint32))


def _mbar_selftest_lib():
    """The bounded-wait harness of tests/cuda (the staged router's chunk wait),
    built with nvcc for sm_103a."""
    import ctypes
    import os
    import subprocess
    from moe_token_routing_gb300 import build
    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(here, "cuda", "mbar_wait_selftest.cu")
    so = os.path.join(here, "cuda", "libmbar_wait_selftest.so")
    hdr = os.path.join(os.path.dirname(os.path.abspath(build.__file__)), "csrc")
    deps = [src, os.path.join(hdr, "mbarrier.cuh"), os.path.join(hdr, "tagged_sync.cuh")]
    if not os.path.exists(so) or any(os.path.getmtime(so) < os.path.getmtime(d) for d in deps):
        subprocess.run([build.nvcc()] + build.ARCH_FLAGS + ["-O2", "-std=c++17", "-Xcompiler",
                        "-fPIC", "-shared", "-I", hdr, "-I", os.path.join(build.ROOT, "include"),
                        src, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    vp = ctypes.c_void_p
    lib.mbar_wait_selftest.argtypes = [vp, ctypes.c_int, vp, vp]
    lib.mbar_wait_selftest.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("complete", [True, False])
def test_bounded_chunk_wait(complete):
    """The staged router's wait for a score chunk: when the bulk copy lands the
    wait returns at once with the data; when nothing arrives (a barrier no copy
    completes) it gives up after its one-second limit and reports failure, and
    the GPU stays usable. A router warp that gives up writes id -1 for its
    tokens, which moe_route_index reports as a bad expert id."""
    lib = _mbar_selftest_lib()
    src = torch.tensor([0x1234, 5, 6, 7], dtype=torch.int32, device="cuda")
    out = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    rc = lib.mbar_wait_selftest(src.data_ptr(), int(complete), out.data_ptr(), elapsed.data_ptr())
    assert rc == 0
    ok, first = out.cpu().tolist()
    seconds = elapsed.item() * 1e-9
    if complete:
        assert ok == 1 and first == 0x1234 and seconds < 0.5
    else:
        assert ok == 0 and 0.9 < seconds < 5.0
    assert torch.ones(4, device="cuda").sum().item() == 4.0
