"""The chained route -> create_indices -> finalize path (device buffers and the
end-to-end host-buffer call) against the chained oracle."""
import numpy as np
import pytest
import torch

import synth
from _workloads import (bits_to_f32, f32_to_bf16_bits, finalize_tolerance_ok, workload,
                        workload_down, workload_finalize_ref)

pytestmark = pytest.mark.gpu


def _pipe(cfg, fused=True):
    import moe_token_routing_gb300 as moe
    return moe.RoutingPipeline(cfg.T, cfg.E, cfg.K, cfg.H, cfg.G, cfg.M, cfg.norm_weights,
                               cfg.scale, device="cuda", fused=fused)


@pytest.mark.parametrize("fused", [True, False], ids=["route_index", "separate"])
@pytest.mark.parametrize("name", [c.name for c in synth.CONFIGS])
def test_chain_matches_oracle_chain(name, fused):
    cfg, scores, bias, ids, w, idx = workload(name)
    down = workload_down(name)
    pipe = _pipe(cfg, fused)
    d = torch.from_numpy(down.view(np.int16)).cuda().view(torch.bfloat16)
    out = pipe(torch.from_numpy(scores).cuda(), torch.from_numpy(bias).cuda(), d)
    torch.cuda.synchronize()
    assert np.array_equal(pipe.expert_indices.cpu().numpy(), ids)
    np.testing.assert_allclose(pipe.expert_weights.cpu().numpy(), w, rtol=1e-6, atol=0)
    for k in ("token_expert_order", "restore_token_order", "expert_start_indices"):
        assert np.array_equal(getattr(pipe.index, k).cpu().numpy().view(np.uint32), idx[k]), k
    assert np.array_equal(pipe.index.expert_ids.cpu().numpy(), idx["expert_ids"])
    ref = workload_finalize_ref(name)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert finalize_tolerance_ok(got, ref).all()
    assert np.array_equal(got, f32_to_bf16_bits(ref))
    assert pipe.device_status() == 0


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "skewed_ungrouped"])
def test_host_buffer_call(name):
    """run_host: pinned host inputs -> device -> three kernels -> host output."""
    cfg, scores, bias, *_ = workload(name)
    down = workload_down(name)
    pipe = _pipe(cfg)
    s_h = torch.from_numpy(scores).pin_memory()
    b_h = torch.from_numpy(bias).pin_memory()
    d_h = torch.from_numpy(down.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_h = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    for _ in range(2):
        out_h.zero_()
        pipe.run_host(s_h, b_h, d_h, out_h)
        torch.cuda.synchronize()
        ref = workload_finalize_ref(name)
        got = out_h.view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, f32_to_bf16_bits(ref))


def test_host_streamer_overlapped_batches():
    """HostStreamer: several batches with different inputs, copies overlapped
    across batches; every output equals the synchronous host-buffer call's."""
    import synth
    cfg0 = synth.get_config("dsv3_decode")
    pipe = _pipe(cfg0)
    batches = []
    for seed in (3, 4, 5, 6, 7):
        c = cfg0.replace(seed=seed)
        s_h = torch.from_numpy(synth.make_scores(c)).pin_memory()
        b_h = torch.from_numpy(synth.make_bias(c)).pin_memory()
        d_h = torch.from_numpy(synth.make_down(c).view(np.int16)).view(torch.bfloat16).pin_memory()
        batches.append((s_h, b_h, d_h))
    expected = []
    for s_h, b_h, d_h in batches:
        out_h = torch.empty((c.T, c.H), dtype=torch.bfloat16).pin_memory()
        pipe.run_host(s_h, b_h, d_h, out_h)
        torch.cuda.synchronize()
        expected.append(out_h.clone())
    streamer = pipe.stream_from_host(depth=2)
    outs = [torch.zeros((c.T, c.H), dtype=torch.bfloat16).pin_memory() for _ in batches]
    for (s_h, b_h, d_h), out_h in zip(batches, outs):
        streamer.submit(s_h, b_h, d_h, out_h)
    streamer.synchronize()
    for got, exp in zip(outs, expected):
        assert torch.equal(got.view(torch.int16), exp.view(torch.int16))
    assert not torch.equal(expected[0].view(torch.int16), expected[1].view(torch.int16))


@pytest.mark.parametrize("fused", [True, False], ids=["route_index", "separate"])
@pytest.mark.parametrize("name", ["dsv3_decode", "skewed_ungrouped"])
def test_cuda_graph_replay(name, fused):
    """One step captured in a CUDA graph: replaying it three times on the same
    inputs gives the oracle's outputs every time (the index workspace carries
    nothing from one replay into the next), and after new inputs are copied
    into the captured buffers a replay gives the oracle's outputs for those."""
    cfg, scores, bias, ids, w, idx = workload(name)
    down = workload_down(name)
    pipe = _pipe(cfg, fused)
    s_d = torch.from_numpy(scores).cuda()
    b_d = torch.from_numpy(bias).cuda()
    d_d = torch.from_numpy(down.view(np.int16)).cuda().view(torch.bfloat16)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        pipe(s_d, b_d, d_d, stream=st)  # first calls outside the capture (module load)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        pipe(s_d, b_d, d_d, stream=st)

    def check(ids_ref, w_ref, idx_ref, fin_ref):
        torch.cuda.synchronize()
        assert np.array_equal(pipe.expert_indices.cpu().numpy(), ids_ref)
        assert np.array_equal(pipe.expert_weights.cpu().numpy().view(np.uint32),
                              w_ref.view(np.uint32))
        for k in ("token_expert_order", "restore_token_order", "expert_start_indices"):
            assert np.array_equal(getattr(pipe.index, k).cpu().numpy().view(np.uint32),
                                  idx_ref[k]), k
        got = pipe.output.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, f32_to_bf16_bits(fin_ref))
        assert pipe.device_status() == 0

    for _ in range(3):
        pipe.output.zero_()
        pipe.index.token_expert_order.fill_(-1)
        graph.replay()
        check(ids, w, idx, workload_finalize_ref(name))
    # another seed's inputs, copied into the captured buffers
    import oracle
    c2 = cfg.replace(seed=cfg.seed + 1)
    scores2, bias2, down2 = synth.make_scores(c2), synth.make_bias(c2), synth.make_down(c2)
    ids2, w2 = oracle.route(scores2, bias2, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    idx2 = oracle.create_indices(ids2, cfg.E)
    fin2 = oracle.finalize(down2, idx2["restore_token_order"], w2, cfg.T, cfg.K, cfg.H)
    s_d.copy_(torch.from_numpy(scores2))
    b_d.copy_(torch.from_numpy(bias2))
    d_d.view(torch.int16).copy_(torch.from_numpy(down2.view(np.int16)))
    graph.replay()
    check(ids2, w2, idx2, fin2)


@pytest.mark.parametrize("fused", [True, False], ids=["route_index", "separate"])
def test_concurrent_pipelines_on_two_streams(fused):
    """Two pipelines (their own buffers and workspaces) enqueued in alternation
    on two streams, four batches each, so that their kernels can run at the
    same time: the library keeps no shared device state on these paths, and
    every batch matches the oracle chain."""
    names = ("dsv3_decode", "skewed_ungrouped")
    runs = []
    for name in names:
        cfg, scores, bias, *_ = workload(name)
        down = workload_down(name)
        runs.append(dict(
            name=name, pipe=_pipe(cfg, fused), stream=torch.cuda.Stream(),
            s=torch.from_numpy(scores).cuda(), b=torch.from_numpy(bias).cuda(),
            d=torch.from_numpy(down.view(np.int16)).cuda().view(torch.bfloat16),
            outs=[torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
                  for _ in range(4)]))
    torch.cuda.synchronize()
    for i in range(4):
        for r in runs:
            r["stream"].wait_stream(torch.cuda.current_stream())
            r["pipe"].route_and_index(r["s"], r["b"], r["stream"])
            r["pipe"].finalize(r["d"], r["stream"], output=r["outs"][i])
    torch.cuda.synchronize()
    for r in runs:
        want = f32_to_bf16_bits(workload_finalize_ref(r["name"]))
        for out in r["outs"]:
            assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), want), \
                r["name"]
        assert r["pipe"].device_status() == 0
