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
