"""Benchmark of the MoE routing hot path: route -> create_indices -> finalize.

One step = the three stages over one batch of seeded synthetic input
(default: the DeepSeek-V3-shaped prefill workload, T=16384 tokens, E=256
experts in 8 groups, top-4 groups, K=8, H=7168), inputs resident in HBM,
L2 flushed before every step outside the timed events: a 256 MB write evicts
everything, then a 256 MB read writes back the dirty lines the write left and
leaves L2 holding only clean data that no step uses.

Prints ONE JSON line. `value` is whole-job tokens/s from CUDA-event device
time per step; `e2e` is the same metric through the host-buffer call
(pinned host inputs copied in, output copied back, every step); `roofline`
is the finalize kernel's algorithmic bytes / its event-timed duration
against the measured HBM copy bandwidth; `cpu_baseline` is the CPU oracle
on the host cores. `--impl reference` times only the CPU oracle.

Multi-GPU (torchrun): every rank runs its own batch (weak scaling), with no
collective on the data path; the barrier and max-over-ranks only bracket
the timing.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "route+index+finalize tokens/s; finalize & router HBM GB/s vs ~8 TB/s peak"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--config", default="dsv3_prefill")
    p.add_argument("--tokens", type=int, default=None,
                   help="override the workload's token count (profiling runs)")
    p.add_argument("--e2e-steps", type=int, default=100)
    p.add_argument("--separate-index", action="store_true",
                   help="time moe_route followed by moe_create_indices in the steps "
                        "instead of the fused moe_route_index")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the router back-to-back / large-batch measurements, the "
                        "secondary workloads and the host-link windows (profiling runs)")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--router-only", action="store_true",
                   help="launch only the router (moe_route) on the workload's scores, "
                        "--warmup untimed then --steps timed launches back to back, and "
                        "print their time (profiling runs of the router at other sizes)")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def index_launches(num_slots: int, n_experts: int) -> int:
    """Kernels one moe_create_indices call launches: one CTA does everything for
    N <= 1024 slots; otherwise count, row prefixes and scatter."""
    return 1 if num_slots <= 1024 else 3


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (the timing reduction; not on the data path)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, worst_ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own batch in each step."""
    return tokens_per_rank * world / (worst_ms_per_step * 1e-3)


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            v = float(json.load(fh)["hbm_gbs"])
            return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(cfg):
    N = cfg.T * cfg.K
    return {
        "route": 4 * cfg.T * cfg.E + 4 * cfg.E + 8 * cfg.T * cfg.K,
        "index": 4 * N + 8 * N + 4 * (cfg.E + 1) + 4 * cfg.E + 8,
        "finalize": 2 * N * cfg.H + 4 * N + 4 * N + 2 * cfg.T * cfg.H,
    }


def profile_traffic(kernel_file: str, summary_name: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (the summary records the source's hash)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", summary_name)
    src = os.path.join(ROOT, "moe_token_routing_gb300", "csrc", kernel_file)
    try:
        fields = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if fields.get("source_sha256_16") != digest:
            return None
        return int(fields["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.uuid and self.uuid not in parts[0] and parts[0] not in self.uuid:
                    continue
                rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def device_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------- CPU oracle
def host_threads() -> int:
    """Host threads this process may run on (std::thread::hardware_concurrency
    counts the same logical CPUs unless an affinity mask narrows them)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model string (``model name`` in /proc/cpuinfo; on Arm
    hosts, which do not list one there, lscpu's ``Model name``)."""
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def _ranges(n: int, parts: int):
    return [(n * i // parts, n * (i + 1) // parts) for i in range(parts) if n * i // parts < n * (i + 1) // parts]


def oracle_chain_seconds(cfg, scores, bias, down, t0: int, n_tok: int, pool=None,
                         threads: int = 1) -> float:
    """Oracle route -> index -> finalize over tokens [t0, t0+n_tok); returns seconds.

    With a thread pool, route and finalize run on `threads` contiguous token
    ranges at once (each range is an independent oracle call; the oracle
    releases the interpreter lock while it runs); the index build stays one
    sequential call, since its stability comes from one ordered walk."""
    import numpy as np

    import oracle
    s = scores[t0:t0 + n_tok]
    N = n_tok * cfg.K
    start = time.perf_counter()
    if pool is None or threads <= 1:
        ids, w = oracle.route(s, bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
        idx = oracle.create_indices(ids, cfg.E)
        oracle.finalize(down[:N], idx["restore_token_order"], w, n_tok, cfg.K, cfg.H)
        return time.perf_counter() - start
    parts = _ranges(n_tok, threads)
    routed = [pool.submit(oracle.route, s[a:b], bias, cfg.K, cfg.G, cfg.M, cfg.norm_weights,
                          cfg.scale) for a, b in parts]
    res = [f.result() for f in routed]
    ids = np.concatenate([r[0] for r in res])
    w = np.concatenate([r[1] for r in res])
    idx = oracle.create_indices(ids, cfg.E)
    restore = idx["restore_token_order"]
    fin = [pool.submit(oracle.finalize, down[:N], restore, w, n_tok, cfg.K, cfg.H,
                       np.arange(a, b, dtype=np.int64)) for a, b in parts]
    for f in fin:
        f.result()
    return time.perf_counter() - start


def _timed_sample(cfg, scores, bias, down, target_s, pool, threads):
    probe_tok = min(cfg.T, max(256, 64 * threads))
    probe = oracle_chain_seconds(cfg, scores, bias, down, 0, probe_tok, pool, threads)
    per_tok = max(probe / probe_tok, 1e-9)
    n_tok = int(min(cfg.T, max(1, target_s / 2 / per_tok)))
    oracle_chain_seconds(cfg, scores, bias, down, 0, n_tok, pool, threads)  # warm-up pass
    reps, total, done = 0, 0.0, 0
    while total < target_s and reps < 64:
        total += oracle_chain_seconds(cfg, scores, bias, down, 0, n_tok, pool, threads)
        done += n_tok
        reps += 1
    return done / total, n_tok, reps, total


def cpu_baseline(cfg, scores, bias, down, target_s: float):
    """The oracle as it stands on a bounded sample of the workload: single
    thread, and over every host thread (token ranges for route and finalize,
    the index build sequential). `value` and `cores` are the all-threads run."""
    from concurrent.futures import ThreadPoolExecutor
    threads = host_threads()
    v1, n1, r1, s1 = _timed_sample(cfg, scores, bias, down, target_s / 2, None, 1)
    with ThreadPoolExecutor(threads) as pool:
        vn, nn, rn, sn = _timed_sample(cfg, scores, bias, down, target_s / 2, pool, threads)
    return {"value": vn, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{cfg.name}: tokens 0..{nn - 1} of {cfg.T}, route+index+finalize, "
                      f"{rn} pass(es), {sn:.1f} s on {threads} threads (route and finalize "
                      f"split by token range, index build sequential)",
            "single_thread": {"value": v1, "unit": "tokens/s", "cores": 1,
                              "sample": f"tokens 0..{n1 - 1}, {r1} pass(es), {s1:.1f} s"},
            "hardware_concurrency": os.cpu_count(), "cpu_model": cpu_model()}


def host_inputs(cfg, seed_offset=0, pinned=False):
    import numpy as np
    import torch

    import synth
    c = cfg.replace(seed=cfg.seed + seed_offset)
    scores = synth.make_scores(c)
    bias = synth.make_bias(c)
    down_t = torch.empty((c.N, c.H), dtype=torch.bfloat16, pin_memory=pinned)
    synth.make_down(c, out_ptr=down_t.data_ptr())
    down_np = down_t.view(torch.int16).numpy().view(np.uint16)
    return scores, bias, down_t, down_np


# ---------------------------------------------------------------- reference arm
def run_reference(args, cfg, rank, world):
    if rank != 0:
        return
    from concurrent.futures import ThreadPoolExecutor
    scores, bias, _, down = host_inputs(cfg)
    threads = host_threads()
    with ThreadPoolExecutor(threads) as pool:
        probe_tok = min(cfg.T, max(256, 64 * threads))
        per_tok = oracle_chain_seconds(cfg, scores, bias, down, 0, probe_tok, pool,
                                       threads) / probe_tok
        budget = 150.0  # seconds for warmup + timed steps
        n_tok = int(max(1, min(cfg.T, budget / max(1, args.steps + args.warmup)
                               / max(per_tok, 1e-9))))
        t0 = 0
        for _ in range(args.warmup):
            oracle_chain_seconds(cfg, scores, bias, down, t0, n_tok, pool, threads)
            t0 = (t0 + n_tok) % max(1, cfg.T - n_tok + 1)
        total = 0.0
        for _ in range(args.steps):
            total += oracle_chain_seconds(cfg, scores, bias, down, t0, n_tok, pool, threads)
            t0 = (t0 + n_tok) % max(1, cfg.T - n_tok + 1)
    value = n_tok * args.steps / total
    sample = (f"{cfg.name}: {n_tok} of {cfg.T} tokens per step, route+index+finalize on "
              f"{threads} threads (route and finalize split by token range, index build "
              f"sequential)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)",
        "config": config_dict(cfg),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample, "hardware_concurrency": os.cpu_count(),
                         "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(cfg):
    return {"workload": cfg.name, "tokens": cfg.T, "n_routed_experts": cfg.E,
            "n_groups": cfg.G, "topk_group": cfg.M, "n_experts_per_tok": cfg.K,
            "hidden": cfg.H, "norm_weights": cfg.norm_weights,
            "routed_scaling_factor": cfg.scale, "scores": cfg.scores, "bias": cfg.bias,
            "down_dtype": "bf16", "weights_dtype": "f32", "output_dtype": "bf16",
            "l2": "flushed before every step outside the timed events: 256 MB write, then "
                  "256 MB read (so no dirty flush lines are written back inside the step)"}



# ---------------------------------------------------------------- extra measurements
def router_bytes(T: int, E: int, K: int) -> int:
    return 4 * T * E + 4 * E + 8 * T * K


def time_back_to_back(fn, n: int, stream, host=None) -> float:
    """Mean device time (us) of n calls of fn(i) launched back to back
    between one pair of events; `host` (a dict) receives the host time per
    call spent enqueueing them."""
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    h0 = time.perf_counter()
    for i in range(n):
        fn(i)
    h1 = time.perf_counter()
    e1.record(stream)
    torch.cuda.synchronize()
    if host is not None:
        host["host_enqueue_us_per_launch"] = (h1 - h0) * 1e6 / n
    return e0.elapsed_time(e1) * 1e3 / n


def time_graph_replay(fn, n: int, dev, reps: int = 10):
    """Mean device time (us) per call when n calls of fn(i, stream), captured
    in a CUDA graph, are replayed `reps` times back to back: no host work per
    launch. None if the capture fails."""
    import torch
    s = torch.cuda.Stream(dev)
    try:
        with torch.cuda.stream(s):
            for i in range(n):
                fn(i, s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for i in range(n):
                fn(i, s)
    except Exception:
        torch.cuda.synchronize()
        return None
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * n)


def router_roofline(single_gbs, single_ms, peak, nbytes, evidence):
    """The router's roofline entry. Its headline is the per-launch time of 48
    launches back to back between one event pair (inputs rotating over more
    than twice the L2), the steady state of a stream of batches; one launch
    between two events after an L2 flush carries the event-to-kernel latency
    too and is reported beside it. Without the back-to-back evidence (a
    --no-extras run) the single launch is the headline."""
    single = {"us_per_launch": single_ms * 1e3, "achieved_gbs": single_gbs,
              "frac": single_gbs / peak,
              "timing": "one launch between two events after an L2 flush, mean of the stage pass"}
    out = {"bound": "hbm", "peak": peak, "unit": "GB/s", "algorithmic_bytes_per_launch": nbytes}
    if evidence and evidence.get("back_to_back"):
        b2b = evidence["back_to_back"]
        gbs = b2b["achieved_gbs"]
        out.update({"achieved": gbs, "frac": gbs / peak,
                    "frac_vs_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
                    "timing": "48 launches back to back from the host between one event pair, "
                              "inputs rotating over more than twice the L2"})
    else:
        out.update({"achieved": single_gbs, "frac": single_gbs / peak,
                    "frac_vs_nominal_8tbs": single_gbs / NOMINAL_HBM_GBS,
                    "timing": single["timing"]})
    out["single_launch"] = single
    if evidence:
        out.update(evidence)
    return out


def host_link_evidence(streamer, pipe, s_h, b_h, down_h, outs_h):
    """The host link right after the e2e steps, in the same process: the step's
    input copies alone (5 back to back), the same copies with the output copy
    of each step behind them but no compute (10 steps, pipelined as in the
    e2e steps), and 20 more e2e steps. Its throughput moves by 10-20% between
    boxes and runs, so the e2e value is read against these."""
    import torch

    def window(submit, first, last, n):
        for i in range(2):
            submit(i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(first)
        for i in range(n):
            submit(i + 2)
        e1.record(last)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def inputs(i):
        slot = streamer.slots[i % 2]
        with torch.cuda.stream(streamer.copy_in):
            slot["scores"].copy_(s_h, non_blocking=True)
            slot["bias"].copy_(b_h, non_blocking=True)
            slot["down"].copy_(down_h, non_blocking=True)
            slot["copied_in"].record(streamer.copy_in)

    def copies(i):
        inputs(i)
        slot = streamer.slots[i % 2]
        streamer.copy_out.wait_event(slot["copied_in"])
        with torch.cuda.stream(streamer.copy_out):
            outs_h[i % 2].copy_(slot["out"], non_blocking=True)

    return {
        "h2d_only_ms": window(inputs, streamer.copy_in, streamer.copy_in, 5),
        "copies_only_ms": window(copies, streamer.copy_in, streamer.copy_out, 10),
        "e2e_again_ms": window(lambda i: streamer.submit(s_h, b_h, down_h, outs_h[i % 2]),
                               streamer.copy_in, streamer.copy_out, 20),
        "note": "ms per step: input copies alone; input and output copies pipelined without "
                "compute; 20 more e2e steps"}


READ_FLOOR_SHAPES = [(152 * m, b) for m in (1, 2, 4, 8) for b in (256, 512)]


def pick_read_floor(times: dict):
    """The fastest (grid, block) of a sweep {shape: us per launch, or None};
    None when no shape was timed."""
    timed = {k: v for k, v in times.items() if v is not None}
    if not timed:
        return None
    best = min(timed, key=timed.get)
    return best, timed[best]


def streaming_read_floor(bufs, n: int, dev, peak):
    """What one launch that only reads the score bytes costs: the bench's
    streaming-read kernel (bench_read_floor.cu: 16-byte loads at a grid
    stride, summed in registers, one partial sum per CTA) over the same
    rotating score copies, captured in a CUDA graph and replayed like the
    router, at the fastest of a few grid and block sizes. Its per-CTA sums are
    checked against torch.sum of the same buffer, so the timed kernel is known
    to read every word. None when the kernel was not built."""
    import ctypes

    import torch
    path = os.path.join(ROOT, "bench_read_floor.so")
    if not os.path.exists(path):
        return {"note": "bench_read_floor.so not built (__graft_entry__.build builds it)"}
    lib = ctypes.CDLL(path)
    lib.read_floor_launch.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.read_floor_launch.restype = ctypes.c_int
    n4 = bufs[0].numel() // 4
    nbytes = 16 * n4
    partial = torch.zeros(max(g for g, _ in READ_FLOOR_SHAPES), dtype=torch.float32, device=dev)
    ptrs = [b.data_ptr() for b in bufs]

    def launcher(grid, block):
        def call(i, st):
            rc = lib.read_floor_launch(ptrs[i % len(ptrs)], n4, partial.data_ptr(), grid, block,
                                       st.cuda_stream)
            if rc != 0:
                raise RuntimeError(f"read_floor_launch failed: {rc}")
        return call

    times = {shape: time_graph_replay(launcher(*shape), n, dev) for shape in READ_FLOOR_SHAPES}
    pick = pick_read_floor(times)
    if pick is None:
        return {"note": "graph capture failed"}
    (grid, block), us = pick
    # the check: one launch on buffer 0 at the chosen shape
    s = torch.cuda.current_stream(dev)
    partial.zero_()
    launcher(grid, block)(0, s)
    torch.cuda.synchronize(dev)
    got = float(partial[:grid].double().sum())
    want = float(bufs[0].double().sum())
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us_per_launch": us, "achieved_gbs": gbs, "frac": gbs / peak,
            "shape": f"{grid} CTAs x {block} threads",
            "sweep_us": {f"{g}x{b}": t for (g, b), t in times.items()},
            "sum_rel_err": abs(got - want) / max(abs(want), 1e-30)}


def router_evidence(moe, cfg, s_d, b_d, dev, stream, peak):
    """The router alone, launched back to back: on the workload's batch
    rotating over copies whose total exceeds L2 twice over, on a 262144-token
    batch (one 268 MB input, larger than L2), and on 8 tokens (one chunk: the
    per-launch floor of the same kernel, with next to no data)."""
    import torch

    import synth
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    T, E, K = cfg.T, cfg.E, cfg.K
    nbuf = max(2, -(-2 * l2 // (4 * T * E)))
    bufs = [s_d.clone() for _ in range(nbuf)]
    n = 48

    lib = moe.load_library()
    sh = stream.cuda_stream

    def route_fn(src, ids, w, on_stream=False):
        # the C ABI called directly with the pointers taken once, so that the
        # host enqueues faster than the device runs the launches
        ptrs = [x.data_ptr() for x in src]
        Tn = src[0].shape[0]
        a = (ids.data_ptr(), w.data_ptr())

        def call(i, st=None):
            rc = lib.moe_route(a[0], a[1], ptrs[i % len(ptrs)], b_d.data_ptr(), Tn, E, K, cfg.G,
                               cfg.M, int(cfg.norm_weights), float(cfg.scale),
                               st.cuda_stream if st is not None else sh)
            if rc != 0:
                raise RuntimeError(f"moe_route failed: {rc}")
        return call

    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    f = route_fn(bufs, ids, w)
    for i in range(3):
        f(i)
    hb = {}
    b2b = time_back_to_back(f, n, stream, hb)
    graph_b2b = time_graph_replay(f, n, dev)
    # the same bytes read by a library reduction (torch.sum of each score row,
    # into a preallocated vector), replayed the same way: what one launch that
    # only reads the scores costs with a stock kernel on this GPU
    acc = torch.empty((T,), dtype=torch.float32, device=dev)

    def read_fn(i, st=None):
        torch.sum(bufs[i % len(bufs)], dim=1, out=acc)
    read_graph = time_graph_replay(read_fn, n, dev)
    stream_read = streaming_read_floor(bufs, n, dev, peak)
    del bufs
    big_T = 262144
    big = torch.from_numpy(synth.make_scores(cfg.replace(T=big_T))).to(dev)
    ids_b = torch.empty((big_T, K), dtype=torch.int32, device=dev)
    w_b = torch.empty((big_T, K), dtype=torch.float32, device=dev)
    fb = route_fn([big], ids_b, w_b)
    for i in range(3):
        fb(i)
    big_b2b = time_back_to_back(fb, 20, stream)
    big_graph = time_graph_replay(fb, 20, dev, reps=3)
    del big, ids_b, w_b
    small = s_d[:8].contiguous()
    fs = route_fn([small], ids[:8].contiguous(), w[:8].contiguous())
    for i in range(3):
        fs(i)
    hf = {}
    floor = time_back_to_back(fs, n, stream, hf)
    floor_graph = time_graph_replay(fs, n, dev)
    rb = router_bytes(T, E, K)
    bb = router_bytes(big_T, E, K)

    def graph_entry(us, nbytes):
        if us is None:
            return None
        return {"us_per_launch": us, "achieved_gbs": nbytes / (us * 1e-6) / 1e9,
                "frac": nbytes / (us * 1e-6) / 1e9 / peak}
    return {
        "back_to_back": dict(hb, **{"launches": n, "us_per_launch": b2b,
                         "achieved_gbs": rb / (b2b * 1e-6) / 1e9,
                         "frac": rb / (b2b * 1e-6) / 1e9 / peak,
                         "inputs": f"{nbuf} copies of the {T}-token score matrix in rotation "
                                   f"({nbuf * 4 * T * E / 1e6:.0f} MB, L2 {l2 / 1e6:.0f} MB)"}),
        "large_batch": {"tokens": big_T, "launches": 20, "us_per_launch": big_b2b,
                        "achieved_gbs": bb / (big_b2b * 1e-6) / 1e9,
                        "frac": bb / (big_b2b * 1e-6) / 1e9 / peak,
                        "algorithmic_bytes": bb},
        "launch_floor": dict(hf, **{"tokens": 8, "launches": n, "us_per_launch": floor,
                                    "note": "the same router on one 8-token chunk, back to "
                                            "back"}),
        "graph_replay": {
            "note": "the same launches captured in a CUDA graph and replayed: no host work "
                    "per launch",
            "back_to_back": graph_entry(graph_b2b, rb),
            "large_batch": graph_entry(big_graph, bb),
            "launch_floor_us": floor_graph,
            "read_only_kernel": graph_entry(read_graph, 4 * T * E),
            "streaming_read": stream_read},
        "one_launch_read_ceiling": (
            {"us_per_launch": stream_read["us_per_launch"], "frac": stream_read["frac"],
             "note": "graph_replay.streaming_read: a launch that only reads these bytes"}
            if "frac" in stream_read else None),
        "hbm_time_at_peak_us": rb / (peak * 1e3),
        "residue_over_hbm_time_us": b2b - rb / (peak * 1e3),
    }


def secondary_workload(moe, name, dev, stream, peak, flush_l2, reps=50, graph_steps=0):
    """Route + index and finalize stage times of another workload (an event
    between the two, L2 flushed before each step), the whole step with events
    only at its ends (tokens/s); with graph_steps > 0 also the time
    per whole step when that many steps, captured in a CUDA graph, replay
    back to back (no host work between launches; the inputs stay wherever
    the previous step left them)."""
    import statistics

    import torch

    import synth
    c = synth.get_config(name)
    scores = torch.from_numpy(synth.make_scores(c)).to(dev)
    bias = torch.from_numpy(synth.make_bias(c)).to(dev)
    down = torch.empty((c.N, c.H), dtype=torch.bfloat16)
    synth.make_down(c, out_ptr=down.data_ptr())
    down = down.to(dev)
    pipe = moe.RoutingPipeline(c.T, c.E, c.K, c.H, c.G, c.M, c.norm_weights, c.scale,
                               device=dev, fused=True)
    for _ in range(3):
        pipe(scores, bias, down)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    for i in range(reps):
        flush_l2()
        ev[i][0].record(stream)
        pipe.route_and_index(scores, bias)
        ev[i][1].record(stream)
        pipe.finalize(down)
        ev[i][2].record(stream)
    # whole steps with events only at their ends (finalize launches early)
    wev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    for i in range(reps):
        flush_l2()
        wev[i][0].record(stream)
        pipe(scores, bias, down)
        wev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ri = statistics.fmean([e[0].elapsed_time(e[1]) for e in ev])
    fin = statistics.fmean([e[1].elapsed_time(e[2]) for e in ev])
    step = statistics.fmean([e[0].elapsed_time(e[1]) for e in wev])
    fb = 2 * c.N * c.H + 8 * c.N + 2 * c.T * c.H
    ok = moe.moe_read_device_status(pipe.fused_workspace) == 0
    out = {"tokens": c.T, "n_routed_experts": c.E, "n_experts_per_tok": c.K, "hidden": c.H,
           "route_index_ms": ri, "finalize_ms": fin, "step_ms": step,
           "step_with_stage_event_ms": ri + fin,
           "tokens_per_s": c.T / (step * 1e-3),
           "finalize_gbs": fb / (fin * 1e-3) / 1e9, "finalize_frac": fb / (fin * 1e-3) / 1e9 / peak,
           "finalize_algorithmic_bytes": fb, "device_status_clean": ok, "reps": reps}
    if graph_steps > 0:
        out["graph_replay_step_us"] = time_graph_replay(
            lambda i, st: pipe(scores, bias, down, stream=st), graph_steps, dev)
    del pipe, scores, bias, down
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- GPU arm
def run_gpu(args, cfg, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist

    import moe_token_routing_gb300 as moe

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    moe.load_library()
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    scores, bias, down_h, down_np = host_inputs(cfg, seed_offset=rank, pinned=True)
    s_d = torch.from_numpy(scores).to(dev)
    b_d = torch.from_numpy(bias).to(dev)
    d_d = down_h.to(dev)
    fused = not args.separate_index
    pipe = moe.RoutingPipeline(cfg.T, cfg.E, cfg.K, cfg.H, cfg.G, cfg.M, cfg.norm_weights,
                               cfg.scale, device=dev, fused=True)
    pipe.fused = fused  # both paths stay available for the stage pass
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush_l2():
        flush_w.zero_()
        flush_r.sum()

    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        flush_l2()
        pipe(s_d, b_d, d_d)
    torch.cuda.synchronize(dev)

    K = args.steps
    # Timed region: events only at the step start and end, so the route_index
    # launches (router, rows, scatter; or route -> create_indices with
    # --separate-index) and finalize chain back to back as a caller runs them
    # (an event between two launches keeps the second from starting early).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    sampler = ClockSampler(device_uuid(dev))
    sampler.start()
    time.sleep(0.25)
    barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(K):
        flush_l2()
        e = ev[i]
        e[0].record(stream)
        pipe.route_and_index(s_d, b_d)
        pipe.finalize(d_d)
        e[1].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    wall = time.perf_counter() - wall0
    # The same K steps again with an event between route + index and
    # finalize: finalize's own duration in the steps (the roofline) and
    # route + index's.
    sev_steps = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        flush_l2()
        e = sev_steps[i]
        e[0].record(stream)
        pipe.route_and_index(s_d, b_d)
        e[1].record(stream)
        pipe.finalize(d_d)
        e[2].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()

    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    fin_ms = [e[1].elapsed_time(e[2]) for e in sev_steps]
    ri_ms = [e[0].elapsed_time(e[1]) for e in sev_steps]
    split_step_ms = [e[0].elapsed_time(e[2]) for e in sev_steps]
    mean_step = statistics.fmean(step_ms)

    # Per-stage durations (after the timed region): an event between every stage.
    # Each pass starts with untimed calls, so that no first call (module
    # loading, shared-memory opt-in) lands in a timed one.
    ks = min(K, 200)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(ks)]
    for _ in range(3):
        pipe.route(s_d, b_d)
        pipe.create_indices()
        pipe.route_index(s_d, b_d)
    for i in range(ks):
        flush_l2()
        e = sev[i]
        e[0].record(stream)
        pipe.route(s_d, b_d)
        e[1].record(stream)
        pipe.create_indices()
        e[2].record(stream)
        pipe.finalize(d_d)
        e[3].record(stream)
    torch.cuda.synchronize(dev)
    route_ms = [e[0].elapsed_time(e[1]) for e in sev]
    index_ms = [e[1].elapsed_time(e[2]) for e in sev]
    fin_stage_ms = [e[2].elapsed_time(e[3]) for e in sev]
    # moe_route_index (the steps' default route + index) as a stage of its own
    for i in range(ks):
        flush_l2()
        e = sev[i]
        e[0].record(stream)
        pipe.route_index(s_d, b_d)
        e[1].record(stream)
        pipe.finalize(d_d)
        e[2].record(stream)
    torch.cuda.synchronize(dev)
    fused_ms = [e[0].elapsed_time(e[1]) for e in sev]
    # the single-launch variant (one cooperative kernel) on buffers of its own
    single = moe.RouteIndexBuffers(cfg.T, cfg.E, cfg.K, dev, single_launch=True)
    for _ in range(3):
        single.run(s_d, b_d, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    for i in range(ks):
        flush_l2()
        e = sev[i]
        e[0].record(stream)
        single.run(s_d, b_d, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
        e[1].record(stream)
    torch.cuda.synchronize(dev)
    single_ms = [e[0].elapsed_time(e[1]) for e in sev]
    single_ok = single.device_status() == 0
    del single
    status_ok = (moe.moe_read_device_status(pipe.fused_workspace) == 0
                 and moe.moe_read_device_status(pipe.index.workspace) == 0)

    # whole-job throughput: max over ranks of the mean step time
    worst_ms = max_over_ranks(mean_step, world, dev)

    # correctness spot check of this run's output against the first token rows
    out_ok = bool(torch.isfinite(pipe.output[:4].float()).all().item())

    # ---- next row (not in the step): expert-contiguous token rows for the grouped matmul
    x_h = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, pin_memory=True)
    import synth
    synth.make_input(cfg.replace(seed=cfg.seed + rank), out_ptr=x_h.data_ptr())
    x_d = x_h.to(dev)
    perm_out = torch.empty((cfg.N, cfg.H), dtype=torch.bfloat16, device=dev)
    pipe.permute(x_d, perm_out)
    kp = min(K, 100)
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(kp)]
    for i in range(kp):
        flush_l2()
        pev[i][0].record(stream)
        pipe.permute(x_d, perm_out)
        pev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    perm_ms = statistics.fmean([e[0].elapsed_time(e[1]) for e in pev])
    del perm_out, x_d

    # ---- next row (not in the step): router with the fused sigmoid score loader on logits
    logits = synth.normal_f32(cfg.seed + rank, synth.TENSOR_SCORES, cfg.T * cfg.E)
    logits_d = torch.from_numpy(logits.reshape(cfg.T, cfg.E)).to(dev)
    ids_x = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device=dev)
    w_x = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device=dev)
    for i in range(kp):
        flush_l2()
        pev[i][0].record(stream)
        moe.moe_route_ex(ids_x, w_x, logits_d, b_d, cfg.G, cfg.M, cfg.norm_weights, cfg.scale,
                         moe.SCORES_SIGMOID)
        pev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    sig_ms = statistics.fmean([e[0].elapsed_time(e[1]) for e in pev])
    for i in range(kp):
        flush_l2()
        pev[i][0].record(stream)
        moe.moe_route_ex(ids_x, w_x, logits_d, b_d, cfg.G, cfg.M, cfg.norm_weights, cfg.scale,
                         moe.SCORES_SOFTMAX)
        pev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    soft_ms = statistics.fmean([e[0].elapsed_time(e[1]) for e in pev])

    # ---- the router's own evidence and the other large workloads (rank 0, after
    # the timed steps)
    peak_gbs, _ = measured_hbm_peak()
    extras = {}
    if rank == 0 and not args.no_extras:
        extras["router"] = router_evidence(moe, cfg, s_d, b_d, dev, stream, peak_gbs)
        for name in ("skewed_ungrouped", "few_expert_large_batch", "dsv3_decode"):
            if name != cfg.name:
                extras[name] = secondary_workload(
                    moe, name, dev, stream, peak_gbs, flush_l2,
                    graph_steps=32 if name == "dsv3_decode" else 0)

    # ---- end to end through the host-buffer API: pinned inputs copied in and the
    # output copied back every step, copies of consecutive steps overlapped
    s_h = torch.from_numpy(scores).pin_memory()
    b_h = torch.from_numpy(bias).pin_memory()
    outs_h = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    streamer = pipe.stream_from_host(depth=2)
    for i in range(2):
        streamer.submit(s_h, b_h, down_h, outs_h[i % 2])
    streamer.synchronize()
    ke = max(1, args.e2e_steps)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    # Steady state of a stream of batches: three untimed steps first, then the
    # timed region starts in stream order right behind their copies (after an
    # idle gap, the first copy over this host link measured 30 ms slower).
    for i in range(3):
        streamer.submit(s_h, b_h, down_h, outs_h[i % 2])
    e0.record(streamer.copy_in)
    for i in range(ke):
        streamer.submit(s_h, b_h, down_h, outs_h[(i + 3) % 2])
    e1.record(streamer.copy_out)
    streamer.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / ke, world, dev)
    h2d, d2h = pipe.host_bytes()
    host_link = (None if args.no_extras
                 else host_link_evidence(streamer, pipe, s_h, b_h, down_h, outs_h))

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    nbytes = algorithmic_bytes(cfg)
    peak, peak_kind = measured_hbm_peak()
    fin_mean = statistics.fmean(fin_ms)
    route_mean = statistics.fmean(route_ms)
    fin_gbs = nbytes["finalize"] / (fin_mean * 1e-3) / 1e9
    route_gbs = nbytes["route"] / (route_mean * 1e-3) / 1e9
    launches_per_step = ((2 if cfg.N <= 1024 else 3) if fused
                         else 1 + index_launches(cfg.N, cfg.E)) + 1

    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, scores, bias, down_np, args.cpu_seconds)

    line = {
        "metric": METRIC,
        "value": job_tokens_per_s(cfg.T, world, worst_ms),
        "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": worst_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded)",
        "config": dict(config_dict(cfg), route_index="fused (moe_route_index: counting router, "
                       "row prefixes, scatter)" if fused
                       else "separate (moe_route, moe_create_indices)"),
        "roofline": {"kernel": "finalize", "bound": "hbm", "achieved": fin_gbs, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": fin_gbs / peak,
                     "frac_vs_nominal_8tbs": fin_gbs / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": nbytes["finalize"],
                     "timing": "finalize between events in a second pass of the same K timed "
                               "steps, with an event between route + index and finalize",
                     "traffic": profile_traffic("finalize.cu", "finalize_dsv3_prefill.txt")
                     if cfg.name == "dsv3_prefill" else None},
        "router_roofline": router_roofline(route_gbs, route_mean, peak, nbytes["route"],
                                           extras.get("router")),
        "secondary_workloads": {k: v for k, v in extras.items() if k != "router"},
        "stages_ms": {"route": route_mean, "create_indices": statistics.fmean(index_ms),
                      "route_index_fused": statistics.fmean(fused_ms),
                      "route_index_single_launch": statistics.fmean(single_ms),
                      "finalize": statistics.fmean(fin_stage_ms),
                      "route_plus_index_in_timed_steps": statistics.fmean(ri_ms),
                      "step_with_stage_event": statistics.fmean(split_step_ms),
                      "step_median": statistics.median(step_ms),
                      "timed_steps_route_index": "fused" if fused else "separate",
                      "note": "route/create_indices/finalize and route_index_fused from "
                              "separate passes with an event between every stage; the timed "
                              "steps carry events only at the step start and end; a second "
                              "pass of the same steps with an event before finalize gives "
                              "route_plus_index_in_timed_steps, step_with_stage_event and "
                              "finalize's duration"},
        "next_rows": {"permute": {
            "ms": perm_ms, "tokens_per_s": cfg.T / (perm_ms * 1e-3),
            "achieved_gbs": (2 * cfg.T * cfg.H + 2 * cfg.N * cfg.H + 4 * cfg.N) / (perm_ms * 1e-3) / 1e9,
            "frac_of_peak": (2 * cfg.T * cfg.H + 2 * cfg.N * cfg.H + 4 * cfg.N)
            / (perm_ms * 1e-3) / 1e9 / peak,
            "algorithmic_bytes": 2 * cfg.T * cfg.H + 2 * cfg.N * cfg.H + 4 * cfg.N,
            "note": "measured after the timed steps; not part of the step"},
            "route_sigmoid_logits": {
                "ms": sig_ms, "tokens_per_s": cfg.T / (sig_ms * 1e-3),
                "achieved_gbs": nbytes["route"] / (sig_ms * 1e-3) / 1e9,
                "note": "moe_route_ex with the fused sigmoid loader on gate logits; "
                        "same bytes as route"},
            "route_softmax_logits": {
                "ms": soft_ms, "tokens_per_s": cfg.T / (soft_ms * 1e-3),
                "achieved_gbs": nbytes["route"] / (soft_ms * 1e-3) / 1e9,
                "note": "moe_route_ex with the fused softmax loader on gate logits (sum over "
                        "experts in ascending order); same bytes as route"}},
        "stages_tokens_per_s": {"route": cfg.T / (route_mean * 1e-3),
                                "create_indices": cfg.T / (statistics.fmean(index_ms) * 1e-3),
                                "finalize": cfg.T / (fin_mean * 1e-3)},
        "cpu_baseline": cpu,
        "e2e": {"value": job_tokens_per_s(cfg.T, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": ke,
                "api": "RoutingPipeline.stream_from_host (copies of consecutive steps overlap)",
                "timing": "steady state: the timed steps follow three untimed ones in stream "
                          "order; events on the copy-in stream at the start and the copy-out "
                          "stream at the end",
                "host_link": host_link and dict(
                    host_link, h2d_gbs=h2d / (host_link["h2d_only_ms"] * 1e-3) / 1e9)},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "wall_s_timed_region": wall,
        "output_finite": out_ok,
        "device_status_clean": status_ok and single_ok,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_router_only(args, cfg, local_rank):
    """The router alone on cfg's scores: --warmup untimed launches, then
    --steps launches back to back between one event pair; prints one JSON
    line (a profiling aid, not the bench's metric)."""
    import json as _json

    import torch

    import moe_token_routing_gb300 as moe
    import synth
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    s_d = torch.from_numpy(synth.make_scores(cfg)).to(dev)
    b_d = torch.from_numpy(synth.make_bias(cfg)).to(dev)
    ids = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device=dev)
    w = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device=dev)

    def call():
        moe.moe_route(ids, w, s_d, b_d, cfg.G, cfg.M, cfg.norm_weights, cfg.scale)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) * 1e3 / max(1, args.steps)
    nbytes = 4 * cfg.T * cfg.E + 4 * cfg.E + 8 * cfg.T * cfg.K
    peak, _ = measured_hbm_peak()
    print(_json.dumps({"router_only": cfg.name, "tokens": cfg.T, "launches": args.steps,
                       "us_per_launch": us, "achieved_gbs": nbytes / (us * 1e-6) / 1e9,
                       "frac": nbytes / (us * 1e-6) / 1e9 / peak}))


def main():
    args = parse_args()
    rank, world, local_rank = dist_env()
    import __graft_entry__
    __graft_entry__.build()
    import synth
    cfg = synth.get_config(args.config)
    if args.tokens is not None:
        cfg = cfg.replace(T=args.tokens)
    if args.impl == "reference":
        run_reference(args, cfg, rank, world)
        return
    if args.router_only:
        run_router_only(args, cfg, local_rank)
        return
    run_gpu(args, cfg, rank, world, local_rank)


if __name__ == "__main__":
    main()
