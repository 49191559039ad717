"""Host logic of bench.py that needs no GPU: the hash-gated ncu traffic figure
and the command-line defaults."""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _tree(tmp_path, kernel_text, summary_hash, dram="2090510848"):
    src = tmp_path / "moe_token_routing_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text(kernel_text)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k_summary.txt").write_text(
        "# a comment: with a colon\n"
        f"dram_bytes_per_launch: {dram}\n"
        f"source_sha256_16: {summary_hash}\n")


def test_traffic_reported_only_for_the_profiled_source(tmp_path, monkeypatch):
    import bench
    text = "__global__ void k() {}\n"
    digest = hashlib.sha256(text.encode()).hexdigest()[:16]
    _tree(tmp_path, text, digest)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("k.cu", "k_summary.txt") == 2090510848
    # the kernel changed after the capture: no traffic figure
    (tmp_path / "moe_token_routing_gb300" / "csrc" / "k.cu").write_text(text + "// edited\n")
    assert bench.profile_traffic("k.cu", "k_summary.txt") is None


def test_traffic_missing_summary_is_none(tmp_path, monkeypatch):
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("finalize.cu", "absent.txt") is None


def test_committed_finalize_summary_matches_the_source():
    """The committed finalize summary carries the hash of the current
    finalize.cu, so the bench line's roofline.traffic is not null."""
    import bench
    assert bench.profile_traffic("finalize.cu", "finalize_dsv3_prefill.txt") is not None


def test_default_arguments(monkeypatch):
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse_args()
    assert a.gpus == 1 and a.impl == "gb300" and a.config == "dsv3_prefill"
    assert a.warmup >= 3 and not a.separate_index
    monkeypatch.setattr(sys, "argv", ["bench.py", "--separate-index", "--steps", "7"])
    a = bench.parse_args()
    assert a.separate_index and a.steps == 7 and not a.router_only
    monkeypatch.setattr(sys, "argv", ["bench.py", "--router-only", "--tokens", "262144"])
    a = bench.parse_args()
    assert a.router_only and a.tokens == 262144


def test_router_roofline_headline():
    """The router's headline is the back-to-back launches when they were
    measured, and the single launch (kept beside it) otherwise."""
    import bench
    ev = {"back_to_back": {"us_per_launch": 8.0, "achieved_gbs": 2000.0, "frac": 0.3}}
    r = bench.router_roofline(1500.0, 0.012, 6787.6, 17826816, ev)
    assert r["achieved"] == 2000.0 and abs(r["frac"] - 2000.0 / 6787.6) < 1e-12
    assert r["single_launch"]["achieved_gbs"] == 1500.0
    assert abs(r["single_launch"]["us_per_launch"] - 12.0) < 1e-9
    assert r["back_to_back"] is ev["back_to_back"]
    r = bench.router_roofline(1500.0, 0.012, 6787.6, 17826816, None)
    assert r["achieved"] == 1500.0
    assert r["timing"] == r["single_launch"]["timing"]


def test_read_floor_pick_and_shapes():
    """The streaming-read floor takes the fastest timed shape of its sweep; the
    shapes are whole multiples of the 152 SMs with block sizes the kernel
    accepts (a multiple of 32, at most 512)."""
    import bench
    assert bench.pick_read_floor({(152, 256): 5.0, (304, 512): 4.6, (608, 256): None}) == \
        ((304, 512), 4.6)
    assert bench.pick_read_floor({(152, 256): None}) is None
    for grid, block in bench.READ_FLOOR_SHAPES:
        assert grid % 152 == 0 and block % 32 == 0 and 32 <= block <= 512


def test_read_floor_kernel_is_built_for_sm_103a():
    """build() compiles the bench's streaming-read kernel and its launcher
    rejects shapes outside what the kernel handles without launching."""
    import ctypes
    import shutil
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("no nvcc")
    import __graft_entry__ as g
    path = g.build_read_floor()
    lib = ctypes.CDLL(path)
    lib.read_floor_launch.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.read_floor_launch.restype = ctypes.c_int
    # argument checks happen before any CUDA call
    assert lib.read_floor_launch(None, 4, 16, 152, 256, None) == -1
    assert lib.read_floor_launch(16, 4, 16, 152, 1024, None) == -1
    assert lib.read_floor_launch(18, 4, 16, 152, 256, None) == -1


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the contract's keys, on the tiny workload."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
