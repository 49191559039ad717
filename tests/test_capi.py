"""The C ABI library without a GPU: it loads, exports every entry point that
include/moe_routing.h declares, and rejects bad arguments on the host before
touching CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe_routing.h")


@pytest.fixture(scope="module")
def lib():
    from moe_token_routing_gb300 import build
    build.build()
    import moe_token_routing_gb300 as moe
    return moe.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z_]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(
        ["moe_status_string", "moe_route", "moe_create_indices_workspace_size",
         "moe_create_indices", "moe_finalize", "moe_read_device_status",
         "moe_create_indices_no_alloc", "moe_permute", "moe_finalize_ex", "moe_route_ex",
         "moe_route_index_workspace_size", "moe_route_index",
         "moe_route_index_single_launch_workspace_size", "moe_route_index_single_launch"])


def test_every_declared_symbol_is_exported(lib):
    import moe_token_routing_gb300 as moe
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(moe.EXPORTED_SYMBOLS) == declared_functions()


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(6) == b"MOE_ERR_WORKSPACE"
    assert lib.moe_status_string(7) == b"MOE_ERR_DEVICE_DATA"
    assert lib.moe_status_string(99) == b"MOE_ERR_UNKNOWN"


def test_workspace_size_query(lib):
    assert lib.moe_create_indices_workspace_size(0, 8) == 256
    assert lib.moe_create_indices_workspace_size(1024, 8) == 256   # one CTA: no count matrix
    assert lib.moe_create_indices_workspace_size(1025, 8) > 256
    big = lib.moe_create_indices_workspace_size(131072, 256)
    assert big >= 64 * 256 * 4 and big % 256 == 0
    assert lib.moe_create_indices_workspace_size(-1, 8) == 0
    assert lib.moe_create_indices_workspace_size(10, 0) == 0
    assert lib.moe_create_indices_workspace_size(10, 1025) == 0


def route_index_workspace_bytes(T, E, K):
    """256-byte header, a fixed [1024] block of per-expert totals, then room
    for the [E][row] count and prefix matrices (row = the 1024-slot chunks
    rounded up to 4), each rounded up to 256 bytes."""
    chunks = max(-(-(T * K) // 1024), 1)
    row = (chunks + 3) // 4 * 4
    return 256 + 4 * 1024 + 2 * ((4 * E * row + 255) // 256 * 256)


def test_route_index_workspace_size_query(lib):
    f = lib.moe_route_index_workspace_size
    for T, E, K in ((0, 8, 2), (64, 256, 8), (16384, 256, 8), (131072, 8, 2), (33, 96, 5)):
        assert f(T, E, K) == route_index_workspace_bytes(T, E, K), (T, E, K)
    assert f(0, 8, 1) == 4352 + 512
    assert f(-1, 8, 2) == 0
    assert f(10, 0, 2) == 0
    assert f(10, 8, 0) == 0
    assert f(10, 8, 33) == 0


def single_launch_workspace_bytes(T, E):
    """256-byte header, four 256-byte counter blocks, then [E][R] tagged counts
    and prefixes, E tagged totals
    and R tagged status words (8 bytes each), every part rounded up to 256
    bytes; R = the CTA bound (one CTA per 8 tokens, at most 2048) rounded up to 4."""
    r256 = lambda x: (x + 255) // 256 * 256
    ctas = min(max((T + 7) // 8, 1), 2048)
    R = (ctas + 3) // 4 * 4
    return 256 + 1024 + 2 * r256(8 * E * R) + r256(8 * E) + r256(8 * R)


def test_single_launch_workspace_size_query(lib):
    f = lib.moe_route_index_single_launch_workspace_size
    for T, E in ((0, 8), (64, 256), (16384, 256), (131072, 8), (10 ** 9, 1024), (33, 96)):
        assert f(T, E) == single_launch_workspace_bytes(T, E), (T, E)
    assert f(0, 8) == 2304
    assert f(16384, 256) == 256 + 1024 + 2 * 8 * 256 * 2048 + 2048 + 8 * 2048
    assert f(-1, 8) == 0
    assert f(10, 0) == 0
    assert f(10, 1025) == 0


FAKE = 0x7f0000001000  # never dereferenced: every call below fails host validation


def test_route_host_validation(lib):
    f = lib.moe_route
    ok = (FAKE, FAKE, FAKE, FAKE)
    assert f(*ok, 4, 256, 8, 7, 4, 1, 1.0, None) == 2      # E % n_groups
    assert f(*ok, 4, 256, 8, 8, 9, 1, 1.0, None) == 2      # topk_group > n_groups
    assert f(*ok, 4, 256, 0, 8, 4, 1, 1.0, None) == 2      # K < 1
    assert f(*ok, 4, 16, 5, 4, 1, 1, 1.0, None) == 2       # K > topk_group * group size
    assert f(*ok, -1, 256, 8, 8, 4, 1, 1.0, None) == 2     # T < 0
    assert f(*ok, 4, 2048, 8, 8, 4, 1, 1.0, None) == 4     # E above the limit
    assert f(*ok, 4, 256, 8, 64, 4, 1, 1.0, None) == 4     # n_groups above the limit
    assert f(None, FAKE, FAKE, FAKE, 4, 256, 8, 8, 4, 1, 1.0, None) == 1
    assert f(FAKE + 2, FAKE, FAKE, FAKE, 4, 256, 8, 8, 4, 1, 1.0, None) == 3
    assert f(None, None, None, None, 0, 256, 8, 8, 4, 1, 1.0, None) == 0  # T = 0: nothing to do


def test_route_ex_host_validation(lib):
    f = lib.moe_route_ex
    ok = (FAKE, FAKE, FAKE, FAKE)
    assert f(*ok, 4, 256, 8, 8, 4, 1, 1.0, 7, None) == 4      # unknown score loader
    assert f(*ok, 4, 256, 8, 8, 4, 1, 1.0, 3, None) == 4
    assert f(*ok, 4, 256, 8, 7, 4, 1, 1.0, 1, None) == 2      # E % n_groups
    assert f(None, None, None, None, 0, 256, 8, 8, 4, 1, 1.0, 1, None) == 0


def test_create_indices_host_validation(lib):
    f = lib.moe_create_indices
    outs = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    ws = lib.moe_create_indices_workspace_size(100000, 64)
    # scale offsets would pass 2^32 (N + 127 * E): rejected before anything is enqueued
    assert f(*outs, 0xFFFFFF00, 64, FAKE, ws, FAKE, None) == 4
    assert f(*outs, 100000, 64, FAKE, ws - 1, None, None) == 6      # workspace too small
    assert f(*outs, 100000, 64, None, ws, None, None) == 6          # no workspace
    assert f(*outs, 100000, 64, FAKE + 16, ws, None, None) == 3     # workspace alignment
    assert f(*outs, -1, 64, FAKE, ws, None, None) == 2
    assert f(*outs, 10, 0, FAKE, ws, None, None) == 2
    assert f(*outs, 10, 2000, FAKE, ws, None, None) == 4
    assert f(FAKE, None, FAKE, FAKE, FAKE, FAKE, 10, 64, FAKE, ws, None, None) == 1
    assert f(FAKE + 1, FAKE, FAKE, FAKE, FAKE, FAKE, 10, 64, FAKE, ws, None, None) == 3


@pytest.mark.parametrize("single", [False, True])
def test_route_index_host_validation(lib, single):
    f = lib.moe_route_index_single_launch if single else lib.moe_route_index
    outs = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    ins = (FAKE, FAKE)
    ws = (lib.moe_route_index_single_launch_workspace_size(1000, 256) if single
          else lib.moe_route_index_workspace_size(1000, 256, 8))
    cfg = (1000, 256, 8, 8, 4, 1, 1.0)
    assert f(*outs, *ins, *cfg, 7, FAKE, ws, None, None) == 4          # unknown score loader
    assert f(*outs, *ins, 1000, 256, 8, 7, 4, 1, 1.0, 0, FAKE, ws, None, None) == 2  # E % G
    assert f(*outs, *ins, 1000, 256, 0, 8, 4, 1, 1.0, 0, FAKE, ws, None, None) == 2  # K < 1
    big = 0x80000000  # T * K = 2^32 slots: beyond the uint32 index outputs
    assert f(*outs, *ins, big, 256, 2, 8, 4, 1, 1.0, 0, FAKE, ws, None, None) == 4
    assert f(*outs, *ins, *cfg, 0, FAKE, ws - 1, None, None) == 6      # workspace too small
    assert f(*outs, *ins, *cfg, 0, None, ws, None, None) == 6          # no workspace
    assert f(*outs, *ins, *cfg, 0, FAKE + 64, ws, None, None) == 3     # workspace alignment
    assert f(FAKE, FAKE, None, *outs[3:], *ins, *cfg, 0, FAKE, ws, None, None) == 1
    assert f(*outs[:3], None, *outs[4:], *ins, *cfg, 0, FAKE, ws, None, None) == 1
    assert f(*outs, None, FAKE, *cfg, 0, FAKE, ws, None, None) == 1    # no scores
    assert f(*outs[:2], FAKE + 2, *outs[3:], *ins, *cfg, 0, FAKE, ws, None, None) == 3
    assert f(*outs, *ins, *cfg, 0, FAKE, ws, FAKE + 1, None) == 3      # scales_offset alignment


def test_finalize_host_validation(lib):
    f = lib.moe_finalize
    p = (FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000)
    assert f(*p, 4, 2, 60, None) == 4          # hidden % 8
    assert f(*p, 4, 0, 64, None) == 2
    assert f(*p, 4, 33, 64, None) == 4
    assert f(*p, -1, 2, 64, None) == 2
    assert f(None, *p[1:], 4, 2, 64, None) == 1
    assert f(p[0] + 8, *p[1:], 4, 2, 64, None) == 3
    assert f(p[0], p[0], p[2], p[3], 4, 2, 64, None) == 2   # output overlaps down
    assert f(None, None, None, None, 0, 2, 64, None) == 0   # T = 0


def test_finalize_ex_host_validation(lib):
    f = lib.moe_finalize_ex
    o, d, r, w = FAKE, FAKE + 0x1000000, FAKE + 0x2000000, FAKE + 0x3000000
    assert f(o, 2, d, r, w, 1, 4, 2, 64, None, None) == 4       # unknown output dtype
    assert f(o, 0, d, r, w, 7, 4, 2, 64, None, None) == 4       # unknown weight dtype
    assert f(o, 1, d, r, w + 2, 1, 4, 2, 64, None, None) == 3   # fp32 weights need 4-byte alignment
    assert f(o, 1, d, r, w + 2, 0, 0, 2, 64, None, None) == 0   # T = 0
    assert f(o, 1, o, r, w, 0, 4, 2, 64, None, None) == 2       # output overlaps down
    assert f(o + 8, 1, d, r, w, 0, 4, 2, 64, None, None) == 3
    assert f(o, 1, d, r, w, 0, 4, 2, 64, FAKE + 2, None) == 3   # status word 4-byte aligned


def test_permute_host_validation(lib):
    f = lib.moe_permute
    p = (FAKE, FAKE + 0x1000000, FAKE + 0x2000000)
    assert f(*p, 4, 2, 60, None, None) == 4          # hidden % 8
    assert f(*p, 4, 0, 64, None, None) == 2
    assert f(*p, 4, 33, 64, None, None) == 4
    assert f(None, *p[1:], 4, 2, 64, None, None) == 1
    assert f(p[0] + 8, *p[1:], 4, 2, 64, None, None) == 3
    assert f(p[0], p[0], p[2], 4, 2, 64, None, None) == 2   # permuted overlaps input
    assert f(None, None, None, 0, 2, 64, None, None) == 0   # T = 0
    assert f(*p, 4, 2, 64, FAKE + 2, None) == 3           # status word 4-byte aligned


def test_device_status_host_validation(lib):
    out = ctypes.c_uint32(0)
    assert lib.moe_read_device_status(None, ctypes.byref(out), None) == 1
    assert lib.moe_read_device_status(FAKE, None, None) == 1


def test_binding_refuses_cpu_tensors():
    import torch
    import moe_token_routing_gb300 as moe
    s = torch.rand(4, 16)
    with pytest.raises(ValueError):
        moe.route(s, torch.zeros(16), 2, 4, 2, True, 1.0)
