"""Thin ctypes binding of libmoe_routing.so.

Argument marshalling only: every step of the routing path runs in the CUDA
kernels behind the C ABI (include/moe_routing.h). PyTorch supplies device
memory and the current CUDA stream. There is no fallback: if the library is
missing or a tensor is not on a CUDA device, the call raises.

Names and argument order follow the C ABI, which follows the pages
("group_limited_router_kernel", "moe_create_indices", "moe_finalize").
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_NULL_PTR", 2: "MOE_ERR_INVALID_ARG",
                3: "MOE_ERR_MISALIGNED", 4: "MOE_ERR_UNSUPPORTED", 5: "MOE_ERR_CUDA",
                6: "MOE_ERR_WORKSPACE", 7: "MOE_ERR_DEVICE_DATA"}
MOE_ERR_DEVICE_DATA = 7
DEVICE_STATUS_BAD_EXPERT_ID = 0x1
DEVICE_STATUS_SYNC_TIMEOUT = 0x2
DEVICE_STATUS_SYNC_STATE = 0x4
DEVICE_STATUS_BAD_RESTORE_ORDER = 0x8

# Entry points declared in include/moe_routing.h.
EXPORTED_SYMBOLS = ("moe_status_string", "moe_route", "moe_create_indices_workspace_size",
                    "moe_create_indices", "moe_finalize", "moe_read_device_status",
                    "moe_create_indices_no_alloc", "moe_permute", "moe_finalize_ex",
                    "moe_route_ex", "moe_route_index_workspace_size", "moe_route_index",
                    "moe_route_index_single_launch_workspace_size",
                    "moe_route_index_single_launch")


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


class MoeLibraryMissing(RuntimeError):
    pass


_lib = None


def load_library(path: str = LIB_PATH):
    """Load the shared library (raises MoeLibraryMissing when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise MoeLibraryMissing(
            f"{path} not found: build it with moe_token_routing_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                             ctypes.c_size_t)
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_route.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, f32, vp]
    lib.moe_route.restype = ctypes.c_int
    lib.moe_create_indices_workspace_size.argtypes = [i64, i32]
    lib.moe_create_indices_workspace_size.restype = sz
    lib.moe_create_indices.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, vp, sz, vp, vp]
    lib.moe_create_indices.restype = ctypes.c_int
    lib.moe_finalize.argtypes = [vp, vp, vp, vp, i64, i32, i64, vp]
    lib.moe_finalize.restype = ctypes.c_int
    lib.moe_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.moe_read_device_status.restype = ctypes.c_int
    lib.moe_permute.argtypes = [vp, vp, vp, i64, i32, i64, vp, vp]
    lib.moe_permute.restype = ctypes.c_int
    lib.moe_finalize_ex.argtypes = [vp, ctypes.c_int, vp, vp, vp, ctypes.c_int, i64, i32, i64, vp,
                                    vp]
    lib.moe_finalize_ex.restype = ctypes.c_int
    lib.moe_route_ex.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, f32, ctypes.c_int,
                                 vp]
    lib.moe_route_ex.restype = ctypes.c_int
    lib.moe_route_index_workspace_size.argtypes = [i64, i32, i32]
    lib.moe_route_index_workspace_size.restype = sz
    lib.moe_route_index_single_launch_workspace_size.argtypes = [i64, i32]
    lib.moe_route_index_single_launch_workspace_size.restype = sz
    lib.moe_create_indices_no_alloc.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, vp, vp]
    lib.moe_create_indices_no_alloc.restype = ctypes.c_int
    for fn in (lib.moe_route_index, lib.moe_route_index_single_launch):
        fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, f32,
                       ctypes.c_int, vp, sz, vp, vp]
        fn.restype = ctypes.c_int
    _lib = lib
    return lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr() if t.numel() else 0


def _check(fn: str, rc: int):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def moe_route(expert_indices: torch.Tensor, expert_weights: torch.Tensor,
              expert_scores: torch.Tensor, expert_bias: torch.Tensor, n_groups: int,
              topk_group: int, norm_weights: bool, routed_scaling_factor: float,
              stream=None) -> None:
    """Group-limited top-k router (writes expert_indices [T,K] int32, expert_weights [T,K] fp32)."""
    T, E = expert_scores.shape
    K = expert_indices.shape[1] if expert_indices.dim() == 2 else 0
    args = (_dev(expert_indices, "expert_indices", torch.int32, (T, K)),
            _dev(expert_weights, "expert_weights", torch.float32, (T, K)),
            _dev(expert_scores, "expert_scores", torch.float32),
            _dev(expert_bias, "expert_bias", torch.float32, (E,)))
    rc = load_library().moe_route(*args, T, E, K, int(n_groups), int(topk_group),
                                  int(bool(norm_weights)), float(routed_scaling_factor),
                                  _stream(stream))
    _check("moe_route", rc)


SCORES_AS_GIVEN = 0
SCORES_SIGMOID = 1
SCORES_SOFTMAX = 2


def moe_route_ex(expert_indices: torch.Tensor, expert_weights: torch.Tensor,
                 expert_scores: torch.Tensor, expert_bias: torch.Tensor, n_groups: int,
                 topk_group: int, norm_weights: bool, routed_scaling_factor: float,
                 score_fn: int = SCORES_SIGMOID, stream=None) -> None:
    """moe_route with a fused score loader; with SCORES_SIGMOID expert_scores
    holds gate logits and the scores are their sigmoid."""
    T, E = expert_scores.shape
    K = expert_indices.shape[1] if expert_indices.dim() == 2 else 0
    args = (_dev(expert_indices, "expert_indices", torch.int32, (T, K)),
            _dev(expert_weights, "expert_weights", torch.float32, (T, K)),
            _dev(expert_scores, "expert_scores", torch.float32),
            _dev(expert_bias, "expert_bias", torch.float32, (E,)))
    rc = load_library().moe_route_ex(*args, T, E, K, int(n_groups), int(topk_group),
                                     int(bool(norm_weights)), float(routed_scaling_factor),
                                     int(score_fn), _stream(stream))
    _check("moe_route_ex", rc)


def moe_create_indices_workspace_size(num_slots: int, n_experts: int) -> int:
    return int(load_library().moe_create_indices_workspace_size(int(num_slots), int(n_experts)))


def moe_create_indices(token_expert_order: torch.Tensor, expert_start_indices: torch.Tensor,
                       restore_token_order: torch.Tensor, expert_ids: torch.Tensor,
                       expert_usage_stats: torch.Tensor, topk_ids: torch.Tensor,
                       workspace: torch.Tensor, stream=None) -> None:
    """Stable bucket sort of the flat topk_ids by expert (all outputs written in place).

    Unsigned outputs are carried in torch.int32 tensors (same bits as uint32)."""
    N = topk_ids.numel()
    E = expert_ids.numel()
    flat_ids = topk_ids.reshape(-1)
    args = (_dev(token_expert_order, "token_expert_order", torch.int32, (N,)),
            _dev(expert_start_indices, "expert_start_indices", torch.int32, (E + 1,)),
            _dev(restore_token_order, "restore_token_order", torch.int32, (N,)),
            _dev(expert_ids, "expert_ids", torch.int32, (E,)),
            _dev(expert_usage_stats, "expert_usage_stats", torch.int32, (2,)),
            _dev(flat_ids, "topk_ids", torch.int32))
    ws = _dev(workspace, "workspace", torch.uint8)
    rc = load_library().moe_create_indices(*args, N, E, ws, workspace.numel(), None,
                                           _stream(stream))
    _check("moe_create_indices", rc)


def moe_route_index_workspace_size(num_tokens: int, n_routed_experts: int,
                                   n_experts_per_tok: int) -> int:
    return int(load_library().moe_route_index_workspace_size(
        int(num_tokens), int(n_routed_experts), int(n_experts_per_tok)))


def moe_route_index_single_launch_workspace_size(num_tokens: int, n_routed_experts: int) -> int:
    return int(load_library().moe_route_index_single_launch_workspace_size(
        int(num_tokens), int(n_routed_experts)))


def moe_route_index(expert_indices: torch.Tensor, expert_weights: torch.Tensor,
                    token_expert_order: torch.Tensor, expert_start_indices: torch.Tensor,
                    restore_token_order: torch.Tensor, expert_ids: torch.Tensor,
                    expert_usage_stats: torch.Tensor, expert_scores: torch.Tensor,
                    expert_bias: torch.Tensor, n_groups: int, topk_group: int,
                    norm_weights: bool, routed_scaling_factor: float, workspace: torch.Tensor,
                    score_fn: int = SCORES_AS_GIVEN, scales_offset: torch.Tensor | None = None,
                    stream=None, single_launch: bool = False) -> None:
    """Router and index build with the router counting its own output (or, with
    single_launch, as one cooperative launch); the workspace must be
    zero-filled before its first use and belongs to one of the two."""
    T, E = expert_scores.shape
    K = expert_indices.shape[1] if expert_indices.dim() == 2 else 0
    N = T * K
    args = (_dev(expert_indices, "expert_indices", torch.int32, (T, K)),
            _dev(expert_weights, "expert_weights", torch.float32, (T, K)),
            _dev(token_expert_order, "token_expert_order", torch.int32, (N,)),
            _dev(expert_start_indices, "expert_start_indices", torch.int32, (E + 1,)),
            _dev(restore_token_order, "restore_token_order", torch.int32, (N,)),
            _dev(expert_ids, "expert_ids", torch.int32, (E,)),
            _dev(expert_usage_stats, "expert_usage_stats", torch.int32, (2,)),
            _dev(expert_scores, "expert_scores", torch.float32),
            _dev(expert_bias, "expert_bias", torch.float32, (E,)))
    ws = _dev(workspace, "workspace", torch.uint8)
    so = None if scales_offset is None else _dev(scales_offset, "scales_offset", torch.int32,
                                                 (E + 1,))
    lib = load_library()
    fn = lib.moe_route_index_single_launch if single_launch else lib.moe_route_index
    rc = fn(*args, T, E, K, int(n_groups), int(topk_group), int(bool(norm_weights)),
            float(routed_scaling_factor), int(score_fn), ws, workspace.numel(), so,
            _stream(stream))
    _check("moe_route_index_single_launch" if single_launch else "moe_route_index", rc)


def moe_finalize(output: torch.Tensor, down: torch.Tensor, restore_order: torch.Tensor,
                 router_weight: torch.Tensor, stream=None) -> None:
    """output[t] = sum_k router_weight[t,k] * down[restore_order[t*K+k]] (fp32 sum, bf16 out)."""
    T, K = router_weight.shape
    H = down.shape[1]
    args = (_dev(output, "output", torch.bfloat16, (T, H)),
            _dev(down, "down", torch.bfloat16, (T * K, H)),
            _dev(restore_order, "restore_order", torch.int32, (T * K,)),
            _dev(router_weight, "router_weight", torch.float32, (T, K)))
    rc = load_library().moe_finalize(*args, T, K, H, _stream(stream))
    _check("moe_finalize", rc)


def moe_permute(permuted: torch.Tensor, input: torch.Tensor, restore_token_order: torch.Tensor,
                stream=None, device_status: torch.Tensor | None = None) -> None:
    """permuted[restore_token_order[t*K+k]] = input[t]: the expert-contiguous token rows.
    device_status (optional int32 [1] on the device) receives
    DEVICE_STATUS_BAD_RESTORE_ORDER when an entry is >= T*K (skipped)."""
    T, H = input.shape
    N = restore_token_order.numel()
    K = N // T if T else 1
    if T and N != T * K:
        raise ValueError("restore_token_order must have T*K entries")
    args = (_dev(permuted, "permuted", torch.bfloat16, (N, H)),
            _dev(input, "input", torch.bfloat16),
            _dev(restore_token_order, "restore_token_order", torch.int32, (N,)))
    st = None if device_status is None else _dev(device_status, "device_status", torch.int32, (1,))
    _check("moe_permute", load_library().moe_permute(*args, T, K, H, st, _stream(stream)))


_DTYPE_CODES = {torch.bfloat16: 0, torch.float32: 1}


def moe_finalize_ex(output: torch.Tensor, down: torch.Tensor, restore_order: torch.Tensor,
                    router_weight: torch.Tensor, stream=None,
                    device_status: torch.Tensor | None = None) -> None:
    """moe_finalize with bf16 or fp32 router weights and a bf16 or fp32 output
    (taken from the tensors' dtypes). device_status (optional int32 [1] on the
    device) receives DEVICE_STATUS_BAD_RESTORE_ORDER when a restore_order entry
    is >= T*K (skipped)."""
    T, K = router_weight.shape
    H = down.shape[1]
    if output.dtype not in _DTYPE_CODES or router_weight.dtype not in _DTYPE_CODES:
        raise TypeError("output and router_weight must be bfloat16 or float32")
    args = (_dev(output, "output", output.dtype, (T, H)), _DTYPE_CODES[output.dtype],
            _dev(down, "down", torch.bfloat16, (T * K, H)),
            _dev(restore_order, "restore_order", torch.int32, (T * K,)),
            _dev(router_weight, "router_weight", router_weight.dtype, (T, K)),
            _DTYPE_CODES[router_weight.dtype])
    st = None if device_status is None else _dev(device_status, "device_status", torch.int32, (1,))
    _check("moe_finalize_ex", load_library().moe_finalize_ex(*args, T, K, H, st, _stream(stream)))


def moe_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """The device status word at the start of `workspace` (an index workspace, or
    a status word given to another call); synchronises. Returns the word: 0 is
    clean, otherwise DEVICE_STATUS_* bits."""
    out = ctypes.c_uint32(0)
    rc = load_library().moe_read_device_status(_dev(workspace, "workspace", workspace.dtype),
                                               ctypes.byref(out), _stream(stream))
    if rc != MOE_ERR_DEVICE_DATA:
        _check("moe_read_device_status", rc)
    return int(out.value)


def moe_create_indices_no_alloc(token_expert_order: torch.Tensor,
                                expert_start_indices: torch.Tensor,
                                restore_token_order: torch.Tensor, expert_ids: torch.Tensor,
                                expert_usage_stats: torch.Tensor, topk_ids: torch.Tensor,
                                device_status: torch.Tensor | None = None, stream=None) -> None:
    """moe_create_indices without a workspace, for callers that cannot allocate
    device memory: the library's own static scratch array is used instead
    (see include/moe_routing.h for its size limit and sharing rules).
    device_status, if given, is a 1-element int32 CUDA tensor that receives
    the device status word."""
    f = load_library().moe_create_indices_no_alloc
    N = topk_ids.numel()
    E = expert_ids.numel()
    args = (_dev(token_expert_order, "token_expert_order", torch.int32, (N,)),
            _dev(expert_start_indices, "expert_start_indices", torch.int32, (E + 1,)),
            _dev(restore_token_order, "restore_token_order", torch.int32, (N,)),
            _dev(expert_ids, "expert_ids", torch.int32, (E,)),
            _dev(expert_usage_stats, "expert_usage_stats", torch.int32, (2,)),
            _dev(topk_ids.reshape(-1), "topk_ids", torch.int32))
    status = None if device_status is None else _dev(device_status, "device_status",
                                                     torch.int32, (1,))
    _check("moe_create_indices_no_alloc", f(*args, N, E, status, _stream(stream)))


# ---------------------------------------------------------------- allocating helpers
def route(expert_scores: torch.Tensor, expert_bias: torch.Tensor, n_experts_per_tok: int,
          n_groups: int, topk_group: int, norm_weights: bool, routed_scaling_factor: float,
          stream=None):
    """Returns (expert_indices int32 [T,K], expert_weights fp32 [T,K])."""
    T = expert_scores.shape[0]
    dev = expert_scores.device
    ids = torch.empty((T, n_experts_per_tok), dtype=torch.int32, device=dev)
    w = torch.empty((T, n_experts_per_tok), dtype=torch.float32, device=dev)
    moe_route(ids, w, expert_scores, expert_bias, n_groups, topk_group, norm_weights,
              routed_scaling_factor, stream)
    return ids, w


class IndexBuffers:
    """Preallocated outputs + workspace of moe_create_indices for N slots, E experts."""

    def __init__(self, N: int, E: int, device):
        self.N, self.E = N, E
        z = dict(dtype=torch.int32, device=device)
        self.token_expert_order = torch.empty(N, **z)
        self.expert_start_indices = torch.empty(E + 1, **z)
        self.restore_token_order = torch.empty(N, **z)
        self.expert_ids = torch.empty(E, **z)
        self.expert_usage_stats = torch.empty(2, **z)
        ws = moe_create_indices_workspace_size(N, E)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)

    def run(self, topk_ids: torch.Tensor, stream=None) -> "IndexBuffers":
        moe_create_indices(self.token_expert_order, self.expert_start_indices,
                           self.restore_token_order, self.expert_ids, self.expert_usage_stats,
                           topk_ids, self.workspace, stream)
        return self

    def device_status(self, stream=None) -> int:
        return moe_read_device_status(self.workspace, stream)


class RouteIndexBuffers:
    """Preallocated outputs + zero-filled workspace of moe_route_index (or of
    moe_route_index_single_launch) for T tokens, E experts and K experts per
    token. The index outputs carry the same names as IndexBuffers'."""

    def __init__(self, T: int, E: int, K: int, device, single_launch: bool = False):
        self.single_launch = bool(single_launch)
        self.T, self.E, self.K, self.N = T, E, K, T * K
        z = dict(dtype=torch.int32, device=device)
        self.expert_indices = torch.empty((T, K), **z)
        self.expert_weights = torch.empty((T, K), dtype=torch.float32, device=device)
        self.token_expert_order = torch.empty(T * K, **z)
        self.expert_start_indices = torch.empty(E + 1, **z)
        self.restore_token_order = torch.empty(T * K, **z)
        self.expert_ids = torch.empty(E, **z)
        self.expert_usage_stats = torch.empty(2, **z)
        ws = (moe_route_index_single_launch_workspace_size(T, E) if self.single_launch
              else moe_route_index_workspace_size(T, E, K))
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=device)

    def run(self, expert_scores: torch.Tensor, expert_bias: torch.Tensor, n_groups: int,
            topk_group: int, norm_weights: bool, routed_scaling_factor: float,
            score_fn: int = SCORES_AS_GIVEN, scales_offset: torch.Tensor | None = None,
            stream=None) -> "RouteIndexBuffers":
        moe_route_index(self.expert_indices, self.expert_weights, self.token_expert_order,
                        self.expert_start_indices, self.restore_token_order, self.expert_ids,
                        self.expert_usage_stats, expert_scores, expert_bias, n_groups,
                        topk_group, norm_weights, routed_scaling_factor, self.workspace,
                        score_fn, scales_offset, stream, self.single_launch)
        return self

    def device_status(self, stream=None) -> int:
        return moe_read_device_status(self.workspace, stream)


def route_index(expert_scores: torch.Tensor, expert_bias: torch.Tensor, n_experts_per_tok: int,
                n_groups: int, topk_group: int, norm_weights: bool,
                routed_scaling_factor: float, score_fn: int = SCORES_AS_GIVEN,
                stream=None, single_launch: bool = False) -> RouteIndexBuffers:
    T, E = expert_scores.shape
    bufs = RouteIndexBuffers(T, E, n_experts_per_tok, expert_scores.device, single_launch)
    return bufs.run(expert_scores, expert_bias, n_groups, topk_group, norm_weights,
                    routed_scaling_factor, score_fn, stream=stream)


def create_indices(topk_ids: torch.Tensor, n_experts: int, stream=None) -> IndexBuffers:
    return IndexBuffers(topk_ids.numel(), n_experts, topk_ids.device).run(topk_ids, stream)


def permute(input: torch.Tensor, restore_token_order: torch.Tensor, stream=None) -> torch.Tensor:
    N = restore_token_order.numel()
    out = torch.empty((N, input.shape[1]), dtype=torch.bfloat16, device=input.device)
    moe_permute(out, input, restore_token_order, stream)
    return out


def finalize(down: torch.Tensor, restore_order: torch.Tensor, router_weight: torch.Tensor,
             stream=None) -> torch.Tensor:
    T = router_weight.shape[0]
    out = torch.empty((T, down.shape[1]), dtype=torch.bfloat16, device=down.device)
    moe_finalize(out, down, restore_order, router_weight, stream)
    return out
