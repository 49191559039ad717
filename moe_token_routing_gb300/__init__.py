"""GB300-native (sm_103a) MoE routing and combine hot path.

route (group-limited top-k router) -> create_indices (stable bucket sort by
expert) -> finalize (fused unpermute + weighted top-k sum), each a CUDA
kernel behind the C ABI of libmoe_routing.so (include/moe_routing.h);
route_index runs the first two together (the router counts its own output).
"""
from .binding import (DEVICE_STATUS_BAD_EXPERT_ID, DEVICE_STATUS_BAD_RESTORE_ORDER,
                      DEVICE_STATUS_SYNC_STATE,
                      DEVICE_STATUS_SYNC_TIMEOUT, EXPORTED_SYMBOLS, SCORES_AS_GIVEN,
                      SCORES_SIGMOID, SCORES_SOFTMAX, IndexBuffers, MoeError, MoeLibraryMissing,
                      RouteIndexBuffers, create_indices, finalize, load_library,
                      moe_create_indices, moe_create_indices_no_alloc,
                      moe_create_indices_workspace_size, moe_finalize,
                      moe_finalize_ex, moe_permute, moe_read_device_status, moe_route,
                      moe_route_ex, moe_route_index, moe_route_index_single_launch_workspace_size,
                      moe_route_index_workspace_size, permute,
                      route, route_index)
from .pipeline import HostStreamer, RoutingPipeline

__all__ = [
    "DEVICE_STATUS_BAD_EXPERT_ID", "DEVICE_STATUS_BAD_RESTORE_ORDER", "DEVICE_STATUS_SYNC_STATE",
    "DEVICE_STATUS_SYNC_TIMEOUT",
    "EXPORTED_SYMBOLS", "RouteIndexBuffers", "moe_route_index", "moe_route_index_workspace_size",
    "moe_route_index_single_launch_workspace_size", "route_index", "HostStreamer", "IndexBuffers", "MoeError",
    "MoeLibraryMissing", "RoutingPipeline", "create_indices", "finalize", "load_library",
    "moe_create_indices", "moe_create_indices_no_alloc", "moe_create_indices_workspace_size",
    "moe_finalize",
    "moe_finalize_ex", "moe_permute", "moe_read_device_status", "moe_route", "moe_route_ex",
    "permute", "route", "SCORES_AS_GIVEN", "SCORES_SIGMOID", "SCORES_SOFTMAX",
]
