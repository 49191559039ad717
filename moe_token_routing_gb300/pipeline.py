"""route -> create_indices -> finalize on one stream, with preallocated buffers.

A RoutingPipeline is sized for one workload shape (T tokens, E experts in
n_groups groups, K experts per token, hidden size H). ``__call__`` runs the
three stages on device-resident inputs; ``run_host`` is the end-to-end call
on host (pinned) buffers: it enqueues the host-to-device copies, the three
kernels and the device-to-host copy of the combined output on one stream.

Between route and finalize sits the expert computation (a grouped matmul over
``index.token_expert_order``), which is not part of this path: ``down`` is
taken as given, already in token_expert_order row order.
"""
from __future__ import annotations

import torch

from .binding import (IndexBuffers, moe_finalize, moe_permute, moe_read_device_status,
                      moe_route, moe_route_index,
                      moe_route_index_workspace_size)


class RoutingPipeline:
    """``fused=True`` (the default) builds the indices with moe_route_index,
    whose router counts its own output, so route and create_indices take three
    launches instead of four; ``fused=False`` calls moe_route and then
    moe_create_indices. The outputs are the same bits either way."""

    def __init__(self, T: int, E: int, K: int, H: int, n_groups: int, topk_group: int,
                 norm_weights: bool, routed_scaling_factor: float, device="cuda",
                 fused: bool = True):
        self.T, self.E, self.K, self.H = T, E, K, H
        self.n_groups, self.topk_group = n_groups, topk_group
        self.norm_weights, self.scale = bool(norm_weights), float(routed_scaling_factor)
        self.device = torch.device(device)
        self.fused = bool(fused)
        self.expert_indices = torch.empty((T, K), dtype=torch.int32, device=self.device)
        self.expert_weights = torch.empty((T, K), dtype=torch.float32, device=self.device)
        self.index = IndexBuffers(T * K, E, self.device)
        self.fused_workspace = None
        if self.fused:
            self.fused_workspace = torch.zeros(moe_route_index_workspace_size(T, E, K),
                                               dtype=torch.uint8, device=self.device)
        self.output = torch.empty((T, H), dtype=torch.bfloat16, device=self.device)
        self._staged = None

    def route(self, expert_scores, expert_bias, stream=None):
        moe_route(self.expert_indices, self.expert_weights, expert_scores, expert_bias,
                  self.n_groups, self.topk_group, self.norm_weights, self.scale, stream)

    def create_indices(self, stream=None):
        self.index.run(self.expert_indices, stream)

    def route_index(self, expert_scores, expert_bias, stream=None):
        """route + create_indices through moe_route_index (needs ``fused=True``)."""
        if self.fused_workspace is None:
            raise RuntimeError("RoutingPipeline was built with fused=False")
        ix = self.index
        moe_route_index(self.expert_indices, self.expert_weights, ix.token_expert_order,
                        ix.expert_start_indices, ix.restore_token_order, ix.expert_ids,
                        ix.expert_usage_stats, expert_scores, expert_bias, self.n_groups,
                        self.topk_group, self.norm_weights, self.scale, self.fused_workspace,
                        stream=stream)

    def route_and_index(self, expert_scores, expert_bias, stream=None):
        if self.fused:
            self.route_index(expert_scores, expert_bias, stream)
        else:
            self.route(expert_scores, expert_bias, stream)
            self.create_indices(stream)

    def device_status(self, stream=None) -> int:
        """Device status word of the last index build (0 = clean)."""
        ws = self.fused_workspace if self.fused else self.index.workspace
        return moe_read_device_status(ws, stream)

    def finalize(self, down, stream=None, output=None):
        moe_finalize(self.output if output is None else output, down,
                     self.index.restore_token_order, self.expert_weights, stream)

    def permute(self, x, out, stream=None):
        """Expert-contiguous token rows for the grouped matmul (after create_indices)."""
        moe_permute(out, x, self.index.restore_token_order, stream)
        return out

    def __call__(self, expert_scores, expert_bias, down, stream=None) -> torch.Tensor:
        self.route_and_index(expert_scores, expert_bias, stream)
        self.finalize(down, stream)
        return self.output

    def _staging(self):
        if self._staged is None:
            d = self.device
            self._staged = (torch.empty((self.T, self.E), dtype=torch.float32, device=d),
                            torch.empty((self.E,), dtype=torch.float32, device=d),
                            torch.empty((self.T * self.K, self.H), dtype=torch.bfloat16, device=d))
        return self._staged

    def run_host(self, scores_h: torch.Tensor, bias_h: torch.Tensor, down_h: torch.Tensor,
                 out_h: torch.Tensor, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
        """Copy host inputs in, run the three stages, copy the output back into out_h.

        Asynchronous on ``stream`` (pinned host buffers make the copies truly
        asynchronous); synchronise the stream before reading out_h."""
        stream = stream or torch.cuda.current_stream(self.device)
        scores_d, bias_d, down_d = self._staging()
        with torch.cuda.stream(stream):
            scores_d.copy_(scores_h, non_blocking=True)
            bias_d.copy_(bias_h, non_blocking=True)
            down_d.copy_(down_h, non_blocking=True)
            self(scores_d, bias_d, down_d, stream)
            out_h.copy_(self.output, non_blocking=True)
        return out_h

    def stream_from_host(self, depth: int = 2) -> "HostStreamer":
        """A double-buffered host-buffer runner over this pipeline (see HostStreamer)."""
        return HostStreamer(self, depth)

    def host_bytes(self) -> tuple[int, int]:
        """(host-to-device, device-to-host) bytes that run_host moves per call."""
        h2d = self.T * self.E * 4 + self.E * 4 + self.T * self.K * self.H * 2
        return h2d, self.T * self.H * 2


class HostStreamer:
    """Runs a sequence of batches from host (pinned) buffers through a
    RoutingPipeline with the copies overlapped: while batch i computes and
    its output is copied back, batch i+1's inputs are already being copied in.

    Three CUDA streams (copy-in, compute, copy-out) and ``depth`` sets of
    device staging and output buffers; events order each batch's copy-in ->
    compute -> copy-out and keep a staging set from being overwritten before
    the compute that reads it is done. ``submit`` only enqueues; call
    ``synchronize`` before reading the host outputs.
    """

    def __init__(self, pipe: RoutingPipeline, depth: int = 2):
        self.pipe = pipe
        self.depth = depth
        d = pipe.device
        self.copy_in = torch.cuda.Stream(d)
        self.compute = torch.cuda.Stream(d)
        self.copy_out = torch.cuda.Stream(d)
        T, E, K, H = pipe.T, pipe.E, pipe.K, pipe.H
        self.slots = []
        for _ in range(depth):
            self.slots.append({
                "scores": torch.empty((T, E), dtype=torch.float32, device=d),
                "bias": torch.empty((E,), dtype=torch.float32, device=d),
                "down": torch.empty((T * K, H), dtype=torch.bfloat16, device=d),
                "out": torch.empty((T, H), dtype=torch.bfloat16, device=d),
                "copied_in": torch.cuda.Event(), "computed": torch.cuda.Event(),
                "copied_out": torch.cuda.Event(), "used": False,
            })
        self.count = 0

    def submit(self, scores_h: torch.Tensor, bias_h: torch.Tensor, down_h: torch.Tensor,
               out_h: torch.Tensor) -> None:
        slot = self.slots[self.count % self.depth]
        if slot["used"]:
            self.copy_in.wait_event(slot["computed"])     # staging no longer read
            self.compute.wait_event(slot["copied_out"])   # output no longer read
        with torch.cuda.stream(self.copy_in):
            slot["scores"].copy_(scores_h, non_blocking=True)
            slot["bias"].copy_(bias_h, non_blocking=True)
            slot["down"].copy_(down_h, non_blocking=True)
            slot["copied_in"].record(self.copy_in)
        self.compute.wait_event(slot["copied_in"])
        self.pipe.route_and_index(slot["scores"], slot["bias"], self.compute)
        self.pipe.finalize(slot["down"], self.compute, output=slot["out"])
        slot["computed"].record(self.compute)
        self.copy_out.wait_event(slot["computed"])
        with torch.cuda.stream(self.copy_out):
            out_h.copy_(slot["out"], non_blocking=True)
            slot["copied_out"].record(self.copy_out)
        slot["used"] = True
        self.count += 1

    def synchronize(self) -> None:
        self.copy_out.synchronize()
        self.compute.synchronize()
        self.copy_in.synchronize()
