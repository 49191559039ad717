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

from .binding import IndexBuffers, moe_finalize, moe_route


class RoutingPipeline:
    def __init__(self, T: int, E: int, K: int, H: int, n_groups: int, topk_group: int,
                 norm_weights: bool, routed_scaling_factor: float, device="cuda"):
        self.T, self.E, self.K, self.H = T, E, K, H
        self.n_groups, self.topk_group = n_groups, topk_group
        self.norm_weights, self.scale = bool(norm_weights), float(routed_scaling_factor)
        self.device = torch.device(device)
        self.expert_indices = torch.empty((T, K), dtype=torch.int32, device=self.device)
        self.expert_weights = torch.empty((T, K), dtype=torch.float32, device=self.device)
        self.index = IndexBuffers(T * K, E, self.device)
        self.output = torch.empty((T, H), dtype=torch.bfloat16, device=self.device)
        self._staged = None

    def route(self, expert_scores, expert_bias, stream=None):
        moe_route(self.expert_indices, self.expert_weights, expert_scores, expert_bias,
                  self.n_groups, self.topk_group, self.norm_weights, self.scale, stream)

    def create_indices(self, stream=None):
        self.index.run(self.expert_indices, stream)

    def finalize(self, down, stream=None):
        moe_finalize(self.output, down, self.index.restore_token_order, self.expert_weights,
                     stream)

    def __call__(self, expert_scores, expert_bias, down, stream=None) -> torch.Tensor:
        self.route(expert_scores, expert_bias, stream)
        self.create_indices(stream)
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

    def host_bytes(self) -> tuple[int, int]:
        """(host-to-device, device-to-host) bytes that run_host moves per call."""
        h2d = self.T * self.E * 4 + self.E * 4 + self.T * self.K * self.H * 2
        return h2d, self.T * self.H * 2
