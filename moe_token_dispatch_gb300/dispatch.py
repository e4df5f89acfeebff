"""Device buffers for one dispatch + expert-GEMM step, and the three calls.

``MoeDispatch`` allocates (through torch, once) the outputs and the routing
workspace for a fixed shape, then issues pk_moe_route_counts ->
pk_moe_build_perm -> pk_moe_dispatch_gemm on one stream. All arithmetic is in
the CUDA library.
"""
from __future__ import annotations

import torch

from . import _binding as B


class MoeDispatch:
    def __init__(self, T: int, k: int, E: int, D: int, De: int, device="cuda",
                 with_inv_perm: bool = True):
        self.T, self.k, self.E, self.D, self.De = T, k, E, D, De
        dev = torch.device(device)
        R = T * k
        i32 = dict(dtype=torch.int32, device=dev)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.perm = torch.empty(max(R, 1), **i32)
        self.inv_perm = torch.empty(max(R, 1), **i32) if with_inv_perm else None
        self.out = torch.empty((max(R, 1), De), dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, **i32)
        nbytes = B.pk_moe_workspace_bytes(T, k, E)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)

    def route(self, topk: torch.Tensor, stream=None) -> None:
        B.pk_moe_route_counts(topk, self.E, self.offsets, self.counts, self.workspace,
                              self.status, stream)
        B.pk_moe_build_perm(topk, self.E, self.offsets, self.perm, self.inv_perm,
                            self.workspace, self.status, stream)

    def gemm(self, x: torch.Tensor, W: torch.Tensor, stream=None) -> None:
        B.pk_moe_dispatch_gemm(x, self.perm, self.offsets, W, self.k, self.out, self.status,
                               stream)

    def __call__(self, x: torch.Tensor, topk: torch.Tensor, W: torch.Tensor, stream=None):
        self.route(topk, stream)
        self.gemm(x, W, stream)
        return self.out[: self.T * self.k]

    def status_code(self) -> int:
        return int(self.status.item())

    def clear_status(self) -> None:
        self.status.zero_()
