"""Host-to-host pipelined dispatch + expert GEMM.

``PipelinedDispatch`` runs a stream of batches whose inputs (x, topk_idx) live
in pinned host memory and whose output must come back to host memory. Each
batch goes through three CUDA streams:

  copy-in   x and topk_idx host -> device buffer b
  compute   pk_moe_route_counts -> pk_moe_build_perm -> pk_moe_dispatch_gemm on b
  copy-out  out of b -> pinned host buffer

with two buffer sets (b alternates), so batch i+1 is copied in and batch i-1
copied out while batch i computes. Events order the streams: a buffer set is
refilled only after the compute that read it finished, and its output is
overwritten only after the copy-out of the previous batch on it finished.
The arithmetic is all in the CUDA library; this is stream and buffer
plumbing.
"""
from __future__ import annotations

import torch

from .dispatch import MoeDispatch


class PipelinedDispatch:
    def __init__(self, T: int, k: int, E: int, D: int, De: int, W: torch.Tensor,
                 device=None, depth: int = 2):
        self.dev = torch.device(device) if device is not None else W.device
        self.T, self.k, self.E, self.D, self.De = T, k, E, D, De
        self.W = W
        self.depth = depth
        R = T * k
        self.sets = []
        for _ in range(depth):
            md = MoeDispatch(T, k, E, D, De, device=self.dev)
            x = torch.empty((T, D), dtype=torch.bfloat16, device=self.dev)
            tk = torch.empty((T, k), dtype=torch.int32, device=self.dev)
            out_h = torch.empty((R, De), dtype=torch.bfloat16).pin_memory()
            self.sets.append({"md": md, "x": x, "tk": tk, "out_h": out_h,
                              "in_done": torch.cuda.Event(), "comp_done": torch.cuda.Event(),
                              "out_done": torch.cuda.Event(), "used": False})
        with torch.cuda.device(self.dev):
            self.s_in = torch.cuda.Stream()
            self.s_comp = torch.cuda.Stream()
            self.s_out = torch.cuda.Stream()

    def submit(self, i: int, x_h: torch.Tensor, tk_h: torch.Tensor) -> dict:
        """Enqueues batch i (pinned host tensors); returns its buffer set, whose
        ``out_h`` holds the result once ``out_done`` has completed."""
        b = self.sets[i % self.depth]
        R = self.T * self.k
        if b["used"]:
            self.s_in.wait_event(b["comp_done"])   # inputs of the previous batch on b consumed
        with torch.cuda.stream(self.s_in):
            b["x"].copy_(x_h, non_blocking=True)
            b["tk"].copy_(tk_h, non_blocking=True)
            b["in_done"].record(self.s_in)
        self.s_comp.wait_event(b["in_done"])
        if b["used"]:
            self.s_comp.wait_event(b["out_done"])  # previous output of b copied out
        b["md"].route(b["tk"], self.s_comp)
        b["md"].gemm(b["x"], self.W, self.s_comp)
        b["comp_done"].record(self.s_comp)
        self.s_out.wait_event(b["comp_done"])
        with torch.cuda.stream(self.s_out):
            b["out_h"].copy_(b["md"].out[:R], non_blocking=True)
            b["out_done"].record(self.s_out)
        b["used"] = True
        return b

    def synchronize(self) -> None:
        for s in (self.s_in, self.s_comp, self.s_out):
            s.synchronize()

    def status_codes(self) -> list:
        return [b["md"].status_code() for b in self.sets]
