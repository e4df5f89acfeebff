"""Host-to-host pipelined runs (GPU): each batch's output equals the plain
three-call path's output on the same batch, bit for bit."""
import numpy as np
import pytest
import torch

import inputgen as ig

pytestmark = pytest.mark.gpu


def test_pipelined_batches_match_plain_path(gpu_lib):
    pk = gpu_lib
    from moe_token_dispatch_gb300.pipeline import PipelinedDispatch
    T, D, E, k, De = 300, 256, 8, 2, 384
    W_u16 = ig.make_W(ig.custom(T=T, D=D, E=E, k=k, De=De))
    W = torch.from_numpy(W_u16.view(np.int16)).cuda().view(torch.bfloat16)
    pipe = PipelinedDispatch(T, k, E, D, De, W)
    batches, outs = [], []
    for i in range(5):   # different inputs per batch, more batches than buffer sets
        wl = ig.custom(T=T, D=D, E=E, k=k, De=De, seed=100 + i)
        x = torch.from_numpy(ig.make_x(wl).view(np.int16)).view(torch.bfloat16).pin_memory()
        tk = torch.from_numpy(ig.make_topk(wl)).pin_memory()
        batches.append((x, tk))
        b = pipe.submit(i, x, tk)
        b["out_done"].synchronize()
        outs.append(b["out_h"].clone())
    pipe.synchronize()
    assert pipe.status_codes() == [0, 0]
    for (x, tk), got in zip(batches, outs):
        md = pk.MoeDispatch(T, k, E, D, De)
        ref = md(x.cuda(), tk.cuda(), W)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.cpu().view(torch.int16))
