"""The path inside a CUDA graph: route + GEMM captured once on a side stream
and replayed reproduce the eager results bit for bit (the calls do no host
synchronisation and allocate nothing)."""
import numpy as np
import pytest
import torch

import inputgen as ig
from _gpu_util import u16_to_bf16_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,D,E,k,De", [(512, 576, 8, 2, 640), (96, 64, 300, 4, 64)])
def test_graph_replay_matches_eager(gpu_lib, T, D, E, k, De):
    pk = gpu_lib
    c = ig.make_case(ig.custom(T=T, D=D, E=E, k=k, De=De, seed=12))
    x, W = u16_to_bf16_dev(c.x), u16_to_bf16_dev(c.W)
    tk = torch.from_numpy(c.topk).cuda()
    eager = pk.MoeDispatch(T, k, E, D, De)
    eager(x, tk, W)
    torch.cuda.synchronize()

    md = pk.MoeDispatch(T, k, E, D, De)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        md.route(tk, s)          # warm-up outside the capture (first-call setup)
        md.gemm(x, W, s)
    torch.cuda.synchronize()
    md.out.zero_()
    md.perm.fill_(-1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        md.route(tk, s)
        md.gemm(x, W, s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert md.status_code() == 0
    R = T * k
    assert torch.equal(md.perm[:R], eager.perm[:R])
    assert torch.equal(md.offsets, eager.offsets)
    assert torch.equal(md.out[:R].view(torch.int16), eager.out[:R].view(torch.int16))
