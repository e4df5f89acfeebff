"""The routing entry point that allocates nothing (GPU).

pk_moe_route_noalloc serves callers that cannot call cudaMalloc (a program
whose device memory all belongs to its own pool, a plug-in that may not go
around its host runtime's allocator, a latency-critical path that cannot take
cudaMalloc's implicit synchronisation): its counters live in a fixed array
inside the library instead of a caller workspace. Its results must equal, bit
for bit, those of pk_moe_route_counts + pk_moe_build_perm on the same input,
on consecutive calls (the shared array keeps the previous call's contents).
This file is collected last so that a stop at its first failure comes after
every other test has run.
"""
import numpy as np
import pytest
import torch

import inputgen as ig

pytestmark = pytest.mark.gpu


def _routing(T, k, E, zipf, seed):
    return torch.from_numpy(ig.topk_routing(seed, T, E, k, zipf)).cuda()


def _with_workspace(pk, topk, E):
    T, k = topk.shape
    md = pk.MoeDispatch(T, k, E, 8, 8)
    md.route(topk)
    return md


def test_noalloc_routing_equals_workspace_routing_on_consecutive_calls(gpu_lib):
    pk = gpu_lib
    # three calls in a row: a large balanced routing, a smaller skewed one that
    # leaves most of the array's previous contents untouched, then the first
    # routing again
    cases = [(8192, 8, 256, 0.0, 0), (3000, 6, 64, 1.2, 1), (8192, 8, 256, 0.0, 0)]
    for T, k, E, zipf, seed in cases:
        topk = _routing(T, k, E, zipf, seed)
        ref = _with_workspace(pk, topk, E)
        R = T * k
        counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
        offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
        perm = torch.full((R,), -1, dtype=torch.int32, device="cuda")
        inv = torch.full((R,), -1, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        pk.pk_moe_route_noalloc(topk, E, offsets, perm, counts, inv, status)
        torch.cuda.synchronize()
        assert status.item() == 0 and ref.status_code() == 0
        assert torch.equal(counts, ref.counts)
        assert torch.equal(offsets, ref.offsets)
        assert torch.equal(perm, ref.perm[:R])
        assert torch.equal(inv, ref.inv_perm[:R])


def test_noalloc_rejects_sizes_beyond_its_array(gpu_lib):
    pk = gpu_lib
    # ceil(T*k / 2048) * E * 4 bytes must fit in the fixed array
    T, k, E = 1 << 17, 8, 4096
    assert -(-(T * k) // 2048) * E * 4 > pk.PK_NOALLOC_SCRATCH_BYTES
    topk = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    with pytest.raises(pk.PkError) as ei:
        pk.pk_moe_route_noalloc(topk, E, offsets, perm)
    assert ei.value.code == pk.PK_ERR_UNSUPPORTED


def test_noalloc_inside_a_cuda_graph(gpu_lib):
    """After one call outside capture (its context's first, which looks up the
    array's address), the call can be captured in a CUDA graph; replays give
    the workspace routing's results."""
    pk = gpu_lib
    T, k, E = 4096, 8, 128
    topk = _routing(T, k, E, 0.0, 5)
    ref = _with_workspace(pk, topk, E)
    R = T * k
    i32 = dict(dtype=torch.int32, device="cuda")
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    perm, inv, status = torch.empty(R, **i32), torch.empty(R, **i32), torch.zeros(1, **i32)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pk.pk_moe_route_noalloc(topk, E, offsets, perm, counts, inv, status, stream=s)
    torch.cuda.synchronize()
    for t in (counts, offsets, perm, inv):
        t.fill_(-1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pk.pk_moe_route_noalloc(topk, E, offsets, perm, counts, inv, status, stream=s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(counts, ref.counts) and torch.equal(offsets, ref.offsets)
    assert torch.equal(perm, ref.perm[:R]) and torch.equal(inv, ref.inv_perm[:R])


_FIRST_CALL_IN_CAPTURE = r"""
import torch
import inputgen as ig
import moe_token_dispatch_gb300 as pk
T, k, E = 512, 4, 32
R = T * k
topk = torch.from_numpy(ig.topk_routing(3, T, E, k)).cuda()
off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
perm = torch.empty(R, dtype=torch.int32, device="cuda")
s = torch.cuda.Stream()
s.wait_stream(torch.cuda.current_stream())
torch.cuda.synchronize()
code = None
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):
    try:
        pk.pk_moe_route_noalloc(topk, E, off, perm, stream=s)
    except pk.PkError as e:
        code = e.code
assert code == pk.PK_ERR_CAPTURE, code
pk.pk_moe_route_noalloc(topk, E, off, perm)
md = pk.MoeDispatch(T, k, E, 8, 8)
md.route(topk)
torch.cuda.synchronize()
assert torch.equal(off, md.offsets) and torch.equal(perm, md.perm[:R])
print("first call in capture refused, later call ok")
"""


def test_noalloc_first_call_during_capture_is_refused():
    """In a fresh process, a first call made while the stream is captured
    returns PK_ERR_CAPTURE and launches nothing; after the capture the call
    works."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_IN_CAPTURE], cwd=root, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "later call ok" in r.stdout
