"""Routing calls issued back to back on one stream (GPU).

The routing kernels are launched with programmatic stream serialisation: a
kernel's blocks may be scheduled while the kernel ahead of it is still
running, and each waits for that kernel to complete before its first access
to global memory. These tests issue many routing calls with no
synchronisation between them -- calls sharing one counter array, calls whose
routing array a plain kernel writes just before, calls whose results the next
kernel copies away -- and check every call's result against the oracle.
"""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle

pytestmark = pytest.mark.gpu


def _check(ref, counts, offsets, perm, inv):
    assert np.array_equal(counts.cpu().numpy().astype(np.int64), ref["counts"])
    assert np.array_equal(offsets.cpu().numpy().astype(np.int64), ref["offsets"])
    assert np.array_equal(perm.cpu().numpy().astype(np.int64), ref["perm"])
    assert np.array_equal(inv.cpu().numpy().astype(np.int64), ref["inv_perm"])


@pytest.mark.parametrize("T,k,E", [
    (4096, 8, 256),   # three kernels: histogram, scan (rows staged), permutation
    (256, 8, 256),    # two kernels: one-block counts + scan, permutation
])
def test_back_to_back_calls_on_separate_buffers(gpu_lib, T, k, E):
    pk = gpu_lib
    n = 8
    topks = [torch.from_numpy(ig.topk_routing(100 + i, T, E, k, 1.2 * (i % 2))).cuda()
             for i in range(n)]
    mds = [pk.MoeDispatch(T, k, E, 8, 8) for _ in range(n)]
    torch.cuda.synchronize()
    for md, tk in zip(mds, topks):
        md.route(tk)
    torch.cuda.synchronize()
    R = T * k
    for md, tk in zip(mds, topks):
        assert md.status_code() == 0
        _check(oracle.run(tk.cpu().numpy(), E), md.counts, md.offsets, md.perm[:R],
               md.inv_perm[:R])


def test_back_to_back_calls_sharing_one_workspace(gpu_lib):
    """Each call's histogram kernel rewrites the chunk rows that the previous
    call's permutation kernel reads: it must wait for that kernel to finish."""
    pk = gpu_lib
    T, k, E = 8192, 8, 256
    n = 6
    R = T * k
    topks = [torch.from_numpy(ig.topk_routing(200 + i, T, E, k, 0.6 * (i % 3))).cuda()
             for i in range(n)]
    md = pk.MoeDispatch(T, k, E, 8, 8)
    i32 = dict(dtype=torch.int32, device="cuda")
    outs = [(torch.full((E,), -1, **i32), torch.full((E + 1,), -1, **i32),
             torch.full((R,), -1, **i32), torch.full((R,), -1, **i32)) for _ in range(n)]
    torch.cuda.synchronize()
    for tk, (counts, offsets, perm, inv) in zip(topks, outs):
        pk.pk_moe_route_counts(tk, E, offsets, counts, md.workspace, md.status)
        pk.pk_moe_build_perm(tk, E, offsets, perm, inv, md.workspace, md.status)
    torch.cuda.synchronize()
    assert md.status_code() == 0
    for tk, (counts, offsets, perm, inv) in zip(topks, outs):
        _check(oracle.run(tk.cpu().numpy(), E), counts, offsets, perm, inv)


def test_noalloc_back_to_back_calls(gpu_lib):
    """The allocation-free entry point shares one counter array across calls."""
    pk = gpu_lib
    cases = [(8192, 8, 256, 0.0), (3000, 6, 64, 1.2), (128, 8, 256, 0.0), (8192, 8, 256, 1.2)]
    i32 = dict(dtype=torch.int32, device="cuda")
    runs = []
    for i, (T, k, E, z) in enumerate(cases):
        tk = torch.from_numpy(ig.topk_routing(300 + i, T, E, k, z)).cuda()
        R = T * k
        runs.append((tk, E, torch.full((E,), -1, **i32), torch.full((E + 1,), -1, **i32),
                     torch.full((R,), -1, **i32), torch.full((R,), -1, **i32)))
    status = torch.zeros(1, **i32)
    torch.cuda.synchronize()
    for tk, E, counts, offsets, perm, inv in runs:
        pk.pk_moe_route_noalloc(tk, E, offsets, perm, counts, inv, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for tk, E, counts, offsets, perm, inv in runs:
        _check(oracle.run(tk.cpu().numpy(), E), counts, offsets, perm, inv)


def test_routing_array_written_just_before_each_call(gpu_lib):
    """A plain kernel writes the routing array right before each call and
    another copies the results away right after; the next call reuses every
    buffer."""
    pk = gpu_lib
    T, k, E = 4096, 6, 64
    n = 10
    R = T * k
    src = torch.from_numpy(np.stack([ig.topk_routing(400 + i, T, E, k, 0.0)
                                     for i in range(n)])).cuda()
    md = pk.MoeDispatch(T, k, E, 8, 8)
    topk = torch.empty((T, k), dtype=torch.int32, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    perms, invs = torch.empty((n, R), **i32), torch.empty((n, R), **i32)
    offs, cnts = torch.empty((n, E + 1), **i32), torch.empty((n, E), **i32)
    torch.cuda.synchronize()
    for i in range(n):
        topk.copy_(src[i])
        md.route(topk)
        perms[i].copy_(md.perm[:R])
        invs[i].copy_(md.inv_perm[:R])
        offs[i].copy_(md.offsets)
        cnts[i].copy_(md.counts)
    torch.cuda.synchronize()
    assert md.status_code() == 0
    for i in range(n):
        _check(oracle.run(src[i].cpu().numpy(), E), cnts[i], offs[i], perms[i], invs[i])
