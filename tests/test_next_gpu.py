"""GPU parity of the router top-k and combine kernels against the oracle."""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from _gpu_util import bf16_dev_to_f64, u16_to_bf16_dev

pytestmark = pytest.mark.gpu


def _router_gpu(pk, logits, k):
    T, E = logits.shape
    l = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    g = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    pk.pk_moe_router_topk(l, k, idx, g)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), g.cpu().numpy()


def _check_router(pk, logits, k):
    idx, g = _router_gpu(pk, logits, k)
    ridx, rg = oracle.router_topk(logits, k)
    assert np.array_equal(idx.astype(np.int64), ridx)
    assert np.all(np.abs(g - rg) <= 1e-6 + 1e-5 * rg)


@pytest.mark.parametrize("name", ["tiny", "mid", "ep", "skew", "decode"])
def test_router_on_workloads(gpu_lib, name):
    wl = ig.WORKLOADS[name]
    logits = ig.make_logits(wl)
    _check_router(gpu_lib, logits, wl.k)
    # the float32 logits select the same experts as the generator's float64 ones
    if name in ("tiny", "mid"):
        idx, _ = _router_gpu(gpu_lib, logits, wl.k)
        assert np.array_equal(idx, ig.make_topk(wl))


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (33, 100, 1), (70, 1024, 32), (257, 37, 7)])
def test_router_shapes(gpu_lib, T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    _check_router(gpu_lib, rng.standard_normal((T, E)).astype(np.float32), k)


def test_router_ties_and_infinities(gpu_lib):
    rng = np.random.default_rng(5)
    l = rng.integers(-2, 3, size=(200, 64)).astype(np.float32)   # many equal logits
    l[::7, ::3] = -np.inf
    _check_router(gpu_lib, l, 8)
    # signed zeros compare equal: -0 and +0 logits tie and go to the lower expert
    z = np.zeros((50, 40), dtype=np.float32)
    z[rng.random(z.shape) < 0.5] = -0.0
    z[::5, 7] = 1.0
    _check_router(gpu_lib, z, 5)


def _combine_gpu(pk, src, inv, gates, T, k):
    C = src.shape[1]
    s = u16_to_bf16_dev(src)
    i = torch.from_numpy(np.ascontiguousarray(inv, dtype=np.int32)).cuda()
    g = None if gates is None else torch.from_numpy(np.ascontiguousarray(gates, dtype=np.float32)).cuda()
    y = torch.zeros((T, C), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.pk_moe_combine(s, i, g, T, k, y, st)
    torch.cuda.synchronize()
    return bf16_dev_to_f64(y), int(st.item())


def _check_combine(pk, wl, C):
    topk = ig.make_topk(wl)
    _, offsets = oracle.route_counts(topk, wl.E)
    _, inv = oracle.build_perm(topk, wl.E, offsets)
    src = ig.make_src(wl, C)
    gates = ig.make_gates(wl)
    got, st = _combine_gpu(pk, src, inv, gates, wl.T, wl.k)
    assert st == 0
    ref = oracle.combine(src, inv, gates.astype(np.float64), wl.T, wl.k)
    # sum of |gate * src| per element: the same combine on |src| (sign bit cleared)
    absum = oracle.combine(src & np.uint16(0x7FFF), inv, np.abs(gates).astype(np.float64),
                           wl.T, wl.k)
    # bf16 rounding of the result plus fp32 summation of k products
    bound = 2.0 ** -8 * np.abs(ref) + 1e-6 + 1e-6 * np.abs(absum)
    assert np.all(np.abs(got - ref) <= bound)


@pytest.mark.parametrize("name,C", [("tiny", 128), ("mid", 1408), ("decode", 2048),
                                    ("ep", 2048)])
def test_combine_on_workloads(gpu_lib, name, C):
    _check_combine(gpu_lib, ig.WORKLOADS[name], C)


@pytest.mark.parametrize("T,k,E,C", [(1, 1, 1, 8), (37, 3, 5, 264), (300, 8, 16, 7168)])
def test_combine_shapes(gpu_lib, T, k, E, C):
    _check_combine(gpu_lib, ig.custom(T=T, D=8, E=E, k=k, De=8, seed=T), C)


def test_combine_unit_gates_undo_dispatch(gpu_lib):
    # k = 1, no gates: combine(rows dispatched in sorted order) == x
    wl = ig.custom(T=500, D=256, E=7, k=1, De=8)
    x = ig.make_x(wl)
    topk = ig.make_topk(wl)
    _, offsets = oracle.route_counts(topk, wl.E)
    perm, inv = oracle.build_perm(topk, wl.E, offsets)
    got, st = _combine_gpu(gpu_lib, x[perm], inv, None, wl.T, 1)
    assert st == 0 and np.array_equal(got, ig.bf16_bits_to_f64(x))


def test_combine_bad_index_sets_status(gpu_lib):
    T, k, C = 20, 2, 64
    src = ig.normal_bf16(0, 9, 0, T * k * C).reshape(T * k, C)
    inv = np.arange(T * k)
    inv[5] = T * k + 3
    _, st = _combine_gpu(gpu_lib, src, inv, np.ones((T, k), np.float32), T, k)
    assert st == gpu_lib.PK_ERR_BAD_INDEX


# ------------------------------------------------ grouped (down-projection) GEMM
def _grouped_case(R_T, K, E, k, N, seed=0, zipf=0.0):
    """Rows of A in expert order from a routing, and W2 [E, K, N]."""
    wl = ig.custom(T=R_T, D=K, E=E, k=k, De=N, zipf_s=zipf, seed=seed)
    topk = ig.make_topk(wl)
    counts, offsets = oracle.route_counts(topk, E)
    R = R_T * k
    A = ig.normal_bf16(seed, 7, 0, R * K).reshape(R, K)
    W = ig.make_W(wl)
    return A, offsets, W


def _check_grouped(pk, A, offsets, W, rows=None):
    from _gpu_util import assert_gemm_close
    R, K = A.shape
    E, _, N = W.shape
    Ad, Wd = u16_to_bf16_dev(A), u16_to_bf16_dev(W)
    off = torch.from_numpy(offsets.astype(np.int32)).cuda()
    out = torch.zeros((R, N), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.pk_moe_grouped_gemm(Ad, off, Wd, out, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    if rows is None:
        rows = np.arange(R)
    # rows already in expert order: the oracle's GEMM with the identity permutation, k = 1
    ref = oracle.gemm_rows(A, np.arange(R), offsets, W, 1, rows)
    got = bf16_dev_to_f64(out[torch.from_numpy(rows).cuda()])
    assert_gemm_close(got, ref, rows)


@pytest.mark.parametrize("T,K,E,k,N", [(512, 576, 4, 2, 640), (700, 200, 3, 1, 200),
                                       (300, 2048, 8, 3, 1408), (96, 8, 5, 2, 8),
                                       (1000, 64, 2, 2, 256)])
def test_grouped_gemm_all_rows(gpu_lib, T, K, E, k, N):
    A, offsets, W = _grouped_case(T, K, E, k, N)
    _check_grouped(gpu_lib, A, offsets, W)


def test_grouped_gemm_every_last_m_tile_height(gpu_lib):
    from _gpu_util import LAST_TILE_COUNTS, routing_with_counts
    topk = routing_with_counts(LAST_TILE_COUNTS, seed=24)
    E, R = len(LAST_TILE_COUNTS), topk.shape[0]
    _, offsets = oracle.route_counts(topk, E)
    A = ig.normal_bf16(24, 7, 0, R * 256).reshape(R, 256)
    W = ig.make_W(ig.custom(T=R, D=256, E=E, k=1, De=200, seed=24))
    _check_grouped(gpu_lib, A, offsets, W)


def test_grouped_gemm_down_projection_shape(gpu_lib):
    # the ep down-projection: K = D_expert = 2048, N = D = 7168, 256 experts
    from _gpu_util import boundary_rows
    A, offsets, W = _grouped_case(8192, 2048, 256, 8, 7168)
    rows = boundary_rows(offsets, np.random.default_rng(3), 128)
    _check_grouped(gpu_lib, A, offsets, W, rows)


def test_grouped_gemm_skewed(gpu_lib):
    A, offsets, W = _grouped_case(2048, 256, 32, 4, 384, zipf=1.2)
    _check_grouped(gpu_lib, A, offsets, W)
