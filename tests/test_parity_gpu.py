"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Indices (counts, offsets, perm, inv_perm) must match bit for bit. GEMM
outputs must satisfy |gpu - ref| <= 2e-2 + 1e-2 |ref| element-wise against
the float64 oracle.
"""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from _gpu_util import (assert_gemm_close, bf16_dev_to_f64, boundary_rows, check_case,
                       run_gpu, u16_to_bf16_dev)

pytestmark = pytest.mark.gpu


def _case(T, D, E, k, De, zipf=0.0, seed=0):
    wl = ig.custom(T=T, D=D, E=E, k=k, De=De, zipf_s=zipf, seed=seed)
    c = ig.make_case(wl)
    return c.x, c.topk, c.W


def test_tiny_workload_all_rows(gpu_lib, gemm_kernel):
    wl = ig.WORKLOADS["tiny"]
    c = ig.make_case(wl)
    check_case(gpu_lib, c.x, c.topk, c.W, wl.E)


# Several tiles in every direction and ragged tails, small enough for the
# oracle to do every row: m-tiles per expert 1..6 (two-m-tile units and
# several groups), n-tiles of 256 + a ragged one, K-steps past the 3-stage
# ring, K and N not multiples of 64.
MULTI_TILE = [
    # T,   D,   E, k,  De
    (512, 576, 4, 2, 640),      # ~256 rows/expert, 9 K-steps, N tail 128
    (700, 200, 3, 1, 200),      # D and De not multiples of 64
    (300, 1024, 8, 3, 1408),    # mid-like widths, 16 K-steps
    (1000, 64, 2, 2, 256),      # 1000 rows per expert: 8 m-tiles, 4 groups
    (96, 8, 5, 2, 8),           # smallest legal D and De
    (770, 320, 2, 1, 600),      # 3 and 4 m-tiles: a half-empty CTA pair; De = 512 + 88
]


@pytest.mark.parametrize("T,D,E,k,De", MULTI_TILE)
def test_multi_tile_all_rows(gpu_lib, gemm_kernel, T, D, E, k, De):
    x, topk, W = _case(T, D, E, k, De)
    check_case(gpu_lib, x, topk, W, E)


def test_every_last_m_tile_height(gpu_lib, gemm_kernel):
    """Experts whose last m-tile holds 1..128 rows in every unit shape (a last
    m-tile of at most 64 rows runs as an M = 64 MMA)."""
    from _gpu_util import LAST_TILE_COUNTS, routing_with_counts
    topk = routing_with_counts(LAST_TILE_COUNTS, seed=21)
    E, T = len(LAST_TILE_COUNTS), topk.shape[0]
    x, _, W = _case(T, 320, E, 1, 320, seed=21)
    res, _ = check_case(gpu_lib, x, topk, W, E)
    assert res["counts"].tolist() == LAST_TILE_COUNTS


def test_single_token_single_expert(gpu_lib, gemm_kernel):
    x, topk, W = _case(1, 64, 1, 1, 64)
    check_case(gpu_lib, x, topk, W, 1)


def test_empty_experts_and_one_expert_takes_all(gpu_lib, gemm_kernel):
    T, D, E, k, De = 333, 128, 16, 1, 192
    x, _, W = _case(T, D, E, k, De)
    topk = np.full((T, k), 7, dtype=np.int32)
    res, ref = check_case(gpu_lib, x, topk, W, E)
    assert res["counts"].tolist() == [0] * 7 + [T] + [0] * 8


def test_duplicate_experts_in_one_token(gpu_lib, gemm_kernel):
    T, D, E, k, De = 77, 64, 4, 3, 64
    x, _, W = _case(T, D, E, k, De)
    rng = np.random.default_rng(11)
    topk = rng.integers(0, E, size=(T, k)).astype(np.int32)
    topk[:5] = 2  # all three slots of the first tokens to one expert
    check_case(gpu_lib, x, topk, W, E)


def test_skewed_routing_small(gpu_lib, gemm_kernel):
    x, topk, W = _case(2048, 256, 32, 4, 384, zipf=1.2)
    counts = np.bincount(topk.ravel(), minlength=32)
    assert counts.max() > 4 * counts.mean()
    check_case(gpu_lib, x, topk, W, 32)


@pytest.mark.parametrize("T,k,E", [
    (2048, 8, 4096),    # 8 chunks x 4096 experts: three kernels, chunk rows scanned in place
    (16384, 8, 256),    # 64 chunks: chunk rows staged in 67 KiB of shared memory by the scan
    (32768, 8, 256),    # 128 chunks: 128 KiB of chunk rows, scanned in place
    (512, 8, 4096),     # two chunks x 4096 experts: one-block counts + scan, 64 KiB of shared memory
    (100, 3, 7),        # one ragged chunk
])
def test_routing_kernel_paths(gpu_lib, T, k, E):
    pk = gpu_lib
    rng = np.random.default_rng(T + E)
    topk = rng.integers(0, E, size=(T, k)).astype(np.int32)
    md = pk.MoeDispatch(T, k, E, 64, 64)
    md.route(torch.from_numpy(topk).cuda())
    torch.cuda.synchronize()
    assert md.status_code() == 0
    ref = oracle.run(topk, E)
    R = T * k
    assert np.array_equal(md.counts.cpu().numpy().astype(np.int64), ref["counts"])
    assert np.array_equal(md.offsets.cpu().numpy().astype(np.int64), ref["offsets"])
    assert np.array_equal(md.perm[:R].cpu().numpy().astype(np.int64), ref["perm"])
    assert np.array_equal(md.inv_perm[:R].cpu().numpy().astype(np.int64), ref["inv_perm"])


def test_maximum_expert_count(gpu_lib, gemm_kernel):
    """E = PK_MAX_EXPERTS (4096): three routing kernels, ~4 rows per expert,
    thousands of one-m-tile units, every row of the GEMM checked."""
    pk = gpu_lib
    E = pk.PK_MAX_EXPERTS
    x, topk, W = _case(2048, 64, E, 8, 64, seed=3)
    assert pk.pk_moe_route_kernel_launches(2048, 8, E) == 3
    check_case(pk, x, topk, W, E)


def test_every_token_to_every_expert(gpu_lib, gemm_kernel):
    """k = E: each expert receives all T tokens, in token order."""
    T, D, E, De = 300, 128, 4, 192
    x, _, W = _case(T, D, E, E, De, seed=4)
    topk = np.stack([np.random.default_rng(t).permutation(E) for t in range(T)]).astype(np.int32)
    res, ref = check_case(gpu_lib, x, topk, W, E)
    assert res["counts"].tolist() == [T] * E


def test_nan_input_row_propagates_only_to_its_rows(gpu_lib, gemm_kernel):
    """IEEE propagation, no checks: a NaN in token t's row makes exactly the
    output rows gathered from t NaN; every other row stays finite and within
    tolerance of the oracle."""
    T, D, E, k, De = 200, 256, 8, 2, 256
    x, topk, W = _case(T, D, E, k, De, seed=8)
    bad_t = 17
    x = x.copy()
    x[bad_t, 5] = 0x7FC0  # bf16 quiet NaN
    res = run_gpu(gpu_lib, x, topk, u16_to_bf16_dev(W), E, De)
    assert res["status"] == 0
    out = bf16_dev_to_f64(res["out_dev"])
    from_bad = (res["perm"] // k) == bad_t
    assert from_bad.sum() == k
    assert np.isnan(out[from_bad]).all()
    assert np.isfinite(out[~from_bad]).all()
    ref = oracle.run(topk, E)
    rows = np.flatnonzero(~from_bad)
    want = oracle.gemm_rows(x, ref["perm"], ref["offsets"], W, k, rows)
    assert_gemm_close(out[rows], want, rows)


def test_zero_tokens(gpu_lib):
    pk = gpu_lib
    md = pk.MoeDispatch(0, 2, 8, 64, 64)
    md.offsets.fill_(-7)
    md.counts.fill_(-7)
    tk = torch.zeros((0, 2), dtype=torch.int32, device="cuda")
    md.route(tk)
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((8, 64, 64), dtype=torch.bfloat16, device="cuda")
    md.gemm(x, W)
    torch.cuda.synchronize()
    assert md.offsets.tolist() == [0] * 9 and md.counts.tolist() == [0] * 8


def test_bad_index_sets_status(gpu_lib, gemm_kernel):
    pk = gpu_lib
    T, k, E = 40, 2, 4
    topk = np.random.default_rng(1).integers(0, E, size=(T, k)).astype(np.int32)
    topk[3, 1] = E  # out of range
    topk[9, 0] = -1
    md = pk.MoeDispatch(T, k, E, 64, 64)
    md.route(torch.from_numpy(topk).cuda())
    torch.cuda.synchronize()
    assert md.status_code() == pk.PK_ERR_BAD_INDEX
    # the valid entries are still counted
    valid = topk[(topk >= 0) & (topk < E)]
    assert md.counts.cpu().numpy().tolist() == np.bincount(valid, minlength=E).tolist()


def test_repeat_runs_are_bitwise_identical(gpu_lib, gemm_kernel):
    x, topk, W = _case(512, 576, 4, 2, 640)
    Wd = u16_to_bf16_dev(W)
    a = run_gpu(gpu_lib, x, topk, Wd, 4, 640)
    b = run_gpu(gpu_lib, x, topk, Wd, 4, 640)
    assert torch.equal(a["out_dev"].view(torch.int16), b["out_dev"].view(torch.int16))
    assert np.array_equal(a["perm"], b["perm"])


def test_bounded_wait_times_out_and_context_survives(gpu_lib):
    pk = gpu_lib
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    pk.pk_debug_bounded_wait(st, 50_000_000)  # 50 ms
    t1.record()
    torch.cuda.synchronize()
    assert st.item() == pk.PK_ERR_TIMEOUT
    assert t0.elapsed_time(t1) >= 40.0
    # the context still works
    x, topk, W = _case(64, 64, 2, 1, 64)
    check_case(pk, x, topk, W, 2)


@pytest.mark.parametrize("grouped,big_x", [(False, False), (True, False), (False, True)])
def test_gemm_pipeline_timeout_drains_every_role(gpu_lib, grouped, big_x):
    """A K-step whose copies are never issued (test hook on CTA 0) makes the
    MMA thread's bounded wait run out inside the real pipeline: the launch
    ends by itself with PK_ERR_TIMEOUT, every role has left its loop (the
    producers and dispatch warps are blocked on slots that the stalled K-step
    never frees, so they leave through the abort flag), TMEM was freed, and
    the next launches on the same context run normally. big_x: x of 29 MB,
    more than the 24 MiB up to which the dispatch GEMM runs four W slots, so
    the launch takes the three-W-slot ring split."""
    pk = gpu_lib
    pk.pk_moe_set_gemm_kernel(pk.PK_GEMM_KERNEL_SINGLE)
    # 64 experts x 8 n-tiles of 256 columns, 8 K-steps each: CTA 0 owns several
    # units, so its producers fill the ring past the stalled K-step and block.
    # big_x: 16 experts of 256 rows, 112 K-steps per unit (one unit per CTA).
    T, D, E, k, De = (2048, 7168, 16, 2, 256) if big_x else (256, 512, 64, 2, 2048)
    x, topk, W = _case(T, D, E, k, De)
    Wd = u16_to_bf16_dev(W)
    md = pk.MoeDispatch(T, k, E, D, De)
    xd = u16_to_bf16_dev(x)
    md.route(torch.from_numpy(topk).cuda())
    torch.cuda.synchronize()
    assert md.status_code() == 0
    a_sorted = xd[(md.perm[: T * k] // k).long()].contiguous() if grouped else None
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    pk.pk_moe_set_wait_limit_ns(50_000_000)  # 50 ms
    pk.pk_debug_stall_gemm(0, 2)
    try:
        t0.record()
        if grouped:
            pk.pk_moe_grouped_gemm(a_sorted, md.offsets, Wd, md.out, md.status)
        else:
            md.gemm(xd, Wd)
        t1.record()
        torch.cuda.synchronize()
    finally:
        pk.pk_debug_stall_gemm(-1, -1)
        pk.pk_moe_set_wait_limit_ns(0)   # back to the default limit
        pk.pk_moe_set_gemm_kernel(pk.PK_GEMM_KERNEL_AUTO)
    assert md.status_code() == pk.PK_ERR_TIMEOUT
    ms = t0.elapsed_time(t1)
    assert 40.0 <= ms < 1000.0, ms
    # the same context runs the path again, and the same launch is correct
    md.clear_status()
    check_case(pk, x, topk, W, E, rows=boundary_rows(oracle.route_counts(topk, E)[1],
                                                       np.random.default_rng(2), 64),
               W_dev=Wd)
    xs, tks, Ws = _case(64, 64, 2, 1, 64)
    check_case(pk, xs, tks, Ws, 2)


# ------------------------------------------------- the five named workloads
def test_mid_workload(gpu_lib, gemm_kernel):
    wl = ig.WORKLOADS["mid"]
    c = ig.make_case(wl)
    rows = boundary_rows(oracle.route_counts(c.topk, wl.E)[1], np.random.default_rng(0), 256)
    check_case(gpu_lib, c.x, c.topk, c.W, wl.E, rows=rows)


@pytest.fixture(scope="module")
def big_W():
    """W for D=7168, E=256, D_expert=2048 (7.5 GB), shared by the three
    full-size workloads, which use the same seed and shape."""
    wl = ig.WORKLOADS["ep"]
    W = ig.make_W(wl)
    Wd = u16_to_bf16_dev(W)
    yield W, Wd
    del Wd
    torch.cuda.empty_cache()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["ep", "skew", "decode"])
def test_full_size_workloads(gpu_lib, big_W, name):
    wl = ig.WORKLOADS[name]
    W, Wd = big_W
    x = ig.make_x(wl)
    topk = ig.make_topk(wl)
    offsets = oracle.route_counts(topk, wl.E)[1]
    rows = boundary_rows(offsets, np.random.default_rng(1), 128)
    res, ref = check_case(gpu_lib, x, topk, W, wl.E, rows=rows, W_dev=Wd)
    out = res["out_dev"]
    # every row of the output, not only the sampled ones, is finite
    assert bool(torch.isfinite(out.float()).all())
    if name == "skew":
        counts = ref["counts"]
        assert (counts == 0).sum() > 20 and counts.max() > 2000
