"""GPU parity of the FP8 variant: E4M3 quantisation and the FP8 dispatch GEMM.

Quantisation codes and scales must match the oracle bit for bit (both sides
take every decision in IEEE fp32). The GEMM is checked on the oracle's own
codes and scales: |gpu - ref| <= 2e-2 + 1e-2 |ref| element-wise against the
float64 sum of dequantised products, i.e. the same bound as the bf16 path,
since both sides read identical 8-bit inputs and differ only by the fp32
accumulation order and the final bf16 rounding.
"""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from _gpu_util import (assert_gemm_close, bf16_dev_to_f64, boundary_rows, to_blocked,
                       u16_to_bf16_dev)

pytestmark = pytest.mark.gpu


def _u8_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def _gpu_quant_rows(pk, x_u16):
    T, D = x_u16.shape
    xq = torch.empty((T, D), dtype=torch.uint8, device="cuda")
    sx = torch.empty((T,), dtype=torch.float32, device="cuda")
    pk.pk_moe_quant_rows(u16_to_bf16_dev(x_u16), xq, sx)
    torch.cuda.synchronize()
    return xq, sx


def _gpu_quant_weights(pk, W_dev):
    """Blocked codes, viewed as [E, ceil(N/64), ceil(D/128), 64, 128]."""
    E, D, N = W_dev.shape
    wq = torch.full((E, -(-N // 64), -(-D // 128), 64, 128), 0x55, dtype=torch.uint8,
                    device="cuda")  # padding must come back zero
    sw = torch.empty((E, N), dtype=torch.float32, device="cuda")
    pk.pk_moe_quant_weights(W_dev, wq, sw)
    torch.cuda.synchronize()
    return wq, sw


def _awkward_bf16(rng, shape):
    """bf16 bits with zeros, subnormals, huge and tiny magnitudes and exact
    powers of two mixed into normal values."""
    v = rng.standard_normal(shape).astype(np.float32)
    v[..., ::7] *= np.float32(1e-30)
    v[..., 3::11] *= np.float32(1e30)
    v[..., 5::13] = np.float32(2.0) ** rng.integers(-20, 20, size=v[..., 5::13].shape)
    bits = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    return bits


@pytest.mark.parametrize("D", [7168 + 8, 8192 + 8, 64])  # block-per-row kernel, two-pass kernel, tiny
def test_quant_rows_bit_exact(gpu_lib, D):
    rng = np.random.default_rng(3)
    T = 301
    x = ig.normal_bf16(1, ig.STREAM_X, 0, T * D).reshape(T, D)
    x[5] = 0                     # all-zero row: scale 1, codes 0
    x[6] = _awkward_bf16(rng, (D,))
    x[7, :] = 0
    x[7, 17] = 0x0001            # smallest bf16 subnormal alone
    x[8] = x[8] | 0x8000         # all negative
    xq, sx = _gpu_quant_rows(gpu_lib, x)
    q_ref, s_ref = oracle.quant_rows(x)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), q_ref)


@pytest.mark.parametrize("E,D,N", [(3, 200, 136), (2, 7168, 64), (1, 16, 8)])
def test_quant_weights_bit_exact(gpu_lib, E, D, N):
    rng = np.random.default_rng(E * 1000 + D)
    W = ig.normal_bf16(2, ig.STREAM_W, 0, E * D * N).reshape(E, D, N)
    W[0, :, 1] = 0                              # zero column
    W[E - 1, :, N - 1] = _awkward_bf16(rng, (D,))
    wq, sw = _gpu_quant_weights(gpu_lib, u16_to_bf16_dev(W))
    q_ref, s_ref = oracle.quant_cols(W)
    assert np.array_equal(sw.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(wq.cpu().numpy(), to_blocked(q_ref))


def _fp8_case(pk, x, topk, W, E, rows=None):
    """Routes on the GPU, checks the GPU codes against the oracle's, runs the
    FP8 GEMM on the oracle's codes and compares rows with the oracle."""
    T, k = topk.shape
    D = x.shape[1]
    De = W.shape[2]
    md = pk.MoeDispatch(T, k, E, D, De)
    md.route(torch.from_numpy(np.ascontiguousarray(topk, dtype=np.int32)).cuda())
    xq_g, sx_g = _gpu_quant_rows(pk, x)
    wq_g, sw_g = _gpu_quant_weights(pk, u16_to_bf16_dev(W))
    ref = oracle.run(topk, E)
    xq, sx = oracle.quant_rows(x)
    wq, sw = oracle.quant_cols(W)
    assert np.array_equal(xq_g.cpu().numpy(), xq)
    assert np.array_equal(wq_g.cpu().numpy(), to_blocked(wq))
    assert np.array_equal(sx_g.cpu().numpy(), sx) and np.array_equal(sw_g.cpu().numpy(), sw)
    del xq_g, wq_g
    out = torch.full((T * k, De), float("nan"), dtype=torch.bfloat16, device="cuda")
    pk.pk_moe_dispatch_gemm_fp8(_u8_dev(xq), torch.from_numpy(sx).cuda(), md.perm, md.offsets,
                                _u8_dev(to_blocked(wq)), torch.from_numpy(sw).cuda(), k, out,
                                md.status)
    torch.cuda.synchronize()
    assert md.status_code() == 0, pk.pk_status_str(md.status_code())
    assert np.array_equal(md.perm[:T * k].cpu().numpy().astype(np.int64), ref["perm"])
    if rows is None:
        rows = np.arange(T * k, dtype=np.int64)
    want = oracle.gemm_fp8_rows(xq, sx, ref["perm"], ref["offsets"], wq, sw, k, rows)
    got = bf16_dev_to_f64(out[torch.from_numpy(rows).cuda()])
    assert_gemm_close(got, want, rows)
    return out


FP8_MULTI_TILE = [
    # T,   D,   E, k,  De
    (512, 576, 4, 2, 640),      # ~256 rows/expert, 5 K-steps of 128, N tail 128
    (700, 208, 3, 1, 200),      # D not a multiple of 128, De not of 64
    (300, 1024, 8, 3, 1408),    # 8 K-steps, 3-m-tile units
    (1000, 64, 2, 2, 256),      # 1000 rows per expert: groups of two m-tiles
    (96, 16, 5, 2, 8),          # smallest legal D and De
    (2048, 1280, 32, 4, 384),   # many experts, ring wraps many times
    (770, 320, 2, 1, 600),      # half-empty CTA pair; De = 512 + 88
]


@pytest.mark.parametrize("T,D,E,k,De", FP8_MULTI_TILE)
def test_fp8_gemm_all_rows(gpu_lib, gemm_kernel, T, D, E, k, De):
    c = ig.make_case(ig.custom(T=T, D=D, E=E, k=k, De=De, seed=5))
    _fp8_case(gpu_lib, c.x, c.topk, c.W, E)


def test_fp8_gemm_skew_and_empty_experts(gpu_lib, gemm_kernel):
    c = ig.make_case(ig.custom(T=1500, D=256, E=16, k=2, De=320, zipf_s=1.4, seed=9))
    counts = np.bincount(c.topk.ravel(), minlength=16)
    assert counts.max() > 384  # at least one expert with groups of m-tiles
    _fp8_case(gpu_lib, c.x, c.topk, c.W, 16)


def test_fp8_gemm_every_last_m_tile_height(gpu_lib, gemm_kernel):
    from _gpu_util import LAST_TILE_COUNTS, routing_with_counts
    topk = routing_with_counts(LAST_TILE_COUNTS, seed=22)
    E, T = len(LAST_TILE_COUNTS), topk.shape[0]
    c = ig.make_case(ig.custom(T=T, D=384, E=E, k=1, De=320, seed=22))
    _fp8_case(gpu_lib, c.x, topk, c.W, E)


def test_fp8_gemm_bad_perm_entry_sets_status(gpu_lib, gemm_kernel):
    pk = gpu_lib
    T, k, E, D, De = 64, 2, 4, 64, 64
    c = ig.make_case(ig.custom(T=T, D=D, E=E, k=k, De=De, seed=2))
    md = pk.MoeDispatch(T, k, E, D, De)
    md.route(torch.from_numpy(c.topk).cuda())
    xq, sx = oracle.quant_rows(c.x)
    wq, sw = oracle.quant_cols(c.W)
    perm = md.perm.clone()
    perm[3] = T * k + 5
    out = torch.zeros((T * k, De), dtype=torch.bfloat16, device="cuda")
    pk.pk_moe_dispatch_gemm_fp8(_u8_dev(xq), torch.from_numpy(sx).cuda(), perm, md.offsets,
                                _u8_dev(to_blocked(wq)), torch.from_numpy(sw).cuda(), k, out,
                                md.status)
    torch.cuda.synchronize()
    assert md.status_code() == pk.PK_ERR_BAD_INDEX
    assert bool(torch.isfinite(out.float()).all())


@pytest.mark.slow
def test_fp8_full_size_ep_sampled(gpu_lib):
    """T=8192 D=7168 E=256 k=8 D_expert=2048: GPU codes of x and of a sample
    of experts bit-exact; GEMM rows of those experts against the oracle."""
    pk = gpu_lib
    wl = ig.WORKLOADS["ep"]
    x = ig.make_x(wl)
    topk = ig.make_topk(wl)
    ref = oracle.run(topk, wl.E)
    experts = [0, 1, 77, 128, 200, 255]
    W = ig.make_W(wl, experts=experts)   # other experts all zero
    md = pk.MoeDispatch(wl.T, wl.k, wl.E, wl.D, wl.De)
    md.route(torch.from_numpy(topk).cuda())
    xq_g, sx_g = _gpu_quant_rows(pk, x)
    xq, sx = oracle.quant_rows(x)
    assert np.array_equal(xq_g.cpu().numpy(), xq)
    assert np.array_equal(sx_g.cpu().numpy(), sx)
    Wd = u16_to_bf16_dev(W)
    wq_g, sw_g = _gpu_quant_weights(pk, Wd)
    del Wd
    q_ref, s_ref = oracle.quant_cols(W[experts])
    assert np.array_equal(wq_g[experts].cpu().numpy(), to_blocked(q_ref))
    assert np.array_equal(sw_g[experts].cpu().numpy(), s_ref)
    out = torch.empty((wl.T * wl.k, wl.De), dtype=torch.bfloat16, device="cuda")
    pk.pk_moe_dispatch_gemm_fp8(xq_g, sx_g, md.perm, md.offsets, wq_g, sw_g, wl.k, out,
                                md.status)
    torch.cuda.synchronize()
    assert md.status_code() == 0
    offsets = ref["offsets"]
    rows = boundary_rows(offsets, np.random.default_rng(4), 0)
    in_sample = np.isin(np.searchsorted(offsets, rows, side="right") - 1, experts)
    rows = rows[in_sample]
    assert rows.size > 10
    # expected values from the oracle's codes only: experts outside the sample
    # are zero in W and never read by the sampled rows
    wq_full = np.zeros((wl.E, wl.De, wl.D), dtype=np.uint8)
    sw_full = np.ones((wl.E, wl.De), dtype=np.float32)
    wq_full[experts] = q_ref
    sw_full[experts] = s_ref
    want = oracle.gemm_fp8_rows(xq, sx, ref["perm"], offsets, wq_full, sw_full, wl.k, rows)
    got = bf16_dev_to_f64(out[torch.from_numpy(rows).cuda()])
    assert_gemm_close(got, want, rows)
    assert bool(torch.isfinite(out.float()).all())


def test_fp8_tiny_and_mid_workloads(gpu_lib):
    """The named small workloads: every row of tiny, boundary and random rows of mid."""
    c = ig.make_case(ig.WORKLOADS["tiny"])
    _fp8_case(gpu_lib, c.x, c.topk, c.W, ig.WORKLOADS["tiny"].E)
    wl = ig.WORKLOADS["mid"]
    c = ig.make_case(wl)
    rows = boundary_rows(oracle.route_counts(c.topk, wl.E)[1], np.random.default_rng(5), 256)
    _fp8_case(gpu_lib, c.x, c.topk, c.W, wl.E, rows=rows)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["skew", "decode"])
def test_fp8_full_size_sampled(gpu_lib, name):
    """T=8192 (skew, Zipf-biased routing) or T=128 (decode), D=7168, E=256,
    k=8, D_expert=2048: x codes bit-exact in full, W codes of a sample of
    experts bit-exact, GEMM rows of those experts against the oracle."""
    pk = gpu_lib
    wl = ig.WORKLOADS[name]
    x = ig.make_x(wl)
    topk = ig.make_topk(wl)
    ref = oracle.run(topk, wl.E)
    counts = ref["counts"]
    touched = np.flatnonzero(counts)
    # the heaviest expert, the lightest touched ones, and a few in between
    order = touched[np.argsort(counts[touched])]
    experts = sorted({int(e) for e in list(order[:2]) + list(order[-2:]) +
                      list(order[len(order) // 2:][:2])})
    W = ig.make_W(wl, experts=experts)
    md = pk.MoeDispatch(wl.T, wl.k, wl.E, wl.D, wl.De)
    md.route(torch.from_numpy(topk).cuda())
    xq_g, sx_g = _gpu_quant_rows(pk, x)
    xq, sx = oracle.quant_rows(x)
    assert np.array_equal(xq_g.cpu().numpy(), xq) and np.array_equal(sx_g.cpu().numpy(), sx)
    Wd = u16_to_bf16_dev(W)
    wq_g, sw_g = _gpu_quant_weights(pk, Wd)
    del Wd
    q_ref, s_ref = oracle.quant_cols(W[experts])
    assert np.array_equal(wq_g[experts].cpu().numpy(), to_blocked(q_ref))
    assert np.array_equal(sw_g[experts].cpu().numpy(), s_ref)
    out = torch.empty((wl.T * wl.k, wl.De), dtype=torch.bfloat16, device="cuda")
    pk.pk_moe_dispatch_gemm_fp8(xq_g, sx_g, md.perm, md.offsets, wq_g, sw_g, wl.k, out, md.status)
    torch.cuda.synchronize()
    assert md.status_code() == 0
    offsets = ref["offsets"]
    rows = boundary_rows(offsets, np.random.default_rng(6), 0)
    rows = rows[np.isin(np.searchsorted(offsets, rows, side="right") - 1, experts)]
    assert rows.size >= 6
    wq_full = np.zeros((wl.E, wl.De, wl.D), dtype=np.uint8)
    sw_full = np.ones((wl.E, wl.De), dtype=np.float32)
    wq_full[experts] = q_ref
    sw_full[experts] = s_ref
    want = oracle.gemm_fp8_rows(xq, sx, ref["perm"], offsets, wq_full, sw_full, wl.k, rows)
    got = bf16_dev_to_f64(out[torch.from_numpy(rows).cuda()])
    assert_gemm_close(got, want, rows)


@pytest.mark.parametrize("RT,K,E,k,N", [(512, 640, 4, 2, 576), (300, 208, 3, 1, 200),
                                        (1000, 128, 2, 2, 256), (None, 256, None, 1, 200)])
def test_fp8_grouped_gemm(gpu_lib, RT, K, E, k, N):
    """Down-projection on E4M3 codes: rows already in expert order (A's row
    j is its own token, so the oracle's perm is the identity with k = 1).
    RT = None: experts with every height of the last m-tile."""
    pk = gpu_lib
    topk = None
    if RT is None:
        from _gpu_util import LAST_TILE_COUNTS, routing_with_counts
        topk = routing_with_counts(LAST_TILE_COUNTS, seed=23)
        E, RT = len(LAST_TILE_COUNTS), topk.shape[0]
    wl = ig.custom(T=RT, D=K, E=E, k=k, De=N, seed=14)
    if topk is None:
        topk = ig.make_topk(wl)
    _, offsets = oracle.route_counts(topk, E)
    R = RT * k
    A = ig.normal_bf16(14, 7, 0, R * K).reshape(R, K)
    W2 = ig.make_W(wl)
    aq, sa = oracle.quant_rows(A)
    wq, sw = oracle.quant_cols(W2)
    out = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.pk_moe_grouped_gemm_fp8(_u8_dev(aq), torch.from_numpy(sa).cuda(),
                               torch.from_numpy(offsets.astype(np.int32)).cuda(),
                               _u8_dev(to_blocked(wq)), torch.from_numpy(sw).cuda(), out, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rows = np.arange(R, dtype=np.int64)
    want = oracle.gemm_fp8_rows(aq, sa, rows, offsets, wq, sw, 1, rows)
    assert_gemm_close(bf16_dev_to_f64(out), want, rows)
