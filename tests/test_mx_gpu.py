"""GPU parity of the MXFP8 (microscaled FP8) variant: block quantisation and
the block-scaled dispatch GEMM.

Codes and E8M0 scale bytes must match the oracle bit for bit (both sides take
every decision in IEEE fp32 on the same bf16 inputs). The GEMM is checked on
the oracle's own codes and scales: |gpu - ref| <= 2e-2 + 1e-2 |ref|
element-wise against the float64 sum of dequantised products -- the bound of
the bf16 path, since both sides read identical 8-bit inputs and identical
power-of-two scales and differ only by fp32 accumulation order and the final
bf16 rounding.
"""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from _gpu_util import (assert_gemm_close, bf16_dev_to_f64, boundary_rows, to_blocked,
                       to_mx_scale_pieces, u16_to_bf16_dev)

pytestmark = pytest.mark.gpu


def _u8_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def _awkward_bf16(rng, shape):
    """bf16 bits: zeros, subnormals, huge and tiny magnitudes, exact powers of
    two, and values that land just below and above 448 after scaling."""
    v = rng.standard_normal(shape).astype(np.float32)
    v[..., ::7] *= np.float32(1e-30)
    v[..., 3::11] *= np.float32(1e30)
    v[..., 5::13] = np.float32(2.0) ** rng.integers(-20, 20, size=v[..., 5::13].shape)
    v[..., 9::17] = np.float32(500.0)          # block max that saturates to 448 * 2^s
    v[..., 10::17] = np.float32(447.0)
    return torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _gpu_quant_rows(pk, x_u16):
    T, D = x_u16.shape
    xq = torch.empty((T, D), dtype=torch.uint8, device="cuda")
    sx = torch.empty((T, D // 32), dtype=torch.uint8, device="cuda")
    pk.pk_moe_quant_rows_mx(u16_to_bf16_dev(x_u16), xq, sx)
    torch.cuda.synchronize()
    return xq, sx


def _gpu_quant_weights(pk, W_dev):
    E, D, N = W_dev.shape
    wq = torch.full((pk.pk_moe_fp8_weight_bytes(E, D, N),), 0x55, dtype=torch.uint8, device="cuda")
    swb = torch.full((pk.pk_moe_mx_weight_scale_bytes(E, D, N),), 0x55, dtype=torch.uint8,
                     device="cuda")     # padding must come back zero
    pk.pk_moe_quant_weights_mx(W_dev, wq, swb)
    torch.cuda.synchronize()
    return wq, swb


@pytest.mark.parametrize("D", [7168, 256, 96])
def test_mx_quant_rows_bit_exact(gpu_lib, D):
    rng = np.random.default_rng(7)
    T = 211
    x = ig.normal_bf16(1, ig.STREAM_X, 0, T * D).reshape(T, D)
    x[5] = 0                      # all-zero blocks: byte 0, codes 0
    x[6] = _awkward_bf16(rng, (D,))
    x[7, :] = 0
    x[7, 17] = 0x0001             # smallest bf16 subnormal alone in its block
    x[8] = x[8] | 0x8000          # all negative
    xq, sx = _gpu_quant_rows(gpu_lib, x)
    q_ref, s_ref = oracle.mx_quant_rows(x)
    assert np.array_equal(sx.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), q_ref)


@pytest.mark.parametrize("E,D,N", [(3, 256, 136), (2, 7168, 200), (1, 128, 8), (2, 384, 400)])
def test_mx_quant_weights_bit_exact(gpu_lib, E, D, N):
    rng = np.random.default_rng(E * 1000 + D + N)
    W = ig.normal_bf16(2, ig.STREAM_W, 0, E * D * N).reshape(E, D, N)
    W[0, :, 1] = 0                               # zero column
    W[E - 1, :, N - 1] = _awkward_bf16(rng, (D,))
    wq, swb = _gpu_quant_weights(gpu_lib, u16_to_bf16_dev(W))
    q_ref, s_ref = oracle.mx_quant_cols(W)
    assert np.array_equal(wq.cpu().numpy(), to_blocked(q_ref).reshape(-1))
    assert np.array_equal(swb.cpu().numpy(), to_mx_scale_pieces(s_ref))


def _mx_case(pk, x, topk, W, E, rows=None):
    """Routes on the GPU, checks the GPU codes and scales against the
    oracle's, runs the MX GEMM and compares rows with the oracle."""
    T, k = topk.shape
    D = x.shape[1]
    De = W.shape[2]
    md = pk.MoeDispatch(T, k, E, D, De)
    md.route(torch.from_numpy(np.ascontiguousarray(topk, dtype=np.int32)).cuda())
    xq_g, sx_g = _gpu_quant_rows(pk, x)
    wq_g, swb_g = _gpu_quant_weights(pk, u16_to_bf16_dev(W))
    ref = oracle.run(topk, E)
    xq, sx = oracle.mx_quant_rows(x)
    wq, sw = oracle.mx_quant_cols(W)
    assert np.array_equal(xq_g.cpu().numpy(), xq) and np.array_equal(sx_g.cpu().numpy(), sx)
    assert np.array_equal(wq_g.cpu().numpy(), to_blocked(wq).reshape(-1))
    assert np.array_equal(swb_g.cpu().numpy(), to_mx_scale_pieces(sw))
    out = torch.full((T * k, De), float("nan"), dtype=torch.bfloat16, device="cuda")
    pk.pk_moe_dispatch_gemm_mxfp8(xq_g, sx_g, md.perm, md.offsets, wq_g, swb_g, E, De, k, out,
                                  md.status)
    torch.cuda.synchronize()
    assert md.status_code() == 0, pk.pk_status_str(md.status_code())
    assert np.array_equal(md.perm[:T * k].cpu().numpy().astype(np.int64), ref["perm"])
    if rows is None:
        rows = np.arange(T * k, dtype=np.int64)
    want = oracle.gemm_mx_rows(xq, sx, ref["perm"], ref["offsets"], wq, sw, k, rows)
    got = bf16_dev_to_f64(out[torch.from_numpy(rows).cuda()])
    assert_gemm_close(got, want, rows)
    return out


MX_MULTI_TILE = [
    # T,   D,   E, k,  De
    (512, 640, 4, 2, 640),      # ~256 rows/expert, 5 K-steps, N tail: 192 x 3 + 64
    (700, 256, 3, 1, 200),      # ~233 rows/expert, De not a multiple of 64
    (300, 1024, 8, 3, 1408),    # 8 K-steps, experts of 257..384 rows: groups of 2 + 1 m-tiles
    (1000, 128, 2, 2, 256),     # 1000 rows per expert: four groups
    (96, 128, 5, 2, 8),         # one K-step, smallest De
    (2048, 1280, 32, 4, 384),   # many experts, the rings wrap many times
    (770, 384, 2, 1, 600),      # 3 and 4 m-tiles; De = 576 + 24
]


@pytest.mark.parametrize("T,D,E,k,De", MX_MULTI_TILE)
def test_mx_gemm_all_rows(gpu_lib, T, D, E, k, De):
    c = ig.make_case(ig.custom(T=T, D=D, E=E, k=k, De=De, seed=6))
    _mx_case(gpu_lib, c.x, c.topk, c.W, E)


def _blocky_bf16(rng, rows, cols):
    """bf16 bits whose 32-element blocks differ in magnitude by up to 2^+-20
    (every block its own scale byte), with all-zero blocks, subnormal and
    saturating block maxima (500 and 447 land above and below 448 after
    scaling) mixed in."""
    v = rng.standard_normal((rows, cols)).astype(np.float32)
    v *= np.float32(2.0) ** rng.integers(-20, 20, size=(rows, cols // 32)).repeat(32, 1)
    v[::5, 32:64] = 0
    v[1::5, 0] = np.float32(500.0)
    v[2::5, 64 % cols] = np.float32(447.0)
    v[3::7, :16] = np.float32(1e-39)
    return torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def test_mx_gemm_blocks_of_varied_scale(gpu_lib):
    """Both operands with blocks of widely different magnitude, zero blocks,
    subnormals and saturating block maxima."""
    rng = np.random.default_rng(12)
    T, D, E, k, De = 200, 256, 3, 2, 136
    c = ig.make_case(ig.custom(T=T, D=D, E=E, k=k, De=De, seed=13))
    x = _blocky_bf16(rng, T, D)
    W = _blocky_bf16(rng, E * De, D).reshape(E, De, D).transpose(0, 2, 1).copy()  # blocks along d
    _mx_case(gpu_lib, x, c.topk, W, E)


def test_mx_gemm_skew_and_empty_experts(gpu_lib):
    c = ig.make_case(ig.custom(T=1500, D=256, E=16, k=2, De=320, zipf_s=1.4, seed=9))
    counts = np.bincount(c.topk.ravel(), minlength=16)
    assert counts.max() > 384  # an expert of several row groups
    _mx_case(gpu_lib, c.x, c.topk, c.W, 16)


def test_mx_gemm_bad_perm_entry_sets_status(gpu_lib):
    pk = gpu_lib
    T, k, E, D, De = 64, 2, 4, 128, 64
    c = ig.make_case(ig.custom(T=T, D=D, E=E, k=k, De=De, seed=2))
    md = pk.MoeDispatch(T, k, E, D, De)
    md.route(torch.from_numpy(c.topk).cuda())
    xq, sx = _gpu_quant_rows(pk, c.x)
    wq, swb = _gpu_quant_weights(pk, u16_to_bf16_dev(c.W))
    perm = md.perm.clone()
    perm[3] = T * k + 5
    out = torch.zeros((T * k, De), dtype=torch.bfloat16, device="cuda")
    pk.pk_moe_dispatch_gemm_mxfp8(xq, sx, perm, md.offsets, wq, swb, E, De, k, out, md.status)
    torch.cuda.synchronize()
    assert md.status_code() == pk.PK_ERR_BAD_INDEX


def test_mx_tiny_and_mid_workloads(gpu_lib):
    """The named small workloads: every row of tiny, boundary and random rows of mid."""
    c = ig.make_case(ig.WORKLOADS["tiny"])
    _mx_case(gpu_lib, c.x, c.topk, c.W, ig.WORKLOADS["tiny"].E)
    wl = ig.WORKLOADS["mid"]
    c = ig.make_case(wl)
    rows = boundary_rows(oracle.route_counts(c.topk, wl.E)[1], np.random.default_rng(5), 256)
    _mx_case(gpu_lib, c.x, c.topk, c.W, wl.E, rows=rows)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["ep", "skew", "decode"])
def test_mx_full_size_sampled(gpu_lib, name):
    """D=7168, E=256, k=8, D_expert=2048 with T=8192 (ep, skew) or 128
    (decode): x codes and scales bit-exact in full, W codes and scales of a
    sample of experts bit-exact, GEMM rows of those experts against the
    oracle."""
    pk = gpu_lib
    wl = ig.WORKLOADS[name]
    x = ig.make_x(wl)
    topk = ig.make_topk(wl)
    ref = oracle.run(topk, wl.E)
    counts = ref["counts"]
    touched = np.flatnonzero(counts)
    order = touched[np.argsort(counts[touched])]
    experts = sorted({int(e) for e in list(order[:2]) + list(order[-2:]) +
                      list(order[len(order) // 2:][:2])})
    W = ig.make_W(wl, experts=experts)   # other experts all zero
    md = pk.MoeDispatch(wl.T, wl.k, wl.E, wl.D, wl.De)
    md.route(torch.from_numpy(topk).cuda())
    xq_g, sx_g = _gpu_quant_rows(pk, x)
    xq, sx = oracle.mx_quant_rows(x)
    assert np.array_equal(xq_g.cpu().numpy(), xq) and np.array_equal(sx_g.cpu().numpy(), sx)
    Wd = u16_to_bf16_dev(W)
    wq_g, swb_g = _gpu_quant_weights(pk, Wd)
    del Wd
    q_ref, s_ref = oracle.mx_quant_cols(np.ascontiguousarray(W[experts]))
    NB, KS, NT = -(-wl.De // 64), wl.D // 128, -(-wl.De // 192)
    wq_v = wq_g.view(wl.E, -1)
    swb_v = swb_g.view(wl.E, NT * KS * 1024)
    assert np.array_equal(wq_v[experts].cpu().numpy(), to_blocked(q_ref).reshape(len(experts), -1))
    assert np.array_equal(swb_v[experts].cpu().numpy(),
                          to_mx_scale_pieces(s_ref).reshape(len(experts), -1))
    out = torch.empty((wl.T * wl.k, wl.De), dtype=torch.bfloat16, device="cuda")
    pk.pk_moe_dispatch_gemm_mxfp8(xq_g, sx_g, md.perm, md.offsets, wq_g, swb_g, wl.E, wl.De,
                                  wl.k, out, md.status)
    torch.cuda.synchronize()
    assert md.status_code() == 0
    offsets = ref["offsets"]
    rows = boundary_rows(offsets, np.random.default_rng(6), 0)
    rows = rows[np.isin(np.searchsorted(offsets, rows, side="right") - 1, experts)]
    assert rows.size >= 6
    wq_full = np.zeros((wl.E, wl.De, wl.D), dtype=np.uint8)
    sw_full = np.full((wl.E, wl.De, wl.D // 32), 127, dtype=np.uint8)
    wq_full[experts] = q_ref
    sw_full[experts] = s_ref
    want = oracle.gemm_mx_rows(xq, sx, ref["perm"], offsets, wq_full, sw_full, wl.k, rows)
    got = bf16_dev_to_f64(out[torch.from_numpy(rows).cuda()])
    assert_gemm_close(got, want, rows)
    assert bool(torch.isfinite(out.float()).all())
