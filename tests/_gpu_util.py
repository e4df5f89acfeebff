"""Helpers shared by the GPU parity tests (not collected as a test module)."""
from __future__ import annotations

import numpy as np
import torch

import inputgen as ig
import oracle

# Element-wise GEMM tolerance against the float64 oracle.
ATOL = 2e-2
RTOL = 1e-2


def u16_to_bf16_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)


def bf16_dev_to_f64(t: torch.Tensor) -> np.ndarray:
    bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return ig.bf16_bits_to_f64(bits)


def run_gpu(pk, x_u16, topk, W_dev, E, De, x_dev=None):
    """Runs the three C-ABI calls; returns numpy copies of every output."""
    T, k = topk.shape
    D = x_u16.shape[1]
    md = pk.MoeDispatch(T, k, E, D, De)
    x = x_dev if x_dev is not None else u16_to_bf16_dev(x_u16)
    tk = torch.from_numpy(np.ascontiguousarray(topk, dtype=np.int32)).cuda()
    md.route(tk)
    md.gemm(x, W_dev)
    torch.cuda.synchronize()
    R = T * k
    return {
        "counts": md.counts.cpu().numpy(),
        "offsets": md.offsets.cpu().numpy(),
        "perm": md.perm[:R].cpu().numpy(),
        "inv_perm": md.inv_perm[:R].cpu().numpy(),
        "out_dev": md.out[:R],
        "status": md.status_code(),
        "md": md,
    }


def assert_indices_exact(res, ref):
    assert np.array_equal(res["counts"].astype(np.int64), ref["counts"])
    assert np.array_equal(res["offsets"].astype(np.int64), ref["offsets"])
    assert np.array_equal(res["perm"].astype(np.int64), ref["perm"])
    assert np.array_equal(res["inv_perm"].astype(np.int64), ref["inv_perm"])


def assert_gemm_close(gpu_rows: np.ndarray, ref_rows: np.ndarray, rows=None):
    err = np.abs(gpu_rows - ref_rows)
    bound = ATOL + RTOL * np.abs(ref_rows)
    bad = err > bound
    if bad.any():
        i, n = np.argwhere(bad)[0]
        r = rows[i] if rows is not None else i
        raise AssertionError(
            f"{int(bad.sum())} of {bad.size} elements outside |gpu-ref| <= {ATOL} + {RTOL}|ref|; "
            f"first at row {r} col {n}: gpu={gpu_rows[i, n]!r} ref={ref_rows[i, n]!r}")
    assert np.isfinite(gpu_rows).all()


def boundary_rows(offsets: np.ndarray, rng, n_random: int = 64, per_expert=True) -> np.ndarray:
    """First/last rows of every expert, rows at 128-row tile edges, random rows."""
    R = int(offsets[-1])
    rows = set()
    E = offsets.size - 1
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi <= lo:
            continue
        rows.update((lo, hi - 1))
        if per_expert:
            for b in (31, 32, 127, 128, 255, 256, 257, 383, 384, 511, 512):
                if lo + b < hi:
                    rows.add(lo + b)
    if R:
        rows.update(int(v) for v in rng.integers(0, R, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)


def check_case(pk, x_u16, topk, W_u16, E, rows=None, W_dev=None, threads=None):
    """Full parity check of one case; GEMM on `rows` (all rows when None)."""
    De = W_u16.shape[2]
    if W_dev is None:
        W_dev = u16_to_bf16_dev(W_u16)
    res = run_gpu(pk, x_u16, topk, W_dev, E, De)
    assert res["status"] == 0, pk.pk_status_str(res["status"])
    ref = oracle.run(topk, E)
    assert_indices_exact(res, ref)
    R = topk.size
    if rows is None:
        rows = np.arange(R, dtype=np.int64)
    if len(rows):
        want = oracle.gemm_rows(x_u16, ref["perm"], ref["offsets"], W_u16, topk.shape[1], rows,
                                threads)
        got = bf16_dev_to_f64(res["out_dev"][torch.from_numpy(rows).cuda()])
        assert_gemm_close(got, want, rows)
    return res, ref


def to_blocked(q):
    """E4M3 codes [E, N, D] (column n's codes contiguous) into the blocked
    layout of the C ABI: [E, ceil(N/64), ceil(D/128), 64, 128], zero-padded."""
    E, N, D = q.shape
    NB, KB = -(-N // 64), -(-D // 128)
    p = np.zeros((E, NB * 64, KB * 128), dtype=np.uint8)
    p[:, :N, :D] = q
    return np.ascontiguousarray(p.reshape(E, NB, 64, KB, 128).transpose(0, 1, 3, 2, 4))


def to_mx_scale_pieces(sw):
    """E8M0 bytes [E, N, D // 32] of W's columns into the C ABI's scale pieces:
    per (e, 192-column tile t, 128-code group ks) 1 KiB, byte h*512 + r*16 +
    g*4 + j = scale of block 4 ks + j of column 192 t + 128 h + 32 g + r."""
    E, N, nb = sw.shape
    KS, NT = nb // 4, -(-N // 192)
    out = np.zeros((E, NT, KS, 2, 32, 4, 4), dtype=np.uint8)   # e, t, ks, h, r, g, j
    for t in range(NT):
        for h in range(2):
            for g in range(4):
                if 128 * h + 32 * g >= 192:
                    continue
                n0 = 192 * t + 128 * h + 32 * g
                n1 = min(n0 + 32, N)
                if n1 <= n0:
                    continue
                blk = sw[:, n0:n1, :].reshape(E, n1 - n0, KS, 4)
                out[:, t, :, h, : n1 - n0, g, :] = blk.transpose(0, 2, 1, 3)
    return out.reshape(-1)


# Rows per expert that put every height of a unit's last m-tile on the GPU
# GEMM: 1..64 rows (an M = 64 MMA) and 65..128 (M = 128), as the only m-tile,
# the second of two, the third of a 3-m-tile unit and the last of a group of
# a heavy expert (5 m-tiles: groups of 2, 2, 1; 7 m-tiles: 2, 2, 2, 1), plus
# the edges 64/65, 192/193, 320/321, 448/449 and an empty expert.
LAST_TILE_COUNTS = [1, 17, 64, 65, 100, 128, 129, 160, 192, 193, 250, 256, 257, 290, 320,
                    321, 384, 400, 448, 449, 520, 0, 800]


def routing_with_counts(counts, seed=0):
    """top-1 routing [T, 1] in which expert e gets counts[e] tokens, shuffled."""
    owner = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    np.random.default_rng(seed).shuffle(owner)
    return owner.reshape(-1, 1)
