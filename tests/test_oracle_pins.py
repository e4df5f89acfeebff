"""Pins of the CPU oracle to facts outside itself (CPU only).

The pages print no worked example for token dispatch, so the oracle is pinned
by a hand-worked example, invariants of the routing, library routines
(numpy bincount / stable argsort / float64 matmul), closed forms (identity and
shifted-identity weights, all-ones weights) and brute force on tiny inputs.
The last group plants mistakes in a small pure-Python copy of the path and
checks that the same pins catch each of them.
"""
import math

import numpy as np
import pytest

import inputgen as ig
import oracle


def bf16(v):
    """float -> bf16 bits (values used here are exactly representable)."""
    a = np.asarray(v, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------- checkers
def check_routing(topk, E, counts, offsets, perm, inv):
    """All pins on counts / offsets / perm / inv_perm; raises AssertionError."""
    T, k = topk.shape
    R = T * k
    flat = topk.reshape(-1)
    # counts: library histogram
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    # offsets: exclusive prefix sum
    assert offsets[0] == 0 and offsets[E] == R
    assert np.array_equal(np.diff(offsets), counts)
    # perm: a permutation of the flat indices
    assert np.array_equal(np.sort(perm), np.arange(R))
    # each token exactly k times
    assert np.array_equal(np.bincount(perm // k, minlength=T), np.full(T, k))
    # segment e holds only entries routed to e, in increasing flat order
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)
    # the stable library sort of the expert ids gives the same order
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    # inverse restores the routing
    assert np.array_equal(inv[perm], np.arange(R))
    assert np.array_equal(perm[inv], np.arange(R))
    pos_expert = np.searchsorted(offsets, np.arange(R), side="right") - 1
    assert np.array_equal(pos_expert[inv], flat)


def check_gemm_closed_forms(path, rng):
    """Pins on a GEMM function path(topk, E, x_bits, W_bits) -> (perm, offsets, out)."""
    T, k, E, D, De = 9, 3, 5, 24, 16
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = bf16(rng.integers(-64, 64, size=(T, D)) / 8.0)
    # identity weights: row j reproduces x[perm[j] // k, :De] exactly
    W = np.zeros((E, D, De), dtype=np.float32)
    for e in range(E):
        W[e, :De, :De] = np.eye(De)
    perm, offsets, out = path(topk, E, x, bf16(W))
    xf = ig.bf16_bits_to_f64(x)
    assert np.array_equal(out, xf[perm // k][:, :De])
    # shifted identity W[e, d, n] = [d == (n + e) mod D]: proves which expert is used
    W = np.zeros((E, D, De), dtype=np.float32)
    for e in range(E):
        for n in range(De):
            W[e, (n + e) % D, n] = 1.0
    perm, offsets, out = path(topk, E, x, bf16(W))
    ex = np.searchsorted(offsets, np.arange(T * k), side="right") - 1
    cols = (np.arange(De)[None, :] + ex[:, None]) % D
    assert np.array_equal(out, xf[(perm // k)[:, None], cols])
    # all-ones weights: every column is the exact row sum (math.fsum)
    W = np.ones((E, D, De), dtype=np.float32)
    perm, offsets, out = path(topk, E, x, bf16(W))
    for j in range(T * k):
        s = math.fsum(xf[perm[j] // k])
        assert np.all(out[j] == s)


def check_gemm_library(path, rng, T=40, k=2, E=6, D=96, De=40):
    """float64 matmul of the gathered rows, expert by expert, and brute force."""
    logits = rng.standard_normal((T, E))
    topk = np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)
    x = bf16(rng.standard_normal((T, D)).astype(np.float32))
    W = bf16((rng.standard_normal((E, D, De)) / np.sqrt(D)).astype(np.float32))
    perm, offsets, out = path(topk, E, x, W)
    xf, wf = ig.bf16_bits_to_f64(x), ig.bf16_bits_to_f64(W)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        ref = xf[perm[lo:hi] // k] @ wf[e]
        scale = np.abs(xf[perm[lo:hi] // k]) @ np.abs(wf[e]) + 1e-300
        assert np.all(np.abs(out[lo:hi] - ref) <= 1e-12 * scale)
    # brute force with exact summation on a few rows
    for j in (0, T * k // 2, T * k - 1):
        e = int(np.searchsorted(offsets, j, side="right") - 1)
        t = perm[j] // k
        for n in (0, De // 3, De - 1):
            exact = math.fsum(xf[t, d] * wf[e, d, n] for d in range(D))
            assert abs(out[j, n] - exact) <= 1e-12 * sum(abs(xf[t, d] * wf[e, d, n]) for d in range(D))


def oracle_path(topk, E, x, W):
    res = oracle.run(topk, E, x, W)
    return res["perm"], res["offsets"], res["out"]


# ------------------------------------------------------------ oracle pins
def test_hand_worked_example():
    # T=4 tokens, k=2 slots, E=4 experts (expert 3 receives nothing).
    # flat index f = t*k + s:  f: 0 1 2 3 4 5 6 7
    #                   expert: 2 0 0 2 1 2 2 1
    topk = np.array([[2, 0], [0, 2], [1, 2], [2, 1]], dtype=np.int32)
    counts, offsets = oracle.route_counts(topk, 4)
    assert counts.tolist() == [2, 2, 4, 0]
    assert offsets.tolist() == [0, 2, 4, 8, 8]
    perm, inv = oracle.build_perm(topk, 4, offsets)
    # expert 0: f=1,2; expert 1: f=4,7; expert 2: f=0,3,5,6
    assert perm.tolist() == [1, 2, 4, 7, 0, 3, 5, 6]
    assert inv.tolist() == [4, 0, 1, 5, 2, 6, 7, 3]
    # GEMM with D=2, De=2 and small exact weights, worked by hand:
    x = bf16([[1, 2], [3, -1], [0.5, 4], [-2, 1]])
    W = bf16([[[1, 0], [0, 1]], [[2, 1], [0, 1]], [[1, 1], [1, -1]], [[0, 0], [0, 0]]])
    out = oracle.gemm_all(x, perm, offsets, W, 2)
    expect = [[1, 2], [3, -1],            # expert 0 (identity): tokens 0, 1
              [1, 4.5], [-4, -1],          # expert 1: tokens 2, 3
              [3, -1], [2, 4], [4.5, -3.5], [-1, -3]]  # expert 2: tokens 0, 1, 2, 3
    assert out.tolist() == expect
    assert oracle.expert_of_row(offsets, 3) == 1 and oracle.expert_of_row(offsets, 8) == -1


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_routing_invariants_on_workloads(name):
    wl = ig.WORKLOADS[name]
    topk = ig.make_topk(wl)
    counts, offsets = oracle.route_counts(topk, wl.E)
    perm, inv = oracle.build_perm(topk, wl.E, offsets)
    check_routing(topk, wl.E, counts, offsets, perm, inv)


def test_routing_invariants_with_duplicates_and_empty_experts():
    rng = np.random.default_rng(3)
    for T, k, E in [(1, 1, 1), (7, 3, 2), (50, 4, 9), (300, 2, 40)]:
        topk = rng.integers(0, max(1, E // 2), size=(T, k)).astype(np.int32)  # upper experts empty
        counts, offsets = oracle.route_counts(topk, E)
        perm, inv = oracle.build_perm(topk, E, offsets)
        check_routing(topk, E, counts, offsets, perm, inv)
    # brute-force counts and the (expert, token, slot) order with sorted()
    topk = rng.integers(0, 5, size=(11, 3)).astype(np.int32)
    counts, offsets = oracle.route_counts(topk, 5)
    assert counts.tolist() == [sum(1 for t in range(11) for s in range(3) if topk[t, s] == e)
                               for e in range(5)]
    perm, _ = oracle.build_perm(topk, 5, offsets)
    order = sorted(((int(topk[t, s]), t, s) for t in range(11) for s in range(3)))
    assert perm.tolist() == [t * 3 + s for _, t, s in order]


def test_bad_index_is_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.route_counts(np.array([[0, 4]], dtype=np.int32), 4)
    with pytest.raises(oracle.OracleError):
        oracle.route_counts(np.array([[-1, 0]], dtype=np.int32), 4)


def test_empty_input():
    topk = np.zeros((0, 3), dtype=np.int32)
    counts, offsets = oracle.route_counts(topk, 5)
    assert counts.tolist() == [0] * 5 and offsets.tolist() == [0] * 6
    perm, inv = oracle.build_perm(topk, 5, offsets)
    assert perm.size == 0 and inv.size == 0


def test_gemm_closed_forms():
    check_gemm_closed_forms(oracle_path, np.random.default_rng(5))


def test_gemm_against_float64_matmul_and_brute_force():
    check_gemm_library(oracle_path, np.random.default_rng(6))


def test_gemm_tiny_workload_against_matmul():
    wl = ig.WORKLOADS["tiny"]
    case = ig.make_case(wl)
    res = oracle.run(case.topk, wl.E, case.x, case.W)
    xf, wf = ig.bf16_bits_to_f64(case.x), ig.bf16_bits_to_f64(case.W)
    off, perm = res["offsets"], res["perm"]
    for e in range(wl.E):
        rows = perm[off[e]:off[e + 1]] // wl.k
        ref = xf[rows] @ wf[e]
        scale = np.abs(xf[rows]) @ np.abs(wf[e])
        assert np.all(np.abs(res["out"][off[e]:off[e + 1]] - ref) <= 1e-12 * scale)


def test_gemm_rows_independent_of_threads_and_subset():
    wl = ig.custom(T=33, D=64, E=4, k=2, De=24)
    case = ig.make_case(wl)
    full = oracle.run(case.topk, wl.E, case.x, case.W, threads=1)
    rows = np.array([65, 0, 17, 17, 3])
    part = oracle.gemm_rows(case.x, full["perm"], full["offsets"], case.W, wl.k, rows, threads=3)
    assert np.array_equal(part, full["out"][rows])


# ------------------------------------------- planted mistakes are caught
def python_path(topk, E, x, W, bug=None):
    """A small pure-Python copy of the path, used only to plant mistakes."""
    T, k = topk.shape
    flat = topk.reshape(-1)
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    if bug == "inclusive_scan":
        offsets[:-1] = offsets[1:]
    if bug == "slot_major":     # (expert, slot, token) instead of (expert, token, slot)
        order = sorted(range(T * k), key=lambda f: (flat[f], f % k, f // k))
    else:
        order = sorted(range(T * k), key=lambda f: (flat[f], f))
    perm = np.array(order, dtype=np.int64)
    xf, wf = ig.bf16_bits_to_f64(x), ig.bf16_bits_to_f64(W)
    De = W.shape[2]
    out = np.zeros((T * k, De))
    for j in range(T * k):
        e = int(np.searchsorted(offsets, j, side="right") - 1)
        t = perm[j] // k
        if bug == "token_mod":
            t = perm[j] % k
        if bug == "expert_minus_one":
            e = max(e - 1, 0)
        w = wf[e]
        if bug == "reversed_k":   # W read along d in the wrong direction
            w = wf[e][::-1]
        D = xf.shape[1]
        dmax = D - 1 if bug == "dropped_term" else D
        out[j] = xf[t, :dmax] @ w[:dmax]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(T * k)
    return counts, offsets, perm, inv, out


def test_python_copy_passes_all_pins():
    rng = np.random.default_rng(8)
    topk = np.stack([rng.permutation(6)[:3] for _ in range(20)]).astype(np.int32)
    counts, offsets, perm, inv, _ = python_path(topk, 6, np.zeros((20, 1), np.uint16),
                                                np.zeros((6, 1, 1), np.uint16))
    check_routing(topk, 6, counts, offsets, perm, inv)
    def p(tk, E, x, W):
        _, offsets, perm, _, out = python_path(tk, E, x, W)
        return perm, offsets, out
    check_gemm_closed_forms(p, np.random.default_rng(5))
    check_gemm_library(p, np.random.default_rng(6))


@pytest.mark.parametrize("bug", ["inclusive_scan", "slot_major"])
def test_planted_routing_mistakes_are_caught(bug):
    rng = np.random.default_rng(9)
    topk = np.stack([rng.permutation(6)[:3] for _ in range(20)]).astype(np.int32)
    counts, offsets, perm, inv, _ = python_path(topk, 6, np.zeros((20, 1), np.uint16),
                                                np.zeros((6, 1, 1), np.uint16), bug)
    with pytest.raises(AssertionError):
        check_routing(topk, 6, counts, offsets, perm, inv)


@pytest.mark.parametrize("bug", ["token_mod", "expert_minus_one", "reversed_k", "dropped_term"])
def test_planted_gemm_mistakes_are_caught(bug):
    def p(tk, E, x, W):
        _, offsets, perm, _, out = python_path(tk, E, x, W, bug)
        return perm, offsets, out
    caught = 0
    for checker, seed in ((check_gemm_closed_forms, 5), (check_gemm_library, 6)):
        try:
            checker(p, np.random.default_rng(seed))
        except AssertionError:
            caught += 1
    assert caught >= 1


# ------------------------------------------------ combine and router pins
def check_combine(comb, rng):
    """Pins on comb(src_bits, inv_perm, gates, T, k) -> float64 [T, C]."""
    T, k, E, C = 13, 3, 5, 24
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _, offsets = oracle.route_counts(topk, E)
    perm, inv = oracle.build_perm(topk, E, offsets)
    src = bf16(rng.standard_normal((T * k, C)).astype(np.float32))
    sf = ig.bf16_bits_to_f64(src)
    # one-hot gates pick a single expert output, exactly
    for s in range(k):
        g = np.zeros((T, k))
        g[:, s] = 1.0
        y = comb(src, inv, g, T, k)
        assert np.array_equal(y, sf[inv.reshape(T, k)[:, s]])
    # library reference: gather + einsum in float64
    g = rng.random((T, k))
    y = comb(src, inv, g, T, k)
    ref = np.einsum("ts,tsc->tc", g, sf[inv.reshape(T, k)])
    assert np.all(np.abs(y - ref) <= 1e-12 * (np.abs(g)[:, :, None] * np.abs(sf[inv.reshape(T, k)])).sum(1))
    # dispatch followed by combine with unit gates and k = 1 restores the rows
    tk1 = rng.integers(0, E, size=(T, 1)).astype(np.int32)
    _, off1 = oracle.route_counts(tk1, E)
    p1, i1 = oracle.build_perm(tk1, E, off1)
    x = bf16(rng.standard_normal((T, C)).astype(np.float32))
    dispatched = x[p1]                       # rows in sorted order
    y = comb(dispatched, i1, np.ones((T, 1)), T, 1)
    assert np.array_equal(y, ig.bf16_bits_to_f64(x))


def check_router(router, rng):
    """Pins on router(logits f32 [T,E], k) -> (topk, gates)."""
    from scipy.special import softmax
    T, E, k = 40, 37, 6
    l = rng.standard_normal((T, E)).astype(np.float32)
    idx, g = router(l, k)
    assert np.array_equal(idx, np.argsort(-l, axis=1, kind="stable")[:, :k])
    sel = np.take_along_axis(l.astype(np.float64), idx, axis=1)
    assert np.allclose(g, softmax(sel, axis=1), rtol=1e-14, atol=0)
    # ties go to the lower expert; equal logits give equal gates
    l = np.zeros((3, 9), dtype=np.float32)
    l[1, 4] = 1.0
    idx, g = router(l, 4)
    assert idx.tolist() == [[0, 1, 2, 3], [4, 0, 1, 2], [0, 1, 2, 3]]
    assert np.all(g[0] == 0.25)
    # k = E selects every expert once
    idx, _ = router(rng.standard_normal((5, 7)).astype(np.float32), 7)
    assert all(sorted(r) == list(range(7)) for r in idx.tolist())


def test_combine_pins():
    check_combine(lambda s, i, g, T, k: oracle.combine(s, i, g, T, k), np.random.default_rng(21))


def test_router_pins():
    check_router(oracle.router_topk, np.random.default_rng(22))


def test_planted_combine_and_router_mistakes_are_caught():
    def comb_perm_not_inv(src, inv, g, T, k):     # gathers with perm instead of inv_perm
        perm = np.empty_like(inv)
        perm[inv] = np.arange(inv.size)
        return oracle.combine(src, perm, g, T, k)

    def comb_gates_transposed(src, inv, g, T, k):
        return oracle.combine(src, inv, np.ascontiguousarray(g[:, ::-1]), T, k)

    def router_ties_high(l, k):                    # equal logits to the higher expert
        idx = np.argsort(-l[:, ::-1], axis=1, kind="stable")[:, :k]
        idx = l.shape[1] - 1 - idx
        _, g = oracle.router_topk(l, k)
        return idx, g

    def router_no_shift(l, k):                     # gates of all experts, not the k selected
        idx, _ = oracle.router_topk(l, k)
        from scipy.special import softmax
        return idx, softmax(l.astype(np.float64), axis=1)[np.arange(l.shape[0])[:, None], idx]

    for bad in (comb_perm_not_inv, comb_gates_transposed):
        with pytest.raises(AssertionError):
            check_combine(bad, np.random.default_rng(21))
    for bad in (router_ties_high, router_no_shift):
        with pytest.raises(AssertionError):
            check_router(bad, np.random.default_rng(22))


# ------------------------------------------------------------- FP8 pins
def test_e4m3_conversion_against_torch_and_format():
    import torch
    # every finite code round-trips, and the values follow the format
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            assert math.isnan(oracle.e4m3_to_f64(c))
            continue
        v = oracle.e4m3_to_f64(c)
        assert oracle.f32_to_e4m3(v) == (c if v != 0 or c == 0 else c)
    assert oracle.e4m3_to_f64(0x7E) == 448.0 and oracle.e4m3_to_f64(0x01) == 2.0 ** -9
    # round to nearest even on random in-range floats: torch's cast (library)
    rng = np.random.default_rng(31)
    v = np.concatenate([rng.standard_normal(20000) * 30, rng.standard_normal(5000) * 1e-2,
                        (rng.integers(-60, 60, 2000) + 0.5) / 8.0]).astype(np.float32)
    v = v[np.abs(v) < 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.f32_to_e4m3(float(a)) for a in v], dtype=np.uint8)
    assert np.array_equal(ours, ref)
    # saturation above the largest finite value
    assert oracle.f32_to_e4m3(1e6) == 0x7E and oracle.f32_to_e4m3(-500.0) == 0xFE


def check_quant_rows(qr, rng):
    x = bf16(rng.standard_normal((7, 96)).astype(np.float32) * rng.random((7, 1)).astype(np.float32))
    x[3] = 0                                   # an all-zero row keeps scale 1
    x[5] = 0
    x[5, 9] = 0x0001                           # amax = 2^-133: 448 / amax overflows float32
    x[6] = 0
    x[6, 2] = 0x0C00                           # amax = 2^-103: 448 / amax is finite
    q, s = qr(x)
    xf = ig.bf16_bits_to_f64(x)
    # every row is reconstructed within E4M3's error: half a step of the
    # 3-bit mantissa (2^-4 relative) for normal codes, half the subnormal
    # step 2^-9 (scaled) below 2^-6
    deq = np.array([[oracle.e4m3_to_f64(int(c)) for c in row] for row in q]) * s[:, None]
    assert np.all(np.abs(deq - xf) <= 2.0 ** -4 * np.abs(xf) + 2.0 ** -10 * s[:, None].astype(np.float64))
    assert s[5] == 1.0 and not q[5].any()
    assert s[6] == np.float32(2.0 ** -103 / 448.0) and q[6, 2] == 0x7E
    for t in range(7):
        amax = np.float32(np.abs(xf[t]).max())
        with np.errstate(over="ignore", divide="ignore"):
            overflow = not np.isfinite(np.float32(448.0) / amax)
        if overflow:
            assert s[t] == 1.0 and not q[t].any()
            continue
        assert s[t] == np.float32(amax / np.float32(448.0))
        inv = np.float32(448.0) / amax
        want = np.array([oracle.f32_to_e4m3(float(np.float32(a) * inv)) for a in xf[t]])
        assert np.array_equal(q[t], want)
        # the largest magnitude maps to 448
        assert abs(oracle.e4m3_to_f64(int(q[t][np.abs(xf[t]).argmax()]))) == 448.0


def test_quant_rows_and_cols():
    check_quant_rows(oracle.quant_rows, np.random.default_rng(32))
    rng = np.random.default_rng(33)
    W = bf16(rng.standard_normal((3, 40, 24)).astype(np.float32))
    q, s = oracle.quant_cols(W)
    # columns of W[e] are the rows of W[e].T
    for e in range(3):
        qe, se = oracle.quant_rows(np.ascontiguousarray(W[e].T))
        assert np.array_equal(q[e], qe) and np.array_equal(s[e], se)


def check_gemm_fp8(gemm, rng):
    T, k, E, D, N = 21, 2, 4, 64, 40
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _, offsets = oracle.route_counts(topk, E)
    perm, _ = oracle.build_perm(topk, E, offsets)
    x = bf16(rng.standard_normal((T, D)).astype(np.float32))
    W = bf16((rng.standard_normal((E, D, N)) / 8).astype(np.float32))
    xq, sx = oracle.quant_rows(x)
    wq, sw = oracle.quant_cols(W)
    out = gemm(xq, sx, perm, offsets, wq, sw, k, np.arange(T * k))
    deq = np.vectorize(oracle.e4m3_to_f64)
    xd = deq(xq) * sx[:, None].astype(np.float64)
    wd = deq(wq) * sw[:, :, None].astype(np.float64)          # [E, N, D]
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        ref = xd[perm[lo:hi] // k] @ wd[e].T
        assert np.all(np.abs(out[lo:hi] - ref) <= 1e-12 * (np.abs(xd[perm[lo:hi] // k]) @ np.abs(wd[e]).T))
    # and it approximates the bf16 GEMM within E4M3's precision
    bf = oracle.gemm_rows(x, perm, offsets, W, k, np.arange(T * k))
    assert np.abs(out - bf).max() < 0.2 * np.abs(bf).max()


def test_gemm_fp8_pins():
    check_gemm_fp8(oracle.gemm_fp8_rows, np.random.default_rng(34))


def test_planted_fp8_mistakes_are_caught():
    def scale_swapped(xq, sx, perm, offsets, wq, sw, k, rows):     # W scale by row, x by column
        out = oracle.gemm_fp8_rows(xq, np.ones_like(sx), perm, offsets, wq, np.ones_like(sw), k, rows)
        return out * sw.mean() * sx.mean()

    def unscaled_rows(xq):                                          # amax not mapped to 448
        q, s = oracle.quant_rows(xq)
        return q, s * 2
    with pytest.raises(AssertionError):
        check_gemm_fp8(scale_swapped, np.random.default_rng(34))
    with pytest.raises(AssertionError):
        check_quant_rows(unscaled_rows, np.random.default_rng(32))


# ------------------------------------------------------------ MXFP8 pins
# The MX formats' definition (32-element blocks along the reduction axis,
# one E8M0 power-of-two scale 2^s per block, s = floor(log2 amax) - 8 for
# E4M3 elements, codes E4M3(v / 2^s) with saturation) worked by hand.
def _bf16_vec(vals, n=32):
    v = np.zeros(n, dtype=np.float32)
    v[: len(vals)] = vals
    return (v.view(np.uint32) >> 16).astype(np.uint16)


MX_HAND_WORKED = [
    # (block values, E8M0 byte, codes of the listed values)
    ([448.0], 127, [0x7E]),                        # amax 448: s = 0, 448 itself
    ([1.0, -0.5, 0.25], 119, [0x78, 0xF0, 0x68]),  # s = -8: 256, -128, 64
    ([1.0, -0.5, 0.25, 3.0], 120, [0x70, 0xE8, 0x60, 0x7C]),  # s = -7: 128, -64, 32, 384
    ([500.0, 1.0], 127, [0x7E, 0x38]),             # s = 0: 500 saturates to 448; 1.0 stays
    ([], 0, []),                                   # all zero: byte 0, zero codes
    ([2.0 ** -130], 0, [0x20]),                    # s clamps at -127: 2^-130 / 2^-127 = 2^-3
    ([2.0 ** 127, 2.0 ** 118], 246, [0x78, 0x30]), # s = 119: 2^8 = 256 and 2^-1
]


def test_mx_hand_worked_blocks():
    for vals, byte, codes in MX_HAND_WORKED:
        x = _bf16_vec(vals)[None, :]
        q, s = oracle.mx_quant_rows(x)
        assert s[0, 0] == byte, (vals, s[0, 0])
        assert [int(c) for c in q[0, : len(codes)]] == codes, (vals, [hex(c) for c in q[0]])
        assert not q[0, len(codes):].any()
    assert oracle.e8m0_to_f64(127) == 1.0 and oracle.e8m0_to_f64(0) == 2.0 ** -127
    assert oracle.e8m0_to_f64(254) == 2.0 ** 127 and math.isnan(oracle.e8m0_to_f64(255))


def check_mx_quant_rows(qr, rng):
    x = bf16((rng.standard_normal((6, 128)) * np.exp(rng.uniform(-8, 8, (6, 4)).repeat(32, 1)))
             .astype(np.float32))
    x[2, 32:64] = 0                               # an all-zero block
    q, s = qr(x)
    assert q.shape == x.shape and s.shape == (6, 4) and s.dtype == np.uint8
    xf = ig.bf16_bits_to_f64(x)
    X = np.ldexp(1.0, s.astype(np.int64) - 127).repeat(32, 1)
    deq = np.vectorize(oracle.e4m3_to_f64)(q) * X
    scaled = np.abs(xf) / X
    # each block's largest magnitude lands in [256, 512) before conversion
    for t in range(6):
        for b in range(4):
            blk = scaled[t, 32 * b: 32 * b + 32]
            if blk.max() == 0:
                assert s[t, b] == 0 and not q[t, 32 * b: 32 * b + 32].any()
            else:
                assert 256.0 <= blk.max() < 512.0, (t, b, blk.max())
    # reconstruction within E4M3's error (half a step of the 3-bit mantissa,
    # half the subnormal step below 2^-6), except the values above 448 that
    # saturate
    sat = scaled > 448.0
    err = np.abs(deq - xf)
    ok = err <= 2.0 ** -4 * np.abs(xf) + 2.0 ** -10 * X
    assert np.all(ok | sat)
    assert np.all(np.abs(deq[sat]) == 448.0 * X[sat])
    # without saturation the codes are torch's round-to-nearest-even E4M3 cast
    import torch
    v = torch.from_numpy((xf / X).astype(np.float32)[~sat])
    assert np.array_equal(q[~sat], v.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_mx_quant_rows_and_cols():
    check_mx_quant_rows(oracle.mx_quant_rows, np.random.default_rng(41))
    rng = np.random.default_rng(42)
    W = bf16((rng.standard_normal((3, 96, 40)) / 10).astype(np.float32))
    q, s = oracle.mx_quant_cols(W)
    # blocks run along d: the columns of W[e] are the rows of W[e].T
    for e in range(3):
        qe, se = oracle.mx_quant_rows(np.ascontiguousarray(W[e].T))
        assert np.array_equal(q[e], qe) and np.array_equal(s[e], se)
    # a change inside one block changes that block's codes and scale only
    x = bf16(rng.standard_normal((1, 96)).astype(np.float32))
    q0, s0 = oracle.mx_quant_rows(x)
    x2 = x.copy()
    x2[0, 40] = (np.array([1e3], np.float32).view(np.uint32) >> 16).astype(np.uint16)[0]
    q2, s2 = oracle.mx_quant_rows(x2)
    assert s2[0, 1] != s0[0, 1] and s2[0, 0] == s0[0, 0] and s2[0, 2] == s0[0, 2]
    assert np.array_equal(q2[0, :32], q0[0, :32]) and np.array_equal(q2[0, 64:], q0[0, 64:])
    with pytest.raises(oracle.OracleError):
        oracle.mx_quant_rows(bf16(np.zeros((1, 48), np.float32)))


def check_gemm_mx(gemm, rng):
    T, k, E, D, N = 19, 2, 4, 96, 40
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _, offsets = oracle.route_counts(topk, E)
    perm, _ = oracle.build_perm(topk, E, offsets)
    x = bf16((rng.standard_normal((T, D)) * np.exp(rng.uniform(-3, 3, (T, 3)).repeat(32, 1)))
             .astype(np.float32))
    W = bf16((rng.standard_normal((E, D, N)) / 8).astype(np.float32))
    xq, sx = oracle.mx_quant_rows(x)
    wq, sw = oracle.mx_quant_cols(W)
    out = gemm(xq, sx, perm, offsets, wq, sw, k, np.arange(T * k))
    deq = np.vectorize(oracle.e4m3_to_f64)
    xd = deq(xq) * np.ldexp(1.0, sx.astype(np.int64) - 127).repeat(32, 1)
    wd = deq(wq) * np.ldexp(1.0, sw.astype(np.int64) - 127).repeat(32, 2)   # [E, N, D]
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        ref = xd[perm[lo:hi] // k] @ wd[e].T
        assert np.all(np.abs(out[lo:hi] - ref) <= 1e-12 * (np.abs(xd[perm[lo:hi] // k]) @ np.abs(wd[e]).T))
    # one element by brute force with exact summation
    j, n = 5, 7
    e = int(np.searchsorted(offsets, j, side="right") - 1)
    t = perm[j] // k
    assert math.isclose(out[j, n], math.fsum(xd[t] * wd[e, n]), rel_tol=1e-12, abs_tol=1e-300)
    # and it approximates the bf16 GEMM within E4M3's precision
    bf = oracle.gemm_rows(x, perm, offsets, W, k, np.arange(T * k))
    assert np.abs(out - bf).max() < 0.1 * np.abs(bf).max()


def test_gemm_mx_pins():
    check_gemm_mx(oracle.gemm_mx_rows, np.random.default_rng(43))


def test_planted_mx_mistakes_are_caught():
    def emax7(x):                         # s = floor(log2 amax) - 7: the block max lands in [128, 256)
        q, s = oracle.mx_quant_rows(x)
        xf = ig.bf16_bits_to_f64(x)
        s = np.where(s > 0, s + 1, s).astype(np.uint8)
        X = np.ldexp(1.0, s.astype(np.int64) - 127).repeat(32, 1)
        q = np.array([[oracle.f32_to_e4m3(float(v)) for v in row] for row in xf / X], np.uint8)
        return q, s

    def ceil_exp(x):                      # ceil instead of floor: only exact powers of two agree
        q, s = oracle.mx_quant_rows(x)
        xf = ig.bf16_bits_to_f64(x)
        amax = np.abs(xf).reshape(x.shape[0], -1, 32).max(2)
        s2 = np.where(amax > 0, np.ceil(np.log2(np.where(amax > 0, amax, 1))) - 8 + 127, 0)
        s2 = s2.astype(np.uint8)
        X = np.ldexp(1.0, s2.astype(np.int64) - 127).repeat(32, 1)
        q = np.array([[oracle.f32_to_e4m3(float(v)) for v in row] for row in xf / X], np.uint8)
        return q, s2

    def scale_once(xq, sx, perm, offsets, wq, sw, k, rows):   # W's block scales dropped
        return oracle.gemm_mx_rows(xq, sx, perm, offsets, wq, np.full_like(sw, 127), k, rows)

    def blocks_along_n(xq, sx, perm, offsets, wq, sw, k, rows):  # scale of block n // 32, not d // 32
        E, N, nb = sw.shape
        sw2 = np.ascontiguousarray(np.broadcast_to(sw[:, :, :1], sw.shape))
        return oracle.gemm_mx_rows(xq, sx, perm, offsets, wq, sw2, k, rows)

    for bad in (emax7, ceil_exp):
        with pytest.raises(AssertionError):
            check_mx_quant_rows(bad, np.random.default_rng(41))
    for bad in (scale_once, blocks_along_n):
        with pytest.raises(AssertionError):
            check_gemm_mx(bad, np.random.default_rng(43))
