"""Checks of the shared synthetic-input generator (CPU only)."""
import numpy as np
import pytest
import torch

import inputgen as ig


def test_splitmix64_known_answers():
    # Published splitmix64 outputs for a sequence whose state starts at 0.
    assert ig.splitmix64_at(0, 0) == 0xE220A8397B1DCDAF
    assert ig.splitmix64_at(0, 1) == 0x6E789E6AA1B965F4
    assert ig.splitmix64_at(0, 2) == 0x06C45D188009454F


def test_f32_to_bf16_matches_torch_rne():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # force exact ties (low 16 bits == 0x8000) for half of them
    bits[::2] = (bits[::2] & 0xFFFF0000) | 0x8000
    f = bits.view(np.float32)
    finite = np.isfinite(f)
    f = f[finite]
    ours = np.array([ig.f32_to_bf16_bits(float(v)) for v in f[:4000]], dtype=np.uint16)
    ref = torch.from_numpy(f[:4000].copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_normals_moments_and_ks():
    from scipy import stats
    z = np.array([ig.normal_at(0, ig.STREAM_X, i) for i in range(20000)])
    assert abs(z.mean()) < 0.03
    assert abs(z.std() - 1.0) < 0.03
    assert stats.kstest(z, "norm").pvalue > 1e-3


def test_bf16_fill_is_rounded_normal_and_thread_independent():
    a = ig.normal_bf16(0, ig.STREAM_W, 1000, 50000, 0.5, threads=1)
    b = ig.normal_bf16(0, ig.STREAM_W, 1000, 50000, 0.5, threads=7)
    assert np.array_equal(a, b)
    # element i is bf16(float32(0.5 * normal_at(start + i)))
    for i in (0, 1, 2, 999, 49999):
        v = 0.5 * ig.normal_at(0, ig.STREAM_W, 1000 + i)
        ref = torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
        assert int(a[i]) == ref


def test_streams_differ_and_seed_determinism():
    a = ig.normal_bf16(0, ig.STREAM_X, 0, 4096)
    b = ig.normal_bf16(0, ig.STREAM_W, 0, 4096)
    c = ig.normal_bf16(1, ig.STREAM_X, 0, 4096)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
    assert np.array_equal(a, ig.normal_bf16(0, ig.STREAM_X, 0, 4096))


def test_single_expert_slice_equals_full_W():
    wl = ig.custom(T=4, D=64, E=5, k=2, De=32)
    W = ig.make_W(wl)
    Wp = ig.make_W(wl, experts=[3])
    assert np.array_equal(W[3], Wp[3])
    assert not Wp[2].any()
    w = ig.bf16_bits_to_f64(W)
    assert abs(w.std() * np.sqrt(wl.D) - 1.0) < 0.05


@pytest.mark.parametrize("zipf", [0.0, 1.2])
def test_topk_is_sorted_distinct_top_of_logits(zipf):
    T, E, k = 37, 16, 4
    topk = ig.topk_routing(0, T, E, k, zipf)
    key = ig.stream_key(0, ig.STREAM_LOGITS)
    for t in range(T):
        logits = np.array([ig.normal_at(0, ig.STREAM_LOGITS, t * E + e) - zipf * np.log(e + 1)
                           for e in range(E)])
        order = sorted(range(E), key=lambda e: (-logits[e], e))[:k]
        assert list(topk[t]) == order
    assert key != 0


def test_topk_threads_independent_and_skew_shape():
    a = ig.topk_routing(0, 512, 64, 8, 1.2, threads=1)
    b = ig.topk_routing(0, 512, 64, 8, 1.2, threads=5)
    assert np.array_equal(a, b)
    cnt = np.bincount(a.ravel(), minlength=64)
    assert cnt[0] == cnt.max() and cnt[0] > 4 * np.median(cnt)
    u = ig.topk_routing(0, 512, 64, 8, 0.0)
    cu = np.bincount(u.ravel(), minlength=64)
    assert cu.max() < 3 * cu.mean()


def test_workload_table():
    ep = ig.WORKLOADS["ep"]
    assert (ep.T, ep.D, ep.E, ep.k, ep.De) == (8192, 7168, 256, 8, 2048)
    assert ep.flops == 2 * 8192 * 8 * 7168 * 2048
    assert ig.WORKLOADS["skew"].zipf_s == 1.2
