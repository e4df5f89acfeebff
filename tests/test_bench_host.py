"""Host-side logic of bench.py (CPU only): max-over-ranks timing with two
gloo ranks, the byte accounting and the JSON line of the reference arm."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import inputgen as ig


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        v = bench.max_over_ranks(1.5 + rank)   # rank 1 is the slow one
        bench.barrier()
        q.put((rank, v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25


def test_workload_bytes_counts_only_touched_experts():
    wl = ig.custom(T=4, D=16, E=5, k=2, De=8)
    counts = np.array([3, 0, 5, 0, 0])
    b = bench.workload_bytes(wl, counts)
    assert b["experts_touched"] == 2
    assert b["w_touched"] == 2 * 16 * 8 * 2
    assert b["x_gathered"] == 8 * 16 * 2 and b["out"] == 8 * 8 * 2
    assert b["x_unique"] == 4 * 16 * 2   # each token row once: a lower bound, not in the sum


def test_reference_arm_line(capsys):
    # the tiny workload keeps this fast; the line keeps the contract's keys
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    import json
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
    assert line["steps"] == 2 and line["warmup"] == 3


def test_profiled_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """traffic comes from profiles/<prefix>_<workload>.md (else its smaller
    stand-in, scaled) only while the recorded code fingerprint matches: an
    edit of comments or layout keeps it, a change of code drops it."""
    prof = tmp_path / "profiles"
    src_dir = tmp_path / "moe_token_dispatch_gb300" / "csrc"
    prof.mkdir()
    src_dir.mkdir(parents=True)
    (src_dir / "k.cu").write_text("kernel v1;\n")
    digest = bench.source_digest(str(src_dir / "k.cu"))
    (prof / "kk_ep32.md").write_text(f"kernel_code_sha256_16: {digest}\n"
                                     "traffic_bytes_per_launch: 1.0e+09\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("ep", prefix="kk", src="k.cu") == 1.0e9 * 256 / 32
    (prof / "kk_ep.md").write_text(f"kernel_code_sha256_16: {digest}\n"
                                   "traffic_bytes_per_launch: 3.0e+09\n")
    assert bench.profiled_traffic("ep", prefix="kk", src="k.cu") == 3.0e9   # direct capture wins
    (src_dir / "k.cu").write_text("// a note\nkernel   v1; /* more */\n")   # comments only
    assert bench.profiled_traffic("ep", prefix="kk", src="k.cu") == 3.0e9
    (src_dir / "k.cu").write_text("kernel v2;\n")                           # code changed
    assert bench.profiled_traffic("ep", prefix="kk", src="k.cu") is None


def test_committed_profiles_carry_hash_and_traffic():
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pdir = os.path.join(root, "profiles")
    for name in os.listdir(pdir):
        if name == "launches_ep.md":
            continue
        text = open(os.path.join(pdir, name)).read()
        assert re.search(r"kernel_code_sha256_16: [0-9a-f]{16}", text), name
        assert re.search(r"traffic_bytes_per_launch: [0-9.eE+]+", text), name
        assert "ncu " in text and "--clock-control none" in text, name


def test_code_fingerprint_ignores_comments_not_strings():
    a = 'asm("mov.u32 %0, 1; // not a comment"); int x = 1; // note\n/* block */ char c = \'/\';'
    b = 'asm("mov.u32 %0, 1; // not a comment");\n  int x = 1;\n char c = \'/\';'
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(a.replace("1; //", "2; //"))


def test_binding_roofline_picks_the_slower_limit():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0}
    # 1 GB at 1000 GB/s = 1 ms; 50 TFLOP at 100 TFLOP/s = 0.5 s: tensor binds
    r = bench.binding_roofline(50e12, 1e9, 1000.0, peaks)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - 0.5) < 1e-12 and abs(r["roofline_ms"] - 500.0) < 1e-9
    assert abs(r["achieved"] - 50.0) < 1e-9 and r["peak"] == 100.0
    # 10 GB (10 ms at HBM) against 0.1 TFLOP (1 ms): HBM binds; kernel took 20 ms
    r = bench.binding_roofline(1e11, 1e10, 20.0, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - 0.5) < 1e-12 and abs(r["achieved"] - 500.0) < 1e-9
    assert abs(r["tensor"]["frac"] - 0.05) < 1e-12


def test_both_arms_describe_the_workload_alike():
    # the reference arm and ours print config_of(wl) unchanged
    import inspect
    src = inspect.getsource(bench.run_ours)
    assert '"config": config_of(wl),' in src
    assert '"config": config_of(wl),' in inspect.getsource(bench.run_reference)
    assert set(bench.OTHER_WORKLOADS) == {"tiny", "mid", "skew", "decode"}
