#!/usr/bin/env python3
"""Benchmark: MoE token dispatch + expert GEMM on GB300.

One step = pk_moe_route_counts + pk_moe_build_perm + pk_moe_dispatch_gemm on
one batch of seeded synthetic input (the expert-parallel shape of "Loads and
Loads of Fluffy Kittens", "Key claims", Fig. 17: T=8192 tokens, D=7168,
E=256 experts, top_k=8, D_expert=2048). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload ep|skew|decode|mid|tiny]

``--impl reference`` times the CPU oracle (float64, all host cores) on a
bounded sample of the same workload. N > 1 (torchrun) runs one independent
replica per GPU: the path has no cross-GPU step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "dispatch+expert-GEMM TFLOP/s and % of GB300 BF16 peak at T=8192 D=7168 E=256 k=8"
UNIT = "TFLOP/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# source file and ncu summary prefix of each dispatch GEMM kernel
GEMM_KERNELS = {
    "single": ("dispatch_gemm.cu", "dispatch_gemm", "k_dispatch_gemm"),
    "pair": ("dispatch_gemm_pair.cu", "dispatch_gemm_pair", "k_dispatch_gemm_pair"),
}
GEMM_SOURCE = os.path.join(ROOT, "moe_token_dispatch_gb300", "csrc", "dispatch_gemm.cu")


# --------------------------------------------------------------- utilities
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def strip_comments(text: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed: two
    sources with the same code (comments or layout edited) give the same
    text. String and character literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_digest(path=GEMM_SOURCE) -> str:
    """First 16 hex digits of the sha256 of a kernel source's code (comments
    and whitespace removed): the fingerprint an ncu summary records of the
    code it was captured on."""
    with open(path, encoding="utf-8") as f:
        return hashlib.sha256(strip_comments(f.read()).encode()).hexdigest()[:16]


# Workloads too large for a full ncu capture take the DRAM traffic of a smaller
# case with the same rows per expert and tile shapes, scaled by the units of
# work processed (experts touched): "ep" = 8 x "ep32"; "decode" touches 252 of
# its 256 experts, "decode32" all 32 of its experts.
TRAFFIC_SCALED_FROM = {"ep": ("ep32", 256 / 32), "decode": ("decode32", 252 / 32)}


def profiled_traffic(workload: str, kernel: str = "single", prefix: str | None = None,
                     src: str | None = None):
    """DRAM bytes per launch from the committed ncu summary
    profiles/<prefix>_<workload>.md, if it was taken on the current kernel
    source; else None. Defaults: the dispatch GEMM kernel `kernel`."""
    if prefix is None:
        src, prefix, _ = GEMM_KERNELS[kernel]
    # a capture of the workload itself, else of its smaller stand-in, scaled
    name, scale = workload, 1.0
    path = os.path.join(ROOT, "profiles", f"{prefix}_{name}.md")
    if not os.path.exists(path) and workload in TRAFFIC_SCALED_FROM:
        name, scale = TRAFFIC_SCALED_FROM[workload]
        path = os.path.join(ROOT, "profiles", f"{prefix}_{name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"kernel_code_sha256_16:\s*([0-9a-f]+)", text)
    src_path = os.path.join(ROOT, "moe_token_dispatch_gb300", "csrc", src)
    if not m or not s or s.group(1) != source_digest(src_path):
        return None
    return float(m.group(1)) * scale


def workload_bytes(wl, counts: np.ndarray) -> dict:
    R = wl.T * wl.k
    touched = int((counts > 0).sum())
    return {
        "x_gathered": R * wl.D * 2,
        "w_touched": touched * wl.D * wl.De * 2,
        "out": R * wl.De * 2,
        "indices": R * 4 + (wl.E + 1) * 4,
        "experts_touched": touched,
        # lower bound on x traffic (each token row once), not part of the sum
        "x_unique": wl.T * wl.D * 2,
    }


def binding_roofline(flops: float, alg_bytes: float, kernel_ms: float, peaks: dict,
                     tensor_peak: float | None = None) -> dict:
    """Roofline of one GEMM launch: the slower of its FLOPs at the tensor peak
    and its algorithmic bytes at the HBM peak binds; `frac` is that time over
    the measured kernel time (= achieved / peak in the binding unit)."""
    tp = tensor_peak or peaks["bf16_tflops"]
    t_tensor = flops / (tp * 1e12) * 1e3
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    sec = kernel_ms * 1e-3
    hbm = {"achieved": alg_bytes / sec / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": t_hbm / kernel_ms, "ms": t_hbm}
    tensor = {"achieved": flops / sec / 1e12, "peak": tp, "unit": "TFLOP/s",
              "frac": t_tensor / kernel_ms, "ms": t_tensor}
    b = hbm if t_hbm >= t_tensor else tensor
    return {"bound": "hbm" if b is hbm else "tensor", "achieved": b["achieved"], "peak": b["peak"],
            "unit": b["unit"], "frac": b["frac"], "roofline_ms": max(t_hbm, t_tensor),
            "kernel_ms": kernel_ms, "hbm": hbm, "tensor": tensor}


def config_of(wl) -> dict:
    return {
        "workload": f"{wl.name}: T={wl.T} D={wl.D} E={wl.E} top_k={wl.k} D_expert={wl.De}"
                    + (f" zipf_s={wl.zipf_s}" if wl.zipf_s else ""),
        "T": wl.T, "D": wl.D, "E": wl.E, "top_k": wl.k, "D_expert": wl.De,
        "routing": "top-k of N(0,1) router logits" + (f" + bias -{wl.zipf_s}*ln(e+1)" if wl.zipf_s else ""),
        "x": "bf16 N(0,1)", "W": "bf16 N(0,1)/sqrt(D)", "seed": wl.seed,
        "l2": f"inputs larger than L2: {wl.E * wl.D * wl.De * 2 / 1e9:.2f} GB of W streamed per step"
              if wl.E * wl.D * wl.De * 2 > 256e6 else "L2 flushed (512 MB write) between steps",
    }


# ------------------------------------------------------------ distributed
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.samples = []
        self.proc = None
        self.uuid = (gpu_uuid or "").lower().replace("gpu-", "")
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for t, s in self.samples if t0 <= t <= t1 + 0.15 and len(s) >= 9
                  and (not self.uuid or s[0].lower().replace("gpu-", "") == self.uuid)]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in inside for n, v in zip(names, s[5:9]) if v == "Active"})

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        mx = [num(s[2]) for s in inside if num(s[2]) is not None]
        pw = [num(s[3]) for s in inside if num(s[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------ CPU oracle
def oracle_sample(case, wl, seconds: float, threads: int):
    """Times the oracle on a bounded sample: full routing plus the GEMM of a
    sample of rows, sized to take about `seconds`. Returns (TFLOP/s, info)."""
    import oracle
    t0 = time.perf_counter()
    counts, offsets = oracle.route_counts(case.topk, wl.E)
    perm, _ = oracle.build_perm(case.topk, wl.E, offsets)
    t_route = time.perf_counter() - t0
    rng = np.random.default_rng(0)
    R = wl.T * wl.k
    # calibrate: one row per thread
    probe = rng.integers(0, R, size=threads)
    W = _ensure_w_rows(case, wl, offsets, probe)
    t0 = time.perf_counter()
    oracle.gemm_rows(case.x, perm, offsets, W, wl.k, probe, threads)
    t_probe = time.perf_counter() - t0
    per_row = t_probe / len(probe)
    n = int(max(threads, min(R, (seconds - t_route) / max(per_row, 1e-9))))
    rows = rng.integers(0, R, size=n)
    W = _ensure_w_rows(case, wl, offsets, rows)
    t0 = time.perf_counter()
    oracle.gemm_rows(case.x, perm, offsets, W, wl.k, rows, threads)
    t_gemm = time.perf_counter() - t0
    flops = 2.0 * wl.D * wl.De * n
    sec = t_route + t_gemm
    return flops / sec / 1e12, {"rows": n, "seconds": sec, "route_s": t_route}


def _ensure_w_rows(case, wl, offsets, rows):
    """Fills (lazily) the experts of the given sorted rows in a sparse W."""
    import inputgen as ig
    if case.W is None:
        case.W = np.zeros((wl.E, wl.D, wl.De), dtype=np.uint16)
    ex = np.searchsorted(offsets, rows, side="right") - 1
    for e in sorted(set(int(v) for v in ex)):
        if e not in case.w_filled:
            ig.fill_w_expert(wl, case.W, e)
            case.w_filled.add(e)
    return case.W


# ----------------------------------------------------------------- arms
def run_reference(args, wl):
    import inputgen as ig
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    threads = os.cpu_count() or 1
    case = ig.make_case(wl, with_W=False)
    steps, warm = args.steps, args.warmup
    per_step = max(0.05, min(2.0, 150.0 / (steps + warm)))
    for _ in range(warm):
        oracle_sample(case, wl, per_step, threads)
    vals, rows, secs = [], 0, 0.0
    for _ in range(steps):
        v, info = oracle_sample(case, wl, per_step, threads)
        vals.append(v)
        rows += info["rows"]
        secs += info["seconds"]
    value = 2.0 * wl.D * wl.De * rows / secs / 1e12
    sample = (f"per step: full routing of {wl.T * wl.k} entries + float64 GEMM of ~{rows // steps} "
              f"random sorted rows (of {wl.T * wl.k}), {steps} steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": 1000.0 * secs / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def run_ours(args, wl):
    import torch
    import inputgen as ig
    import moe_token_dispatch_gb300 as pk
    pk.pk_moe_set_gemm_kernel({"auto": pk.PK_GEMM_KERNEL_AUTO, "single": pk.PK_GEMM_KERNEL_SINGLE,
                               "pair": pk.PK_GEMM_KERNEL_PAIR}[args.gemm_kernel])

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    case = ig.make_case(wl, with_W=True)
    W_host = case.W

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    x = to_dev(case.x)
    W = to_dev(W_host)
    topk = torch.from_numpy(case.topk).to(dev)
    md = pk.MoeDispatch(wl.T, wl.k, wl.E, wl.D, wl.De, device=dev, with_inv_perm=True)
    R = wl.T * wl.k
    flops = 2.0 * R * wl.D * wl.De
    flush = None
    if wl.E * wl.D * wl.De * 2 <= 256e6:
        flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step(ev=None, sev=None):
        if sev is not None:
            sev[0].record(stream)
        md.route(topk, stream)
        if ev is not None:
            ev[0].record(stream)
        md.gemm(x, W, stream)
        if ev is not None:
            ev[1].record(stream)
        if sev is not None:
            sev[1].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
        if flush is not None:
            flush.fill_(1)
    torch.cuda.synchronize()
    if md.status_code() != 0:
        raise RuntimeError(f"device status {pk.pk_status_str(md.status_code())}")
    counts = md.counts.cpu().numpy()

    try:
        gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_uuid = None
    sampler = ClockSampler(gpu_uuid) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)

    K = args.steps
    gemm_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    # with an L2 flush between steps, each step is timed by its own events
    step_ev = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(K)] if flush is not None else [None] * K)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    start.record(stream)
    for i in range(K):
        step(gemm_ev[i], step_ev[i])
        if flush is not None:
            flush.fill_(1)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    wall1 = time.time()
    total_ms = start.elapsed_time(end)
    gemm_ms = [a.elapsed_time(b) for a, b in gemm_ev]
    if flush is not None:
        # the flushes between steps are not part of the work
        total_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    if md.status_code() != 0:
        raise RuntimeError(f"device status {pk.pk_status_str(md.status_code())}")
    step_ms = max_over_ranks(total_ms / K)
    gemm_avg_ms = max_over_ranks(sum(gemm_ms) / K)

    # Workloads that fit in L2 are timed above with L2 flushed between steps;
    # the same steps with L2 left warm are reported beside them. The stream
    # is held for a moment first so that the host has queued every step
    # before the first runs (these steps are shorter than their launches).
    l2_warm = None
    if flush is not None:
        Kw = max(1, min(K, 200))
        torch.cuda.synchronize()
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(50_000_000)
        wa, wb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        wa.record(stream)
        for _ in range(Kw):
            step()
        wb.record(stream)
        torch.cuda.synchronize()
        if md.status_code() != 0:
            raise RuntimeError(f"device status {pk.pk_status_str(md.status_code())}")
        warm_ms = max_over_ranks(wa.elapsed_time(wb) / Kw)
        l2_warm = {"ms_per_step": warm_ms, "value": world * flops / (warm_ms * 1e-3) / 1e12,
                   "unit": UNIT, "steps": Kw}

    # ---- end to end through the public API, host buffers, copies timed:
    # every step copies x and topk_idx in from pinned host memory and its
    # output back; copy-in, compute and copy-out of consecutive steps overlap
    # on three streams (PipelinedDispatch)
    from moe_token_dispatch_gb300.pipeline import PipelinedDispatch
    x_h = torch.from_numpy(np.ascontiguousarray(case.x).view(np.int16)).view(torch.bfloat16).pin_memory()
    tk_h = torch.from_numpy(case.topk).pin_memory()
    pipe = PipelinedDispatch(wl.T, wl.k, wl.E, wl.D, wl.De, W, device=dev)
    Ke = max(1, min(K, 200))
    for i in range(3):
        pipe.submit(i, x_h, tk_h)
    pipe.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.s_in)
    for i in range(Ke):
        pipe.submit(i, x_h, tk_h)
    e1.record(pipe.s_out)
    pipe.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / Ke)
    if any(c != 0 for c in pipe.status_codes()):
        raise RuntimeError("device status set during the end-to-end run")
    del pipe

    peaks, peak_kind = load_peaks()
    # the other workloads, each with its own binding roofline and oracle sample
    others = {}
    if rank == 0 and not args.no_others:
        for name in OTHER_WORKLOADS:
            if name != wl.name:
                others[name] = measure_other(args, ig.WORKLOADS[name], wl, x, W, dev, stream,
                                             peaks, peak_kind)
    if sampler:
        sampler.stop()
    if rank != 0:
        return None

    b = workload_bytes(wl, counts)
    alg_bytes = b["x_gathered"] + b["w_touched"] + b["out"] + b["indices"]
    roof = binding_roofline(flops, alg_bytes, gemm_avg_ms, peaks)
    roof["tensor"]["peak_sustained"] = peaks.get("bf16_tflops_sustained")
    value = world * flops / (step_ms * 1e-3) / 1e12
    kernel = "pair" if args.gemm_kernel == "pair" else "single"
    traffic = profiled_traffic(wl.name, kernel)

    cpu_value, cpu_info = oracle_sample(case, wl, args.cpu_seconds, os.cpu_count() or 1)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(wl),
        "gemm_kernel": kernel,
        "pct_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
        "roofline": dict(roof, traffic=traffic, peak_kind=peak_kind,
                         kernel=GEMM_KERNELS[kernel][2], algorithmic_bytes=alg_bytes,
                         bytes_breakdown=b),
        "kernel_share": {GEMM_KERNELS[kernel][2]: gemm_avg_ms / step_ms},
        "cpu_baseline": {"value": cpu_value, "unit": UNIT, "cores": os.cpu_count() or 1,
                         "kind": "oracle",
                         "sample": f"full routing + float64 GEMM of {cpu_info['rows']} random "
                                   f"sorted rows of {R} ({cpu_info['seconds']:.1f} s)"},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": x.numel() * 2 + topk.numel() * 4,
                "d2h_bytes_per_step": R * wl.De * 2, "ms_per_step": e2e_ms,
                "note": "x and topk_idx copied in from pinned host memory and out copied back "
                        "every step, copies of neighbouring steps overlapped with compute on "
                        "three streams; W stays resident (layer weights)"},
        "gpu_launches": (pk.pk_moe_route_kernel_launches(wl.T, wl.k, wl.E) + 1) * K,
        "clocks": sampler.summary(wall0, wall1) if sampler else None,
    }
    if l2_warm is not None:
        line["l2_warm"] = l2_warm
    if others:
        line["workloads"] = others
    return line


# Workloads reported beside the headline one in the default bench line.
OTHER_WORKLOADS = ("tiny", "mid", "skew", "decode")


def measure_other(args, wl, head_wl, head_x, head_W, dev, stream, peaks, peak_kind):
    """One workload's step (route + dispatch GEMM) on resident inputs: CUDA-event
    times, binding roofline and a short oracle CPU sample. Workloads with the
    headline's weight shape and seed reuse its device W (the generator makes
    the same bytes), and the same x rows when D and the seed agree."""
    import torch
    import inputgen as ig
    import moe_token_dispatch_gb300 as pk

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    same_w = (wl.E, wl.D, wl.De, wl.seed) == (head_wl.E, head_wl.D, head_wl.De, head_wl.seed)
    same_x = (wl.D, wl.seed) == (head_wl.D, head_wl.seed) and wl.T <= head_wl.T
    x_host = ig.make_x(wl)
    topk_host = ig.make_topk(wl)
    x = head_x[: wl.T] if same_x else to_dev(x_host)
    W = head_W if same_w else to_dev(ig.make_W(wl))
    topk = torch.from_numpy(topk_host).to(dev)
    md = pk.MoeDispatch(wl.T, wl.k, wl.E, wl.D, wl.De, device=dev, with_inv_perm=True)
    flush = None
    if wl.E * wl.D * wl.De * 2 <= 256e6:
        flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    K = max(1, min(args.steps, 50))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for i in range(max(3, args.warmup) + K):
        e = ev[i - max(3, args.warmup)] if i >= max(3, args.warmup) else None
        if e:
            e[0].record(stream)
        md.route(topk, stream)
        if e:
            e[1].record(stream)
        md.gemm(x, W, stream)
        if e:
            e[2].record(stream)
            e[3].record(stream)
        if flush is not None:
            flush.fill_(1)
    torch.cuda.synchronize()
    if md.status_code() != 0:
        raise RuntimeError(f"device status {pk.pk_status_str(md.status_code())} ({wl.name})")
    step_ms = sum(e[0].elapsed_time(e[3]) for e in ev) / K
    gemm_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    counts = md.counts.cpu().numpy()
    b = workload_bytes(wl, counts)
    alg_bytes = b["x_gathered"] + b["w_touched"] + b["out"] + b["indices"]
    flops = float(wl.flops)
    roof = binding_roofline(flops, alg_bytes, gemm_ms, peaks)
    case = ig.Case(wl, x_host, topk_host, None)
    cpu_value, cpu_info = oracle_sample(case, wl, args.cpu_seconds_other, os.cpu_count() or 1)
    del md, flush
    return {
        "config": config_of(wl), "steps": K, "ms_per_step": step_ms,
        "value": flops / (step_ms * 1e-3) / 1e12, "unit": UNIT,
        "pct_bf16_peak": 100.0 * flops / (step_ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
        "roofline": dict(roof, peak_kind=peak_kind, kernel="k_dispatch_gemm",
                         traffic=profiled_traffic(
                             wl.name, "pair" if args.gemm_kernel == "pair" else "single"),
                         algorithmic_bytes=alg_bytes, flops=flops, bytes_breakdown=b),
        "cpu_baseline": {"value": cpu_value, "unit": UNIT, "cores": os.cpu_count() or 1,
                         "kind": "oracle",
                         "sample": f"full routing + float64 GEMM of {cpu_info['rows']} random "
                                   f"sorted rows of {wl.R} ({cpu_info['seconds']:.1f} s)"},
    }


def run_op(args, wl):
    """Timing of the kernels beside the dispatch + GEMM step (router top-k,
    combine, down-projection grouped GEMM) on the workload's shapes."""
    import torch
    import inputgen as ig
    import moe_token_dispatch_gb300 as pk
    pk.pk_moe_set_gemm_kernel({"auto": pk.PK_GEMM_KERNEL_AUTO, "single": pk.PK_GEMM_KERNEL_SINGLE,
                               "pair": pk.PK_GEMM_KERNEL_PAIR}[args.gemm_kernel])

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peaks, peak_kind = load_peaks()
    R = wl.T * wl.k

    def dev_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    # routing of the workload (GPU) for inv_perm / offsets
    md = pk.MoeDispatch(wl.T, wl.k, wl.E, 8, 8, device=dev)
    md.route(torch.from_numpy(ig.make_topk(wl)).to(dev))
    torch.cuda.synchronize()
    counts = md.counts.cpu().numpy()
    if args.op == "router":
        logits = torch.from_numpy(ig.make_logits(wl)).to(dev)
        idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device=dev)
        g = torch.empty((wl.T, wl.k), dtype=torch.float32, device=dev)
        fn = lambda: pk.pk_moe_router_topk(logits, wl.k, idx, g, stream)
        alg_bytes, flops = wl.T * wl.E * 4 + wl.T * wl.k * 8, 0
        metric = f"router top-k (fp32 logits -> top-{wl.k} of {wl.E} + softmax gates) at T={wl.T}"
    elif args.op == "combine":
        C = wl.D   # combine follows the down-projection: rows of the model width
        src = dev_bf16(ig.make_src(wl, C))
        gates = torch.from_numpy(ig.make_gates(wl)).to(dev)
        y = torch.empty((wl.T, C), dtype=torch.bfloat16, device=dev)
        fn = lambda: pk.pk_moe_combine(src, md.inv_perm, gates, wl.T, wl.k, y, md.status, stream)
        alg_bytes, flops = R * C * 2 + wl.T * C * 2 + R * 4 + R * 4, 0
        metric = f"combine y[t] = sum_s g[t,s] src[inv_perm[t*k+s]] at T={wl.T} k={wl.k} C={C}"
    elif args.op == "grouped_gemm":
        K, N = wl.De, wl.D   # down-projection: [R, D_expert] x W2[e] [D_expert, D]
        A = dev_bf16(ig.normal_bf16(wl.seed, 7, 0, R * K).reshape(R, K))
        W2 = dev_bf16(ig.make_W(ig.custom(T=wl.T, D=K, E=wl.E, k=wl.k, De=N, seed=wl.seed)))
        out = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: pk.pk_moe_grouped_gemm(A, md.offsets, W2, out, md.status, stream)
        touched = int((counts > 0).sum())
        alg_bytes = R * K * 2 + touched * K * N * 2 + R * N * 2 + (wl.E + 1) * 4
        flops = 2.0 * R * K * N
        metric = (f"down-projection grouped GEMM TFLOP/s at R={R} K={K} N={N} E={wl.E}")
    elif args.op == "fp8_gemm":
        # E4M3 codes with per-row / per-(expert, column) fp32 scales; the
        # weights are quantised once, outside the timed region, as a model
        # would at load time. The timed call is the FP8 dispatch GEMM.
        x = dev_bf16(ig.make_x(wl))
        W = dev_bf16(ig.make_W(wl))
        wq = torch.empty((pk.pk_moe_fp8_weight_bytes(wl.E, wl.D, wl.De),), dtype=torch.uint8,
                         device=dev)
        sw = torch.empty((wl.E, wl.De), dtype=torch.float32, device=dev)
        pk.pk_moe_quant_weights(W, wq, sw, stream)
        del W
        xq = torch.empty((wl.T, wl.D), dtype=torch.uint8, device=dev)
        sx = torch.empty((wl.T,), dtype=torch.float32, device=dev)
        pk.pk_moe_quant_rows(x, xq, sx, stream)
        out = torch.empty((R, wl.De), dtype=torch.bfloat16, device=dev)
        fn = lambda: pk.pk_moe_dispatch_gemm_fp8(xq, sx, md.perm, md.offsets, wq, sw, wl.k, out,
                                                 md.status, stream)
        qfn = lambda: pk.pk_moe_quant_rows(x, xq, sx, stream)
        touched = int((counts > 0).sum())
        alg_bytes = (R * wl.D + touched * wl.D * wl.De + R * wl.De * 2 + R * 4 + wl.T * 4
                     + touched * wl.De * 4 + (wl.E + 1) * 4)
        flops = 2.0 * R * wl.D * wl.De
        metric = (f"FP8 (E4M3) dispatch + expert GEMM TFLOP/s at T={wl.T} D={wl.D} E={wl.E} "
                  f"k={wl.k} D_expert={wl.De}")
    elif args.op == "mxfp8_gemm":
        # MXFP8: E4M3 codes with one E8M0 scale per 32 elements along D, on
        # block-scaled tensor-core MMAs; weights quantised once, outside the
        # timed region, as a model would at load time
        x = dev_bf16(ig.make_x(wl))
        W = dev_bf16(ig.make_W(wl))
        wq = torch.empty((pk.pk_moe_fp8_weight_bytes(wl.E, wl.D, wl.De),), dtype=torch.uint8,
                         device=dev)
        swb = torch.empty((pk.pk_moe_mx_weight_scale_bytes(wl.E, wl.D, wl.De),), dtype=torch.uint8,
                          device=dev)
        pk.pk_moe_quant_weights_mx(W, wq, swb, stream)
        del W
        xq = torch.empty((wl.T, wl.D), dtype=torch.uint8, device=dev)
        sx = torch.empty((wl.T, wl.D // 32), dtype=torch.uint8, device=dev)
        pk.pk_moe_quant_rows_mx(x, xq, sx, stream)
        out = torch.empty((R, wl.De), dtype=torch.bfloat16, device=dev)
        fn = lambda: pk.pk_moe_dispatch_gemm_mxfp8(xq, sx, md.perm, md.offsets, wq, swb, wl.E,
                                                   wl.De, wl.k, out, md.status, stream)
        qfn = lambda: pk.pk_moe_quant_rows_mx(x, xq, sx, stream)
        touched = int((counts > 0).sum())
        # codes and scale bytes of the touched experts' W, x codes and scale
        # bytes gathered per routed row, out, perm, offsets
        alg_bytes = (R * wl.D + R * (wl.D // 32) + touched * wl.D * wl.De
                     + touched * wl.De * (wl.D // 32) + R * wl.De * 2 + R * 4 + (wl.E + 1) * 4)
        flops = 2.0 * R * wl.D * wl.De
        metric = (f"MXFP8 (E4M3, E8M0 per 32) dispatch + expert GEMM TFLOP/s at T={wl.T} "
                  f"D={wl.D} E={wl.E} k={wl.k} D_expert={wl.De}")
    elif args.op == "fp8_grouped_gemm":
        # FP8 down-projection: h quantised per row, W2 per (expert, column), once
        K, N = wl.De, wl.D
        A = dev_bf16(ig.normal_bf16(wl.seed, 7, 0, R * K).reshape(R, K))
        W2 = dev_bf16(ig.make_W(ig.custom(T=wl.T, D=K, E=wl.E, k=wl.k, De=N, seed=wl.seed)))
        wq = torch.empty((pk.pk_moe_fp8_weight_bytes(wl.E, K, N),), dtype=torch.uint8, device=dev)
        sw = torch.empty((wl.E, N), dtype=torch.float32, device=dev)
        pk.pk_moe_quant_weights(W2, wq, sw, stream)
        del W2
        aq = torch.empty((R, K), dtype=torch.uint8, device=dev)
        sa = torch.empty((R,), dtype=torch.float32, device=dev)
        pk.pk_moe_quant_rows(A, aq, sa, stream)
        out = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: pk.pk_moe_grouped_gemm_fp8(aq, sa, md.offsets, wq, sw, out, md.status, stream)
        qfn = lambda: pk.pk_moe_quant_rows(A, aq, sa, stream)
        touched = int((counts > 0).sum())
        alg_bytes = R * K + touched * K * N + R * N * 2 + R * 4 + touched * N * 4 + (wl.E + 1) * 4
        flops = 2.0 * R * K * N
        metric = f"FP8 (E4M3) down-projection grouped GEMM TFLOP/s at R={R} K={K} N={N} E={wl.E}"
    else:
        raise SystemExit(f"unknown --op {args.op}")
    for _ in range(max(3, args.warmup)):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    if md.status_code() != 0:
        raise RuntimeError(f"device status {pk.pk_status_str(md.status_code())}")
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    med = ms[len(ms) // 2]
    gbs = alg_bytes / (med * 1e-3) / 1e9
    # ncu summaries of the kernels beside the step (prefix, source file)
    op_profile = {"combine": ("combine", "combine_router.cu"),
                  "grouped_gemm": ("grouped_gemm", "dispatch_gemm.cu"),
                  "fp8_gemm": ("fp8_dispatch_gemm", "dispatch_gemm.cu"),
                  "fp8_grouped_gemm": ("fp8_grouped_gemm", "dispatch_gemm.cu"),
                  "mxfp8_gemm": ("mxfp8_dispatch_gemm", "dispatch_gemm.cu")}.get(args.op)
    traffic = (profiled_traffic(wl.name, prefix=op_profile[0], src=op_profile[1])
               if op_profile else None)
    line = {"op": args.op, "metric": metric, "workload": wl.name, "ms_median": med,
            "ms_p10": ms[len(ms) // 10], "ms_p90": ms[(9 * len(ms)) // 10], "steps": args.steps,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": alg_bytes,
                         "traffic": traffic, "peak_kind": peak_kind}}
    if flops:
        tf = flops / (med * 1e-3) / 1e12
        line["value"], line["unit"] = tf, "TFLOP/s"
        # FP8 peak: the measured bf16 peak times the nominal fp8/bf16 ratio (4.5 / 2.25)
        fp8_op = args.op in ("fp8_gemm", "fp8_grouped_gemm", "mxfp8_gemm")
        tpeak = peaks["bf16_tflops"] * (2.0 if fp8_op else 1.0)
        line["roofline"]["tensor"] = {"achieved": tf, "peak": tpeak, "unit": "TFLOP/s",
                                      "frac": tf / tpeak}
        if fp8_op:
            line["roofline"]["tensor"]["peak_kind"] = "measured bf16 x 2 (nominal fp8/bf16)"
            qa, qb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            qa.record(stream)
            for _ in range(20):
                qfn()
            qb.record(stream)
            torch.cuda.synchronize()
            line["quant_rows_ms"] = qa.elapsed_time(qb) / 20
    else:
        line["value"], line["unit"] = gbs, "GB/s"
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs (one process each, launched by torchrun when > 1); "
                         "every rank runs its own replica")
    ap.add_argument("--steps", type=int, default=1000, help="timed steps")
    ap.add_argument("--warmup", type=int, default=20,
                    help="untimed steps before them (raised to 3 if fewer)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours",
                    help="ours: the CUDA path; reference: the CPU oracle on a bounded sample")
    ap.add_argument("--workload", default="ep",
                    help="tiny, mid, ep, skew, decode, or the profiling cuts ep32, decode32, skew32")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="oracle CPU sample of the headline workload (cpu_baseline)")
    ap.add_argument("--cpu-seconds-other", type=float, default=3.0,
                    help="oracle CPU sample per additional workload")
    ap.add_argument("--no-others", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--gemm-kernel", choices=["auto", "single", "pair"], default="auto",
                    help="dispatch GEMM kernel: auto (= single), single (one CTA per SM) or pair "
                         "(2-CTA clusters)")
    ap.add_argument("--op", default="dispatch_gemm",
                    choices=["dispatch_gemm", "router", "combine", "grouped_gemm", "fp8_gemm",
                             "fp8_grouped_gemm", "mxfp8_gemm"],
                    help="dispatch_gemm: the benchmark step; the others time one kernel")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)

    import inputgen as ig
    wl = ig.WORKLOADS[args.workload]
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            if rank != 0:
                return 0
    if args.op != "dispatch_gemm":
        line = run_op(args, wl) if rank == 0 else None
    elif args.impl == "reference":
        line = run_reference(args, wl)
    else:
        line = run_ours(args, wl)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
