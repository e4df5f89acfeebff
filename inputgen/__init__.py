"""Seeded synthetic inputs for the MoE token-dispatch + expert-GEMM path.

Produces activations ``x[T, D]`` (bf16 bit patterns in ``uint16``), expert
weights ``W[E, D, D_expert]`` (bf16 bits) and routed expert indices
``topk_idx[T, k]`` (int32). It holds none of the dispatch or GEMM arithmetic;
the CPU oracle and the CUDA path both consume the bytes it returns.

The workloads are those of the expert-parallel token-dispatch + GEMM result
of "Loads and Loads of Fluffy Kittens" (section "Key claims", Fig. 17:
top_k=8, num_experts=256, D=7168, D_expert=2048), plus smaller and skewed
variants of the same shape family. Recipe (all seeded, seed 0 by default):

* x ~ N(0, 1), W ~ N(0, 1) / sqrt(D), both rounded float64 -> float32 -> bf16;
* router logits ~ N(0, 1) (+ a per-expert bias -s*ln(e+1) for the skewed
  case), topk_idx[t, s] = expert with the s-th largest logit of token t;
* x, W and the logits use separate counter-based splitmix64 streams, so a
  single expert's W can be produced without the rest.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libinputgen.so")

STREAM_X = 1
STREAM_W = 2
STREAM_LOGITS = 3
STREAM_GATES = 4
STREAM_SRC = 5


def build(force: bool = False) -> str:
    """Compile the generator into a shared library next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.ig_stream_key.restype = ctypes.c_uint64
        lib.ig_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.ig_splitmix64_at.restype = ctypes.c_uint64
        lib.ig_splitmix64_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.ig_normal_at.restype = ctypes.c_double
        lib.ig_normal_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.ig_f32_to_bf16.restype = ctypes.c_uint16
        lib.ig_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.ig_fill_normal_bf16.restype = ctypes.c_int
        lib.ig_fill_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                            ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p,
                                            ctypes.c_int]
        lib.ig_topk_routing.restype = ctypes.c_int
        lib.ig_topk_routing.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                                        ctypes.c_void_p, ctypes.c_int]
        lib.ig_logits_f32.restype = ctypes.c_int
        lib.ig_logits_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                      ctypes.c_int64, ctypes.c_double, ctypes.c_void_p]
        lib.ig_weights_f32.restype = ctypes.c_int
        lib.ig_weights_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_void_p]
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


# ---------------------------------------------------------------- primitives
def splitmix64_at(state: int, i: int) -> int:
    return int(_L().ig_splitmix64_at(state, i))


def stream_key(seed: int, stream: int) -> int:
    return int(_L().ig_stream_key(seed, stream))


def normal_at(seed: int, stream: int, i: int) -> float:
    return float(_L().ig_normal_at(stream_key(seed, stream), i))


def f32_to_bf16_bits(v: float) -> int:
    return int(_L().ig_f32_to_bf16(v))


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def normal_bf16(seed: int, stream: int, start: int, n: int, scale: float = 1.0,
                out: np.ndarray | None = None, threads: int | None = None) -> np.ndarray:
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    if n:
        _L().ig_fill_normal_bf16(seed, stream, start, n, float(scale), out.ctypes.data,
                                 threads or default_threads())
    return out


def topk_routing(seed: int, T: int, E: int, k: int, zipf_s: float = 0.0,
                 threads: int | None = None) -> np.ndarray:
    out = np.empty((T, k), dtype=np.int32)
    if T:
        rc = _L().ig_topk_routing(seed, STREAM_LOGITS, T, E, k, float(zipf_s), out.ctypes.data,
                                  threads or default_threads())
        if rc != 0:
            raise ValueError(f"topk_routing failed ({rc})")
    return out


# ------------------------------------------------------------------ configs
@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    E: int
    k: int
    De: int
    zipf_s: float = 0.0
    seed: int = 0
    desc: str = ""

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def flops(self) -> int:
        return 2 * self.T * self.k * self.D * self.De


WORKLOADS = {
    "tiny": Workload("tiny", 64, 256, 8, 2, 128,
                     desc="tiny MoE dispatch+GEMM, top-2 of 8 experts"),
    "mid": Workload("mid", 4096, 2048, 64, 6, 1408,
                    desc="mid MoE, top-6 of 64 experts, near-uniform load"),
    "ep": Workload("ep", 8192, 7168, 256, 8, 2048,
                   desc="expert-parallel shape top_k=8, 256 experts, D=7168, D_expert=2048"),
    "skew": Workload("skew", 8192, 7168, 256, 8, 2048, zipf_s=1.2,
                     desc="same shape, router logits biased by -1.2*ln(e+1) (Zipf s=1.2)"),
    "decode": Workload("decode", 128, 7168, 256, 8, 2048,
                       desc="decode-like: 128 tokens, weight-bound"),
    # profiling case: the "ep" shape cut to 32 experts and 1024 tokens, so
    # rows per expert (~256) and every tile shape stay those of "ep" while
    # W (0.94 GB) still exceeds L2
    "ep32": Workload("ep32", 1024, 7168, 32, 8, 2048,
                     desc="ep shape with 32 experts and 1024 tokens (profiling size)"),
    # profiling case for the decode workload: ~4 rows per expert as in
    # "decode", 32 experts so that W (0.94 GB) still exceeds L2
    "decode32": Workload("decode32", 16, 7168, 32, 8, 2048,
                         desc="decode shape with 32 experts and 16 tokens (profiling size)"),
    # profiling case for the skewed workload: the Zipf-biased routing of "skew"
    # over 32 experts and 1024 tokens, so one expert holds most tokens (a
    # heavy expert of several row groups next to light and empty ones) while
    # W (0.94 GB) still exceeds L2
    "skew32": Workload("skew32", 1024, 7168, 32, 8, 2048, zipf_s=1.2,
                       desc="skewed routing over 32 experts and 1024 tokens (profiling size)"),
}


def custom(T, D, E, k, De, zipf_s=0.0, seed=0, name="custom") -> Workload:
    return Workload(name, T, D, E, k, De, zipf_s, seed)


@dataclass
class Case:
    wl: Workload
    x: np.ndarray            # uint16 [T, D] (bf16 bits)
    topk: np.ndarray         # int32 [T, k]
    W: np.ndarray | None     # uint16 [E, D, De] (bf16 bits); may be partially filled
    w_filled: set = field(default_factory=set)


def make_x(wl: Workload, threads=None) -> np.ndarray:
    return normal_bf16(wl.seed, STREAM_X, 0, wl.T * wl.D, 1.0, threads=threads).reshape(wl.T, wl.D)


def w_scale(wl: Workload) -> float:
    return 1.0 / float(np.sqrt(wl.D))


def fill_w_expert(wl: Workload, W: np.ndarray, e: int, threads=None) -> None:
    n = wl.D * wl.De
    normal_bf16(wl.seed, STREAM_W, e * n, n, w_scale(wl), out=W[e].reshape(-1), threads=threads)


def make_W(wl: Workload, threads=None, experts=None) -> np.ndarray:
    """Full W, or (experts given) a zero array with only those experts filled.

    np.zeros maps untouched pages lazily, so a partially filled W costs only
    the memory of the experts that are filled.
    """
    if experts is None:
        return normal_bf16(wl.seed, STREAM_W, 0, wl.E * wl.D * wl.De, w_scale(wl),
                           threads=threads).reshape(wl.E, wl.D, wl.De)
    W = np.zeros((wl.E, wl.D, wl.De), dtype=np.uint16)
    for e in sorted(set(int(v) for v in experts)):
        fill_w_expert(wl, W, e, threads)
    return W


def make_topk(wl: Workload, threads=None) -> np.ndarray:
    return topk_routing(wl.seed, wl.T, wl.E, wl.k, wl.zipf_s, threads)


def make_logits(wl: Workload) -> np.ndarray:
    """float32 [T, E] router logits (N(0,1), plus the Zipf bias when set)."""
    out = np.empty((wl.T, wl.E), dtype=np.float32)
    if wl.T:
        _L().ig_logits_f32(wl.seed, STREAM_LOGITS, wl.T, wl.E, float(wl.zipf_s), out.ctypes.data)
    return out


def make_gates(wl: Workload) -> np.ndarray:
    """float32 [T, k] positive weights summing to one per token (combine input)."""
    out = np.empty((wl.T, wl.k), dtype=np.float32)
    if wl.T:
        _L().ig_weights_f32(wl.seed, STREAM_GATES, wl.T, wl.k, out.ctypes.data)
    return out


def make_src(wl: Workload, C: int, threads=None) -> np.ndarray:
    """bf16 bits [T*k, C] ~ N(0,1): expert outputs in sorted row order (combine input)."""
    return normal_bf16(wl.seed, STREAM_SRC, 0, wl.R * C, 1.0, threads=threads).reshape(wl.R, C)


def make_case(wl: Workload | str, with_W: bool = True, threads=None) -> Case:
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    x = make_x(wl, threads)
    topk = make_topk(wl, threads)
    W = make_W(wl, threads) if with_W else None
    return Case(wl, x, topk, W, set(range(wl.E)) if with_W else set())
