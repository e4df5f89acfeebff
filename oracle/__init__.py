"""CPU oracle for MoE token dispatch + expert GEMM. TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. The product path (the
``moe_token_dispatch_gb300`` package and its CUDA library) never imports,
links or calls it, and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, float64); this module only
marshals numpy arrays. What each step computes, following the expert-parallel
"token-dispatch + GEMM" of "Loads and Loads of Fluffy Kittens" (section "Key
claims", Fig. 17) restated for one device:

* ``route_counts``  -- tokens routed to each expert, and the exclusive
  prefix sum of those counts (``offsets[E] == T*k``);
* ``build_perm``    -- flat routing indices ``t*k+s`` grouped by expert, in
  increasing ``t*k+s`` inside each expert; and its inverse;
* ``gemm_rows``     -- for sorted row ``j`` of expert ``e``:
  ``out[j, n] = sum_d x[perm[j] // k, d] * W[e, d, n]`` in float64 from the
  bf16 inputs;
* ``combine``       -- ``y[t] = sum_s gates[t, s] * src[inv_perm[t*k+s]]``;
* ``router_topk``   -- the k largest logits per token (ties to the lower
  expert) and their softmax;
* ``quant_rows`` / ``quant_cols`` / ``gemm_fp8_rows`` -- E4M3 quantisation
  with one float32 scale per row of x and per output column of W, and the
  expert GEMM on the codes.

Parity status: the pages print no worked example, so no function here is
pinned to a value printed on the pages. Each is pinned instead by closed
forms, invariants, library routines and brute force in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2) into a shared library next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int64


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_route_counts.restype = ctypes.c_int
        lib.oracle_route_counts.argtypes = [_P, _I, _I, _I, _P, _P]
        lib.oracle_build_perm.restype = ctypes.c_int
        lib.oracle_build_perm.argtypes = [_P, _I, _I, _I, _P, _P, _P]
        lib.oracle_expert_of_row.restype = ctypes.c_int64
        lib.oracle_expert_of_row.argtypes = [_P, _I, _I]
        lib.oracle_combine.restype = ctypes.c_int
        lib.oracle_combine.argtypes = [_P, _P, _P, _I, _I, _I, _P]
        lib.oracle_router_topk.restype = ctypes.c_int
        lib.oracle_router_topk.argtypes = [_P, _I, _I, _I, _P, _P]
        lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_quant_rows.restype = None
        lib.oracle_quant_rows.argtypes = [_P, _I, _I, _P, _P]
        lib.oracle_quant_cols.restype = None
        lib.oracle_quant_cols.argtypes = [_P, _I, _I, _I, _P, _P]
        lib.oracle_gemm_fp8_rows.restype = ctypes.c_int
        lib.oracle_e8m0_to_f64.restype = ctypes.c_double
        lib.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_mx_quant_rows.restype = ctypes.c_int
        lib.oracle_mx_quant_rows.argtypes = [_P, _I, _I, _P, _P]
        lib.oracle_mx_quant_cols.restype = ctypes.c_int
        lib.oracle_mx_quant_cols.argtypes = [_P, _I, _I, _I, _P, _P]
        lib.oracle_gemm_mx_rows.restype = ctypes.c_int
        lib.oracle_gemm_mx_rows.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I, _P]
        lib.oracle_gemm_fp8_rows.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I,
                                             _P]
        lib.oracle_gemm_rows.restype = ctypes.c_int
        lib.oracle_gemm_rows.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I, _P,
                                         ctypes.c_int]
        _lib = lib
    return _lib


class OracleError(ValueError):
    pass


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def route_counts(topk: np.ndarray, E: int):
    """Return (counts int64[E], offsets int64[E+1])."""
    topk = _c(topk, np.int32)
    T, k = topk.shape
    counts = np.zeros(E, dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    rc = _L().oracle_route_counts(topk.ctypes.data, T, k, E, counts.ctypes.data,
                                  offsets.ctypes.data)
    if rc:
        raise OracleError("expert index outside [0, E)")
    return counts, offsets


def build_perm(topk: np.ndarray, E: int, offsets: np.ndarray):
    """Return (perm int64[T*k], inv_perm int64[T*k])."""
    topk = _c(topk, np.int32)
    T, k = topk.shape
    offsets = _c(offsets, np.int64)
    perm = np.full(T * k, -1, dtype=np.int64)
    inv = np.full(T * k, -1, dtype=np.int64)
    rc = _L().oracle_build_perm(topk.ctypes.data, T, k, E, offsets.ctypes.data,
                                perm.ctypes.data, inv.ctypes.data)
    if rc:
        raise OracleError("expert index outside [0, E)")
    return perm, inv


def expert_of_row(offsets: np.ndarray, j: int) -> int:
    offsets = _c(offsets, np.int64)
    return int(_L().oracle_expert_of_row(offsets.ctypes.data, offsets.size - 1, j))


def gemm_rows(x: np.ndarray, perm: np.ndarray, offsets: np.ndarray, W: np.ndarray, k: int,
              rows, threads: int | None = None) -> np.ndarray:
    """float64 [len(rows), De]: the expert GEMM for the listed sorted rows."""
    x = _c(x, np.uint16)
    W = np.asarray(W)
    assert W.dtype == np.uint16 and W.flags.c_contiguous
    T, D = x.shape
    E, D2, De = W.shape
    assert D2 == D
    perm = _c(perm, np.int64)
    offsets = _c(offsets, np.int64)
    rows = _c(np.asarray(rows).reshape(-1), np.int64)
    out = np.zeros((rows.size, De), dtype=np.float64)
    if rows.size:
        rc = _L().oracle_gemm_rows(x.ctypes.data, perm.ctypes.data, offsets.ctypes.data,
                                   W.ctypes.data, T, k, D, E, De, rows.ctypes.data, rows.size,
                                   out.ctypes.data, threads or max(1, os.cpu_count() or 1))
        if rc:
            raise OracleError("row outside every expert segment, or token out of range")
    return out


def gemm_all(x, perm, offsets, W, k, threads=None) -> np.ndarray:
    return gemm_rows(x, perm, offsets, W, k, np.arange(perm.size), threads)


def combine(src: np.ndarray, inv_perm: np.ndarray, gates: np.ndarray, T: int, k: int):
    """float64 [T, C]: y[t] = sum_s gates[t, s] * src[inv_perm[t*k+s]] (s ascending)."""
    src = _c(src, np.uint16)
    R, C = src.shape
    assert R == T * k
    inv = _c(inv_perm, np.int64).reshape(-1)
    g = _c(gates, np.float64).reshape(-1)
    y = np.zeros((T, C), dtype=np.float64)
    if T:
        rc = _L().oracle_combine(src.ctypes.data, inv.ctypes.data, g.ctypes.data, T, k, C,
                                 y.ctypes.data)
        if rc:
            raise OracleError("inv_perm entry outside [0, T*k)")
    return y


def router_topk(logits: np.ndarray, k: int):
    """(topk int64 [T, k], gates float64 [T, k]) from float32 logits [T, E]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    topk = np.zeros((T, k), dtype=np.int64)
    gates = np.zeros((T, k), dtype=np.float64)
    if T:
        rc = _L().oracle_router_topk(logits.ctypes.data, T, E, k, topk.ctypes.data,
                                     gates.ctypes.data)
        if rc:
            raise OracleError("k outside [1, E]")
    return topk, gates


def f32_to_e4m3(v: float) -> int:
    return int(_L().oracle_f32_to_e4m3(v))


def e4m3_to_f64(c: int) -> float:
    return float(_L().oracle_e4m3_to_f64(c))


def quant_rows(x: np.ndarray):
    """E4M3 codes [T, D] (uint8) and fp32 scales [T] of the rows of bf16 x."""
    x = _c(x, np.uint16)
    T, D = x.shape
    q = np.zeros((T, D), dtype=np.uint8)
    s = np.zeros(T, dtype=np.float32)
    if T:
        _L().oracle_quant_rows(x.ctypes.data, T, D, q.ctypes.data, s.ctypes.data)
    return q, s


def quant_cols(W: np.ndarray):
    """E4M3 codes [E, N, D] (each output column contiguous) and fp32 scales
    [E, N] of the columns of bf16 W [E, D, N]."""
    W = np.asarray(W)
    assert W.dtype == np.uint16 and W.flags.c_contiguous
    E, D, N = W.shape
    q = np.zeros((E, N, D), dtype=np.uint8)
    s = np.zeros((E, N), dtype=np.float32)
    _L().oracle_quant_cols(W.ctypes.data, E, D, N, q.ctypes.data, s.ctypes.data)
    return q, s


def gemm_fp8_rows(xq, sx, perm, offsets, wq, sw, k, rows) -> np.ndarray:
    """float64 [len(rows), N] of the FP8 expert GEMM from codes and scales."""
    xq = _c(xq, np.uint8)
    sx = _c(sx, np.float32)
    wq = np.asarray(wq)
    assert wq.dtype == np.uint8 and wq.flags.c_contiguous
    sw = _c(sw, np.float32)
    T, D = xq.shape
    E, N, D2 = wq.shape
    assert D2 == D
    perm = _c(perm, np.int64)
    offsets = _c(offsets, np.int64)
    rows = _c(np.asarray(rows).reshape(-1), np.int64)
    out = np.zeros((rows.size, N), dtype=np.float64)
    if rows.size and _L().oracle_gemm_fp8_rows(xq.ctypes.data, sx.ctypes.data, perm.ctypes.data,
                                               offsets.ctypes.data, wq.ctypes.data, sw.ctypes.data,
                                               T, k, D, E, N, rows.ctypes.data, rows.size,
                                               out.ctypes.data):
        raise OracleError("row outside every expert segment, or token out of range")
    return out


def e8m0_to_f64(b: int) -> float:
    return float(_L().oracle_e8m0_to_f64(b))


def mx_quant_rows(x: np.ndarray):
    """MXFP8 of the rows of bf16 x [T, D] (D a multiple of 32): E4M3 codes
    [T, D] and E8M0 scale bytes [T, D // 32] (one per 32 consecutive d)."""
    x = _c(x, np.uint16)
    T, D = x.shape
    q = np.zeros((T, D), dtype=np.uint8)
    s = np.zeros((T, D // 32), dtype=np.uint8)
    if T and _L().oracle_mx_quant_rows(x.ctypes.data, T, D, q.ctypes.data, s.ctypes.data):
        raise OracleError("D must be a multiple of 32")
    return q, s


def mx_quant_cols(W: np.ndarray):
    """MXFP8 of the columns of bf16 W [E, D, N] (blocks of 32 along d): codes
    [E, N, D] (each output column contiguous) and E8M0 bytes [E, N, D // 32]."""
    W = np.asarray(W)
    assert W.dtype == np.uint16 and W.flags.c_contiguous
    E, D, N = W.shape
    q = np.zeros((E, N, D), dtype=np.uint8)
    s = np.zeros((E, N, D // 32), dtype=np.uint8)
    if _L().oracle_mx_quant_cols(W.ctypes.data, E, D, N, q.ctypes.data, s.ctypes.data):
        raise OracleError("D must be a multiple of 32")
    return q, s


def gemm_mx_rows(xq, sx, perm, offsets, wq, sw, k, rows) -> np.ndarray:
    """float64 [len(rows), N] of the MXFP8 expert GEMM from codes and E8M0
    block scales (mx_quant_rows of x, mx_quant_cols of W)."""
    xq, sx = _c(xq, np.uint8), _c(sx, np.uint8)
    wq, sw = np.asarray(wq), np.asarray(sw)
    assert wq.dtype == np.uint8 and wq.flags.c_contiguous
    assert sw.dtype == np.uint8 and sw.flags.c_contiguous
    T, D = xq.shape
    E, N, D2 = wq.shape
    assert D2 == D and sx.shape == (T, D // 32) and sw.shape == (E, N, D // 32)
    perm, offsets = _c(perm, np.int64), _c(offsets, np.int64)
    rows = _c(np.asarray(rows).reshape(-1), np.int64)
    out = np.zeros((rows.size, N), dtype=np.float64)
    if rows.size and _L().oracle_gemm_mx_rows(xq.ctypes.data, sx.ctypes.data, perm.ctypes.data,
                                              offsets.ctypes.data, wq.ctypes.data, sw.ctypes.data,
                                              T, k, D, E, N, rows.ctypes.data, rows.size,
                                              out.ctypes.data):
        raise OracleError("row outside every expert segment, token out of range or D % 32")
    return out


def bf16_to_f64(h: int) -> float:
    return float(_L().oracle_bf16_to_f64(h))


def run(topk, E, x=None, W=None, rows=None, threads=None):
    """Whole path on the CPU: counts, offsets, perm, inv_perm and (if x, W
    given) the GEMM for ``rows`` (all rows when None)."""
    topk = np.asarray(topk)
    counts, offsets = route_counts(topk, E)
    perm, inv = build_perm(topk, E, offsets)
    res = {"counts": counts, "offsets": offsets, "perm": perm, "inv_perm": inv}
    if x is not None and W is not None:
        k = topk.shape[1]
        if rows is None:
            rows = np.arange(perm.size)
        res["rows"] = np.asarray(rows, dtype=np.int64)
        res["out"] = gemm_rows(x, perm, offsets, W, k, rows, threads)
    return res
