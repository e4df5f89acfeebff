"""ctypes binding of libpkmoe.so: argument marshalling only.

Each function has the name of the C entry point it calls and takes torch
tensors that must already live on the GPU with the dtype and layout the C ABI
documents (``include/pk_moe.h``). Nothing here computes any part of the path;
if the library is missing the import fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkmoe.so")

PK_OK = 0
PK_ERR_INVALID_ARG = 1
PK_ERR_UNSUPPORTED = 2
PK_ERR_CUDA = 3
PK_ERR_TIMEOUT = 4
PK_ERR_BAD_INDEX = 5
PK_ERR_CAPTURE = 6
PK_MAX_EXPERTS = 4096
PK_NOALLOC_SCRATCH_BYTES = 1 << 20
PK_ROUTER_MAX_EXPERTS = 1024
PK_GEMM_KERNEL_AUTO = 0
PK_GEMM_KERNEL_SINGLE = 1
PK_GEMM_KERNEL_PAIR = 2


class PkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {pk_status_str(code)} ({code})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run moe_token_dispatch_gb300._build.build() "
                          "(or __graft_entry__.build()) first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.pk_status_str.restype = ctypes.c_char_p
    lib.pk_status_str.argtypes = [ctypes.c_int]
    lib.pk_abi_version.restype = ctypes.c_int
    lib.pk_abi_version.argtypes = []
    lib.pk_moe_workspace_bytes.restype = SZ
    lib.pk_moe_workspace_bytes.argtypes = [I32, I32, I32]
    lib.pk_moe_route_counts.restype = ctypes.c_int
    lib.pk_moe_route_counts.argtypes = [P, I32, I32, I32, P, P, P, SZ, P, P]
    lib.pk_moe_build_perm.restype = ctypes.c_int
    lib.pk_moe_build_perm.argtypes = [P, I32, I32, I32, P, P, P, P, SZ, P, P]
    lib.pk_moe_dispatch_gemm.restype = ctypes.c_int
    lib.pk_moe_dispatch_gemm.argtypes = [P, P, P, P, I32, I32, I32, I32, I32, P, P, P]
    lib.pk_moe_route_noalloc.restype = ctypes.c_int
    lib.pk_moe_route_noalloc.argtypes = [P, I32, I32, I32, P, P, P, P, P, P]
    lib.pk_moe_grouped_gemm.restype = ctypes.c_int
    lib.pk_moe_grouped_gemm.argtypes = [P, P, P, I32, I32, I32, I32, P, P, P]
    lib.pk_moe_dispatch_gemm_fp8.restype = ctypes.c_int
    lib.pk_moe_dispatch_gemm_fp8.argtypes = [P, P, P, P, P, P, I32, I32, I32, I32, I32, P, P, P]
    lib.pk_moe_quant_rows.restype = ctypes.c_int
    lib.pk_moe_quant_rows.argtypes = [P, I32, I32, P, P, P]
    lib.pk_moe_fp8_weight_bytes.restype = SZ
    lib.pk_moe_fp8_weight_bytes.argtypes = [I32, I32, I32]
    lib.pk_moe_quant_weights.restype = ctypes.c_int
    lib.pk_moe_quant_weights.argtypes = [P, I32, I32, I32, P, P, P]
    lib.pk_moe_grouped_gemm_fp8.restype = ctypes.c_int
    lib.pk_moe_grouped_gemm_fp8.argtypes = [P, P, P, P, P, I32, I32, I32, I32, P, P, P]
    lib.pk_moe_router_topk.restype = ctypes.c_int
    lib.pk_moe_router_topk.argtypes = [P, I32, I32, I32, P, P, P]
    lib.pk_moe_combine.restype = ctypes.c_int
    lib.pk_moe_combine.argtypes = [P, P, P, I32, I32, I32, P, P, P]
    lib.pk_moe_route_kernel_launches.restype = ctypes.c_int
    lib.pk_moe_route_kernel_launches.argtypes = [I32, I32, I32]
    lib.pk_moe_set_gemm_kernel.restype = ctypes.c_int
    lib.pk_moe_set_gemm_kernel.argtypes = [ctypes.c_int]
    lib.pk_moe_set_wait_limit_ns.restype = None
    lib.pk_moe_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.pk_debug_bounded_wait.restype = ctypes.c_int
    lib.pk_debug_bounded_wait.argtypes = [P, ctypes.c_uint64, P]
    lib.pk_moe_quant_rows_mx.restype = ctypes.c_int
    lib.pk_moe_quant_rows_mx.argtypes = [P, I32, I32, P, P, P]
    lib.pk_moe_mx_weight_scale_bytes.restype = SZ
    lib.pk_moe_mx_weight_scale_bytes.argtypes = [I32, I32, I32]
    lib.pk_moe_quant_weights_mx.restype = ctypes.c_int
    lib.pk_moe_quant_weights_mx.argtypes = [P, I32, I32, I32, P, P, P]
    lib.pk_moe_dispatch_gemm_mxfp8.restype = ctypes.c_int
    lib.pk_moe_dispatch_gemm_mxfp8.argtypes = [P, P, P, P, P, P, I32, I32, I32, I32, I32, P, P, P]
    lib.pk_debug_stall_gemm.restype = None
    lib.pk_debug_stall_gemm.argtypes = [I32, ctypes.c_int64]
    return lib


lib = _load()


# ----------------------------------------------------------------- helpers
def _ptr(t: torch.Tensor | None, dtype, name: str, numel: int | None = None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: needs at least {numel} elements, has {t.numel()}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _check(rc: int, where: str):
    if rc != PK_OK:
        raise PkError(rc, where)


# ------------------------------------------------------- the C entry points
def pk_status_str(code: int) -> str:
    return lib.pk_status_str(int(code)).decode()


def pk_abi_version() -> int:
    return int(lib.pk_abi_version())


def pk_moe_workspace_bytes(T: int, k: int, E: int) -> int:
    return int(lib.pk_moe_workspace_bytes(T, k, E))


def pk_moe_route_counts(topk_idx: torch.Tensor, E: int, expert_offsets: torch.Tensor,
                        expert_counts: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None,
                        status_word: torch.Tensor | None = None, stream=None) -> None:
    T, k = topk_idx.shape
    ws_bytes = pk_moe_workspace_bytes(T, k, E)
    if workspace is None:
        raise ValueError("workspace: pass a uint8 CUDA tensor of pk_moe_workspace_bytes(T, k, E) bytes")
    rc = lib.pk_moe_route_counts(
        _ptr(topk_idx, torch.int32, "topk_idx"), T, k, E,
        _ptr(expert_counts, torch.int32, "expert_counts", E),
        _ptr(expert_offsets, torch.int32, "expert_offsets", E + 1),
        _ptr(workspace, torch.uint8, "workspace", ws_bytes), workspace.numel(),
        _ptr(status_word, torch.int32, "status_word", 1), _stream(stream))
    _check(rc, "pk_moe_route_counts")


def pk_moe_build_perm(topk_idx: torch.Tensor, E: int, expert_offsets: torch.Tensor,
                      perm: torch.Tensor, inv_perm: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None,
                      status_word: torch.Tensor | None = None, stream=None) -> None:
    T, k = topk_idx.shape
    if workspace is None:
        raise ValueError("workspace: pass the workspace filled by pk_moe_route_counts")
    rc = lib.pk_moe_build_perm(
        _ptr(topk_idx, torch.int32, "topk_idx"), T, k, E,
        _ptr(expert_offsets, torch.int32, "expert_offsets", E + 1),
        _ptr(perm, torch.int32, "perm", T * k),
        _ptr(inv_perm, torch.int32, "inv_perm", T * k),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _ptr(status_word, torch.int32, "status_word", 1), _stream(stream))
    _check(rc, "pk_moe_build_perm")


def pk_moe_dispatch_gemm(x: torch.Tensor, perm: torch.Tensor, expert_offsets: torch.Tensor,
                         W: torch.Tensor, k: int, out: torch.Tensor,
                         status_word: torch.Tensor | None = None, stream=None) -> None:
    T, D = x.shape
    E, D2, De = W.shape
    if D2 != D:
        raise ValueError(f"W is [E, {D2}, De] but x has D={D}")
    rc = lib.pk_moe_dispatch_gemm(
        _ptr(x, torch.bfloat16, "x"), _ptr(perm, torch.int32, "perm", T * k),
        _ptr(expert_offsets, torch.int32, "expert_offsets", E + 1),
        _ptr(W, torch.bfloat16, "W"), T, k, D, E, De,
        _ptr(out, torch.bfloat16, "out", T * k * De),
        _ptr(status_word, torch.int32, "status_word", 1), _stream(stream))
    _check(rc, "pk_moe_dispatch_gemm")


def pk_moe_grouped_gemm(A: torch.Tensor, expert_offsets: torch.Tensor, W: torch.Tensor,
                        out: torch.Tensor, status_word: torch.Tensor | None = None,
                        stream=None) -> None:
    R, K = A.shape
    E, K2, N = W.shape
    if K2 != K:
        raise ValueError(f"W is [E, {K2}, N] but A has K={K}")
    rc = lib.pk_moe_grouped_gemm(_ptr(A, torch.bfloat16, "A"),
                                 _ptr(expert_offsets, torch.int32, "expert_offsets", E + 1),
                                 _ptr(W, torch.bfloat16, "W"), R, K, N, E,
                                 _ptr(out, torch.bfloat16, "out", R * N),
                                 _ptr(status_word, torch.int32, "status_word", 1), _stream(stream))
    _check(rc, "pk_moe_grouped_gemm")


def pk_moe_dispatch_gemm_fp8(xq: torch.Tensor, sx: torch.Tensor, perm: torch.Tensor,
                             expert_offsets: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor,
                             k: int, out: torch.Tensor, status_word: torch.Tensor | None = None,
                             stream=None) -> None:
    """xq: uint8 E4M3 codes [T, D]; wq: the blocked codes pk_moe_quant_weights
    writes; sw: fp32 [E, D_expert] (gives E and D_expert)."""
    T, D = xq.shape
    E, De = sw.shape
    rc = lib.pk_moe_dispatch_gemm_fp8(
        _ptr(xq, torch.uint8, "xq"), _ptr(sx, torch.float32, "sx", T),
        _ptr(perm, torch.int32, "perm", T * k),
        _ptr(expert_offsets, torch.int32, "expert_offsets", E + 1),
        _ptr(wq, torch.uint8, "wq", pk_moe_fp8_weight_bytes(E, D, De)),
        _ptr(sw, torch.float32, "sw", E * De), T, k, D, E, De,
        _ptr(out, torch.bfloat16, "out", T * k * De),
        _ptr(status_word, torch.int32, "status_word", 1), _stream(stream))
    _check(rc, "pk_moe_dispatch_gemm_fp8")


def pk_moe_quant_rows(x: torch.Tensor, xq: torch.Tensor, sx: torch.Tensor, stream=None) -> None:
    T, D = x.shape
    rc = lib.pk_moe_quant_rows(_ptr(x, torch.bfloat16, "x"), T, D,
                               _ptr(xq, torch.uint8, "xq", T * D),
                               _ptr(sx, torch.float32, "sx", T), _stream(stream))
    _check(rc, "pk_moe_quant_rows")


def pk_moe_fp8_weight_bytes(E: int, D: int, N: int) -> int:
    return int(lib.pk_moe_fp8_weight_bytes(E, D, N))


def pk_moe_quant_weights(W: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor,
                         stream=None) -> None:
    """W: bf16 [E, D, N] -> wq uint8 blocked codes (pk_moe_fp8_weight_bytes
    bytes), sw fp32 [E, N]."""
    E, D, N = W.shape
    rc = lib.pk_moe_quant_weights(_ptr(W, torch.bfloat16, "W"), E, D, N,
                                  _ptr(wq, torch.uint8, "wq", pk_moe_fp8_weight_bytes(E, D, N)),
                                  _ptr(sw, torch.float32, "sw", E * N), _stream(stream))
    _check(rc, "pk_moe_quant_weights")


def pk_moe_quant_rows_mx(x: torch.Tensor, xq: torch.Tensor, sx: torch.Tensor,
                         stream=None) -> None:
    """x: bf16 [T, D] -> xq uint8 E4M3 codes [T, D], sx uint8 E8M0 scale bytes
    [T, D // 32]."""
    T, D = x.shape
    rc = lib.pk_moe_quant_rows_mx(_ptr(x, torch.bfloat16, "x"), T, D,
                                  _ptr(xq, torch.uint8, "xq", T * D),
                                  _ptr(sx, torch.uint8, "sx", T * (D // 32)), _stream(stream))
    _check(rc, "pk_moe_quant_rows_mx")


def pk_moe_mx_weight_scale_bytes(E: int, D: int, N: int) -> int:
    return int(lib.pk_moe_mx_weight_scale_bytes(E, D, N))


def pk_moe_quant_weights_mx(W: torch.Tensor, wq: torch.Tensor, swb: torch.Tensor,
                            stream=None) -> None:
    """W: bf16 [E, D, N] -> wq uint8 blocked codes (pk_moe_fp8_weight_bytes
    bytes), swb uint8 scale pieces (pk_moe_mx_weight_scale_bytes bytes)."""
    E, D, N = W.shape
    rc = lib.pk_moe_quant_weights_mx(
        _ptr(W, torch.bfloat16, "W"), E, D, N,
        _ptr(wq, torch.uint8, "wq", pk_moe_fp8_weight_bytes(E, D, N)),
        _ptr(swb, torch.uint8, "swb", pk_moe_mx_weight_scale_bytes(E, D, N)), _stream(stream))
    _check(rc, "pk_moe_quant_weights_mx")


def pk_moe_dispatch_gemm_mxfp8(xq: torch.Tensor, sx: torch.Tensor, perm: torch.Tensor,
                               expert_offsets: torch.Tensor, wq: torch.Tensor,
                               swb: torch.Tensor, E: int, D_expert: int, k: int,
                               out: torch.Tensor, status_word: torch.Tensor | None = None,
                               stream=None) -> None:
    """xq, sx from pk_moe_quant_rows_mx; wq, swb from pk_moe_quant_weights_mx."""
    T, D = xq.shape
    De = D_expert
    rc = lib.pk_moe_dispatch_gemm_mxfp8(
        _ptr(xq, torch.uint8, "xq"), _ptr(sx, torch.uint8, "sx", T * (D // 32)),
        _ptr(perm, torch.int32, "perm", T * k),
        _ptr(expert_offsets, torch.int32, "expert_offsets", E + 1),
        _ptr(wq, torch.uint8, "wq", pk_moe_fp8_weight_bytes(E, D, De)),
        _ptr(swb, torch.uint8, "swb", pk_moe_mx_weight_scale_bytes(E, D, De)), T, k, D, E, De,
        _ptr(out, torch.bfloat16, "out", T * k * De),
        _ptr(status_word, torch.int32, "status_word", 1), _stream(stream))
    _check(rc, "pk_moe_dispatch_gemm_mxfp8")


def pk_moe_grouped_gemm_fp8(Aq: torch.Tensor, sa: torch.Tensor, expert_offsets: torch.Tensor,
                            wq: torch.Tensor, sw: torch.Tensor, out: torch.Tensor,
                            status_word: torch.Tensor | None = None, stream=None) -> None:
    """Aq: uint8 codes [R, K]; wq: blocked codes of W2 [E, K, N]; sw: fp32 [E, N]."""
    R, K = Aq.shape
    E, N = sw.shape
    rc = lib.pk_moe_grouped_gemm_fp8(
        _ptr(Aq, torch.uint8, "Aq"), _ptr(sa, torch.float32, "sa", R),
        _ptr(expert_offsets, torch.int32, "expert_offsets", E + 1),
        _ptr(wq, torch.uint8, "wq", pk_moe_fp8_weight_bytes(E, K, N)),
        _ptr(sw, torch.float32, "sw", E * N), R, K, N, E,
        _ptr(out, torch.bfloat16, "out", R * N),
        _ptr(status_word, torch.int32, "status_word", 1), _stream(stream))
    _check(rc, "pk_moe_grouped_gemm_fp8")


def pk_moe_router_topk(logits: torch.Tensor, k: int, topk_idx: torch.Tensor,
                       gates: torch.Tensor | None = None, stream=None) -> None:
    T, E = logits.shape
    rc = lib.pk_moe_router_topk(_ptr(logits, torch.float32, "logits"), T, E, k,
                                _ptr(topk_idx, torch.int32, "topk_idx", T * k),
                                _ptr(gates, torch.float32, "gates", T * k), _stream(stream))
    _check(rc, "pk_moe_router_topk")


def pk_moe_combine(src: torch.Tensor, inv_perm: torch.Tensor, gates: torch.Tensor | None,
                   T: int, k: int, y: torch.Tensor, status_word: torch.Tensor | None = None,
                   stream=None) -> None:
    R, C = src.shape
    if R < T * k:
        raise ValueError(f"src has {R} rows, needs T*k = {T * k}")
    rc = lib.pk_moe_combine(_ptr(src, torch.bfloat16, "src"),
                            _ptr(inv_perm, torch.int32, "inv_perm", T * k),
                            _ptr(gates, torch.float32, "gates", T * k), T, k, C,
                            _ptr(y, torch.bfloat16, "y", T * C),
                            _ptr(status_word, torch.int32, "status_word", 1), _stream(stream))
    _check(rc, "pk_moe_combine")


def pk_moe_route_noalloc(topk_idx: torch.Tensor, E: int, expert_offsets: torch.Tensor,
                         perm: torch.Tensor, expert_counts: torch.Tensor | None = None,
                         inv_perm: torch.Tensor | None = None,
                         status_word: torch.Tensor | None = None, stream=None) -> None:
    """Counts, offsets, perm and inv_perm without a caller workspace: for
    callers that cannot allocate device memory (the C call allocates none;
    its counters live in a fixed 1 MiB array inside the library). The first
    call in a CUDA context must come before any stream capture (made during
    capture it raises PkError with PK_ERR_CAPTURE); calls that overlap on the
    GPU share that array and race."""
    T, k = topk_idx.shape
    rc = lib.pk_moe_route_noalloc(
        _ptr(topk_idx, torch.int32, "topk_idx"), T, k, E,
        _ptr(expert_counts, torch.int32, "expert_counts", E),
        _ptr(expert_offsets, torch.int32, "expert_offsets", E + 1),
        _ptr(perm, torch.int32, "perm", T * k),
        _ptr(inv_perm, torch.int32, "inv_perm", T * k),
        _ptr(status_word, torch.int32, "status_word", 1), _stream(stream))
    _check(rc, "pk_moe_route_noalloc")


def pk_moe_route_kernel_launches(T: int, k: int, E: int) -> int:
    return int(lib.pk_moe_route_kernel_launches(T, k, E))


def pk_moe_set_gemm_kernel(kernel: int) -> None:
    _check(lib.pk_moe_set_gemm_kernel(int(kernel)), "pk_moe_set_gemm_kernel")


def pk_moe_set_wait_limit_ns(limit_ns: int) -> None:
    lib.pk_moe_set_wait_limit_ns(int(limit_ns))


def pk_debug_bounded_wait(status_word: torch.Tensor, limit_ns: int, stream=None) -> None:
    rc = lib.pk_debug_bounded_wait(_ptr(status_word, torch.int32, "status_word", 1), int(limit_ns),
                                   _stream(stream))
    _check(rc, "pk_debug_bounded_wait")


def pk_debug_stall_gemm(cta: int, kstep: int) -> None:
    """Test hook: CTA `cta` of each one-CTA GEMM launch skips the copies of its
    K-step `kstep`; a negative value turns it off."""
    lib.pk_debug_stall_gemm(int(cta), int(kstep))
