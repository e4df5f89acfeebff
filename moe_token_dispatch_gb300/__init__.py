"""GB300 (sm_103a) MoE token dispatch + expert GEMM.

The hot path -- routing histogram and scan, stable (expert, token, slot)
permutation, and the per-expert GEMM fed by a row gather -- runs in the CUDA
kernels of ``libpkmoe.so`` behind the C ABI in ``include/pk_moe.h``. This
package is its ctypes binding (same function names) plus ``MoeDispatch``, a
holder of the device buffers one step needs. PyTorch provides device memory
and streams only.
"""
from ._binding import (  # noqa: F401
    LIB_PATH,
    PK_ERR_BAD_INDEX,
    PK_ERR_CAPTURE,
    PK_ERR_CUDA,
    PK_ERR_INVALID_ARG,
    PK_ERR_TIMEOUT,
    PK_ERR_UNSUPPORTED,
    PK_GEMM_KERNEL_AUTO,
    PK_GEMM_KERNEL_PAIR,
    PK_GEMM_KERNEL_SINGLE,
    PK_MAX_EXPERTS,
    PK_NOALLOC_SCRATCH_BYTES,
    PK_OK,
    PK_ROUTER_MAX_EXPERTS,
    PkError,
    lib,
    pk_abi_version,
    pk_debug_bounded_wait,
    pk_debug_stall_gemm,
    pk_moe_dispatch_gemm_mxfp8,
    pk_moe_mx_weight_scale_bytes,
    pk_moe_quant_rows_mx,
    pk_moe_quant_weights_mx,
    pk_moe_build_perm,
    pk_moe_combine,
    pk_moe_dispatch_gemm,
    pk_moe_dispatch_gemm_fp8,
    pk_moe_fp8_weight_bytes,
    pk_moe_grouped_gemm,
    pk_moe_grouped_gemm_fp8,
    pk_moe_quant_rows,
    pk_moe_quant_weights,
    pk_moe_route_counts,
    pk_moe_route_kernel_launches,
    pk_moe_route_noalloc,
    pk_moe_router_topk,
    pk_moe_set_gemm_kernel,
    pk_moe_set_wait_limit_ns,
    pk_moe_workspace_bytes,
    pk_status_str,
)
from .dispatch import MoeDispatch  # noqa: F401
