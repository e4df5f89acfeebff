"""The C ABI library loads, exports every declared entry point, and rejects
bad arguments on the host (CPU only: no call here reaches the device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pk_moe.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import moe_token_dispatch_gb300 as pk
    return pk


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(pk_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("pk_moe_route_counts", "pk_moe_build_perm", "pk_moe_dispatch_gemm",
              "pk_moe_workspace_bytes", "pk_status_str"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(so, name), name


def test_status_strings(lib):
    assert lib.pk_status_str(0) == "PK_OK"
    assert lib.pk_status_str(lib.PK_ERR_TIMEOUT) == "PK_ERR_TIMEOUT"
    assert lib.pk_status_str(99) == "PK_ERR_UNKNOWN"
    assert lib.pk_abi_version() >= 10000
    import re
    m = re.search(r"#define PK_ABI_VERSION (\d+)", open(HEADER).read())
    assert m and lib.pk_abi_version() == int(m.group(1))


def test_workspace_bytes(lib):
    assert lib.pk_moe_workspace_bytes(0, 8, 256) == 0
    # 2048 routed entries per block, E int32 counters per block, 256-byte rounding
    assert lib.pk_moe_workspace_bytes(8192, 8, 256) == 32 * 256 * 4
    assert lib.pk_moe_workspace_bytes(1, 1, 3) == 256
    assert lib.pk_moe_workspace_bytes(2049, 1, 64) == 2 * 64 * 4
    assert lib.pk_moe_workspace_bytes(2049, 1, 5) == 256


def _raw(lib):
    return lib.lib


FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: every call below fails its checks
FAKE_ODD = ctypes.c_void_p(0x10008)   # not 16-byte aligned


@pytest.mark.parametrize("args,code", [
    ((FAKE, -1, 2, 8, None, FAKE, FAKE, 4096, None, None), 1),   # T < 0
    ((FAKE, 4, 0, 8, None, FAKE, FAKE, 4096, None, None), 1),    # k < 1
    ((FAKE, 4, 9, 8, None, FAKE, FAKE, 4096, None, None), 1),    # k > E
    ((FAKE, 4, 2, 8, None, None, FAKE, 4096, None, None), 1),    # no offsets
    ((FAKE, 4, 2, 5000, None, FAKE, FAKE, 1 << 20, None, None), 2),  # E too large
    ((FAKE, 4, 2, 8, None, FAKE, FAKE, 16, None, None), 1),      # workspace too small
    ((FAKE, 4, 2, 8, None, FAKE, FAKE_ODD, 4096, None, None), 1),  # workspace misaligned
    ((FAKE, 1 << 29, 8, 8, None, FAKE, FAKE, 1 << 40, None, None), 2),  # T*k >= 2^31
])
def test_route_counts_rejects(lib, args, code):
    assert _raw(lib).pk_moe_route_counts(*args) == code


@pytest.mark.parametrize("args,code", [
    ((FAKE, FAKE, FAKE, FAKE, 4, 2, 7, 8, 64, FAKE, None, None), 1),     # D % 8
    ((FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 8, 12, FAKE, None, None), 1),    # De % 8
    ((FAKE_ODD, FAKE, FAKE, FAKE, 4, 2, 64, 8, 64, FAKE, None, None), 1),  # x misaligned
    ((FAKE, FAKE, FAKE, FAKE_ODD, 4, 2, 64, 8, 64, FAKE, None, None), 1),  # W misaligned
    ((FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 8, 64, FAKE_ODD, None, None), 1),  # out misaligned
    ((FAKE, None, FAKE, FAKE, 4, 2, 64, 8, 64, FAKE, None, None), 1),    # no perm
    ((FAKE, FAKE, FAKE, FAKE, 4, 0, 64, 8, 64, FAKE, None, None), 1),    # k < 1
    ((FAKE, FAKE, FAKE, FAKE, 1 << 29, 8, 64, 8, 64, FAKE, None, None), 2),  # T*k >= 2^31
])
def test_dispatch_gemm_rejects(lib, args, code):
    assert _raw(lib).pk_moe_dispatch_gemm(*args) == code


def test_zero_rows_are_a_no_op(lib):
    # T == 0: nothing to launch for build_perm and dispatch_gemm
    assert _raw(lib).pk_moe_build_perm(None, 0, 2, 8, None, None, None, None, 0, None, None) == 0
    assert _raw(lib).pk_moe_dispatch_gemm(None, None, None, None, 0, 2, 64, 8, 64, None, None,
                                          None) == 0


def test_build_perm_rejects(lib):
    assert _raw(lib).pk_moe_build_perm(FAKE, 4, 2, 8, FAKE, None, None, FAKE, 4096, None,
                                       None) == 1
    assert _raw(lib).pk_moe_build_perm(FAKE, 4, 2, 8, FAKE, FAKE, None, FAKE, 8, None,
                                       None) == 1
    assert _raw(lib).pk_debug_bounded_wait(None, 10, None) == 1


@pytest.mark.parametrize("args,code", [
    # xq, sx, perm, offsets, wq, sw, T, k, D, E, De, out, status, stream
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 56, 8, 64, FAKE, None, None), 1),   # D % 16
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 8, 12, FAKE, None, None), 1),   # De % 8
    ((FAKE_ODD, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 8, 64, FAKE, None, None), 1),  # xq
    ((FAKE, FAKE, FAKE, FAKE, FAKE_ODD, FAKE, 4, 2, 64, 8, 64, FAKE, None, None), 1),  # wq
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE_ODD, 4, 2, 64, 8, 64, FAKE, None, None), 1),  # sw
    ((FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 8, 64, FAKE, None, None), 1),   # no sx
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 29, 8, 64, 8, 64, FAKE, None, None), 2),
])
def test_dispatch_gemm_fp8_rejects(lib, args, code):
    assert _raw(lib).pk_moe_dispatch_gemm_fp8(*args) == code


def test_quant_entry_points_reject(lib):
    L = _raw(lib)
    assert L.pk_moe_quant_rows(FAKE, 4, 12, FAKE, FAKE, None) == 1        # D % 8
    assert L.pk_moe_quant_rows(FAKE_ODD, 4, 16, FAKE, FAKE, None) == 1    # x misaligned
    assert L.pk_moe_quant_rows(None, 0, 16, None, None, None) == 0        # T == 0: no-op
    assert L.pk_moe_quant_weights(FAKE, 0, 16, 16, FAKE, FAKE, None) == 1
    assert L.pk_moe_quant_weights(FAKE, 70000, 16, 16, FAKE, FAKE, None) == 2
    # W and wq 16-byte aligned, sw 4-byte aligned, checked before any CUDA call
    assert L.pk_moe_quant_weights(FAKE_ODD, 2, 16, 16, FAKE, FAKE, None) == 1
    assert L.pk_moe_quant_weights(FAKE, 2, 16, 16, FAKE_ODD, FAKE, None) == 1
    assert L.pk_moe_quant_weights(FAKE, 2, 16, 16, FAKE, ctypes.c_void_p(0x10002), None) == 1
    assert L.pk_moe_dispatch_gemm_fp8(None, None, None, None, None, None, 0, 2, 64, 8, 64,
                                      None, None, None) == 0


def test_fp8_weight_bytes(lib):
    L = _raw(lib)
    # 64-column x 128-code blocks of 8 KiB, padded in both directions
    assert L.pk_moe_fp8_weight_bytes(256, 7168, 2048) == 256 * 32 * 56 * 8192
    assert L.pk_moe_fp8_weight_bytes(3, 200, 136) == 3 * 3 * 2 * 8192
    assert L.pk_moe_fp8_weight_bytes(0, 16, 8) == 0


def test_set_gemm_kernel(lib):
    L = _raw(lib)
    assert L.pk_moe_set_gemm_kernel(7) == 1
    assert L.pk_moe_set_gemm_kernel(-1) == 1
    for v in (1, 2, 0):
        assert L.pk_moe_set_gemm_kernel(v) == 0


def test_route_kernel_launches(lib):
    L = _raw(lib)
    assert L.pk_moe_route_kernel_launches(128, 8, 256) == 2      # one chunk
    assert L.pk_moe_route_kernel_launches(512, 8, 4096) == 2     # two chunks x 4096 experts
    assert L.pk_moe_route_kernel_launches(513, 8, 256) == 3      # three chunks
    assert L.pk_moe_route_kernel_launches(8192, 8, 256) == 3
    assert L.pk_moe_route_kernel_launches(0, 8, 256) == 1
    assert L.pk_moe_route_kernel_launches(-1, 8, 256) == -1


def test_grouped_gemm_fp8_rejects(lib):
    L = _raw(lib)
    # Aq, sa, offsets, wq, sw, R, K, N, E, out, status, stream
    assert L.pk_moe_grouped_gemm_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 56, 64, 2, FAKE, None, None) == 1
    assert L.pk_moe_grouped_gemm_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 64, 12, 2, FAKE, None, None) == 1
    assert L.pk_moe_grouped_gemm_fp8(FAKE, None, FAKE, FAKE, FAKE, 8, 64, 64, 2, FAKE, None, None) == 1
    assert L.pk_moe_grouped_gemm_fp8(None, None, None, None, None, 0, 64, 64, 2, None, None, None) == 0


def _code_only(path):
    """C/C++ source without comments or string literals."""
    import re
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r'"(?:\\.|[^"\\])*"', '""', text)


def test_noalloc_path_names_no_allocation_call():
    """The allocation-free routing entry point and the routing launch helpers
    it calls contain no device or host allocation call (comments aside)."""
    import re
    csrc = os.path.join(ROOT, "moe_token_dispatch_gb300", "csrc")
    pat = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cuMemAlloc\w*|cuMemFree\w*|cuMemCreate|"
                     r"cudaHostAlloc|cudaMallocHost|malloc|calloc|realloc|new)\s*[\(\[]")
    for name in ("route_noalloc.cu", "route.cu"):
        hits = pat.findall(_code_only(os.path.join(csrc, name)))
        assert not hits, (name, hits)
