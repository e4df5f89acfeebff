import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (seconds to minutes)")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library, built in-tree if missing; fails loudly without a GPU."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    import __graft_entry__
    __graft_entry__._build_module().build()
    import moe_token_dispatch_gb300 as pk
    return pk


@pytest.fixture(params=["pair", "single"])
def gemm_kernel(request, gpu_lib):
    """Runs a GEMM test once with the CTA-pair kernel and once with the
    one-CTA kernel (both behind the same C entry points)."""
    pk = gpu_lib
    pk.pk_moe_set_gemm_kernel(pk.PK_GEMM_KERNEL_PAIR if request.param == "pair"
                              else pk.PK_GEMM_KERNEL_SINGLE)
    yield request.param
    pk.pk_moe_set_gemm_kernel(pk.PK_GEMM_KERNEL_AUTO)
