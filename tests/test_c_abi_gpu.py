"""The C ABI from a plain C program (tests/c_abi/abi_demo.c): no Python, no
torch on the calling side; gcc links it against libpkmoe.so, the CUDA
runtime and, for checking only, the oracle and input-generator libraries."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_runs_the_path(gpu_lib, tmp_path):
    import inputgen
    import oracle
    inputgen.build()
    oracle.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdirs = [os.path.join(ROOT, "moe_token_dispatch_gb300"), os.path.join(ROOT, "oracle"),
               os.path.join(ROOT, "inputgen"), os.path.join(cuda, "lib64")]
    exe = str(tmp_path / "abi_demo")
    cmd = ["gcc", "-O2", "-std=c11", os.path.join(ROOT, "tests", "c_abi", "abi_demo.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"), "-o", exe]
    for d in libdirs:
        cmd += ["-L", d, "-Wl,-rpath," + d]
    cmd += ["-lpkmoe", "-loracle", "-linputgen", "-lcudart", "-lm"]
    subprocess.check_call(cmd)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi demo ok" in r.stdout
