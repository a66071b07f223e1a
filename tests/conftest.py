import json
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle._load()


@pytest.fixture(scope="session")
def kernel_constants(tmp_path_factory):
    """The kernels' pipeline constants (tests/kernel_constants.cu, compiled with
    nvcc for the host), which the CPU models of their protocols must match."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("kernel_constants") / "kernel_constants")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "exact_attention_10_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "kernel_constants.cu"), "-o", exe], check=True, capture_output=True)
    return json.loads(subprocess.run([exe], check=True, capture_output=True, text=True).stdout)
