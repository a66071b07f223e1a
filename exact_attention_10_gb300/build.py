"""Build the CUDA library (libfa_gb300.so) in-tree with nvcc for sm_103a.

One translation unit (csrc/fa_api.cu, which includes the kernel header) so the
build stays quick on both the x86_64 build machine and the aarch64 GPU host.
The runtime is linked statically and the driver's tensor-map encoder is
resolved at run time, so the library loads on a machine without a GPU driver
(its compute calls then return FA_ERR_UNSUPPORTED_DEVICE).
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "fa_api.cu")
LIB_PATH = os.path.join(PKG, "libfa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(out: str = LIB_PATH, verbose: bool = False, extra=None) -> str:
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(PKG, "csrc"),
           *(["-Xptxas", "-v"] if verbose else []), *(extra or []), SRC, "-o", out]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"CUDA library build failed:\n{' '.join(cmd)}\n{res.stderr}")
    if verbose:
        sys.stderr.write(res.stderr)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
