"""Build the CUDA library (libfa_gb300.so) in-tree with nvcc for sm_103a.

Four translation units, compiled in parallel and linked into one shared
library: csrc/fa_api.cu (the C ABI and the whole-tile kernel variants without
a mask or with the causal one), csrc/fa_split.cu (the same for the balanced
schedule), csrc/fa_band.cu (left-bounded band masks, both schedules) and
csrc/fa_bwd.cu (the backward), so the build stays quick on both the x86_64
build machine and the aarch64 GPU host.
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
SRCS = [os.path.join(PKG, "csrc", f) for f in ("fa_api.cu", "fa_split.cu", "fa_band.cu", "fa_bwd.cu")]
LIB_PATH = os.path.join(PKG, "libfa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(out: str = LIB_PATH, verbose: bool = False, extra=None) -> str:
    common = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", os.path.join(ROOT, "include"), "-I", os.path.join(PKG, "csrc"),
              *(["-Xptxas", "-v"] if verbose else []), *(extra or [])]
    objs = [out + "." + os.path.splitext(os.path.basename(src))[0] + ".o" for src in SRCS]
    procs = [(src, subprocess.Popen([nvcc(), *common, "-c", src, "-o", obj], stdout=subprocess.PIPE,
                                    stderr=subprocess.PIPE, text=True))
             for src, obj in zip(SRCS, objs)]
    errors = []
    for src, proc in procs:
        _, err = proc.communicate()
        if proc.returncode != 0:
            errors.append(f"{src}:\n{err}")
        elif verbose:
            sys.stderr.write(err)
    if errors:
        raise RuntimeError("CUDA library build failed:\n" + "\n".join(errors))
    cmd = [nvcc(), *ARCH, "-shared", *objs, "-o", out]
    res = subprocess.run(cmd, capture_output=True, text=True)
    for obj in objs:
        try:
            os.remove(obj)
        except OSError:
            pass
    if res.returncode != 0:
        raise RuntimeError(f"CUDA library link failed:\n{' '.join(cmd)}\n{res.stderr}")
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
