"""Compile the fp64 oracle (attn_ref.c) into oracle/_attn_ref.so with gcc.

Test infrastructure: the library build in ``__graft_entry__.build()`` also runs
this, so the checker exists on every machine the tests run on.  Plain C99 with
OpenMP, no intrinsics and no -march flags, so the same source builds on x86_64
and aarch64.  FMA contraction is off so both machines round the same way.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_ref.c")
LIB_PATH = os.path.join(HERE, "_attn_ref.so")

CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math"]


def build(src: str = SRC, out: str = LIB_PATH, extra_flags=None) -> str:
    """Compile ``src`` into the shared library ``out``; returns ``out``."""
    cmd = ["gcc", *CFLAGS, *(extra_flags or []), src, "-o", out, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"oracle build failed ({' '.join(cmd)}):\n{res.stderr}")
    return out


if __name__ == "__main__":
    print(build(*sys.argv[1:2]))
