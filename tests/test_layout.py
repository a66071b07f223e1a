"""Shared-memory layouts of the forward and backward kernels (tests/layout_check.cu),
compiled with nvcc for the host and run on the CPU: every region lies inside
the launch's shared memory with the alignment its users need and overlaps no
other.  Two planted mistakes in a copy of the forward header (the split ring's
V barriers laid over the misc words; the K/V ring moved off its 1024-byte
swizzle alignment) must each be caught."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_10_gb300", "csrc")
NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"

pytestmark = pytest.mark.skipif(not os.path.exists(NVCC), reason="nvcc not available")


def _build_and_run(tmp, csrc):
    exe = os.path.join(tmp, "layout_check")
    subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1",
                    "-I", os.path.join(ROOT, "include"), "-I", csrc,
                    os.path.join(ROOT, "tests", "layout_check.cu"), "-o", exe],
                   check=True, capture_output=True)
    return subprocess.run([exe], capture_output=True, text=True)


def test_layouts_fit_and_do_not_overlap(tmp_path):
    r = _build_and_run(str(tmp_path), CSRC)
    print(r.stdout)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout


@pytest.mark.parametrize("old,new,expect", [
    ("split ? ((kJobOff + kJobSlots * (int)sizeof(MergeJob) + 7) & ~7) : kMiscOff + 16;",
     "split ? ((kJobOff + kJobSlots * (int)sizeof(MergeJob) + 7) & ~7) : kMiscOff + 8;",
     "FAIL forward D=128 whole: V barriers"),
    ("static constexpr int kStageOff = kQBufs * kQBufBytes;",
     "static constexpr int kStageOff = kQBufs * kQBufBytes + 512;",
     "K/V ring at"),
])
def test_planted_layout_mistakes_are_caught(tmp_path, old, new, expect):
    csrc = os.path.join(str(tmp_path), "csrc")
    shutil.copytree(CSRC, csrc)
    path = os.path.join(csrc, "fa_fwd_kernel.cuh")
    with open(path) as f:
        src = f.read()
    assert src.count(old) == 1, old
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    try:
        r = _build_and_run(str(tmp_path), csrc)
    except subprocess.CalledProcessError as e:   # a static_assert in the header may stop it first
        assert b"shared memory" in e.stderr or b"static assertion" in e.stderr, e.stderr[-400:]
        return
    assert r.returncode != 0 and expect in r.stdout, r.stdout
