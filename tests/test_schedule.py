"""The CTA work decomposition (exact_attention_10_gb300/csrc/fa_schedule.h),
compiled with g++ and checked exhaustively on the CPU: every unit of work is
assigned exactly once, partial-result slots are distinct, the merge of split
tiles expects exactly the parts that hold work, and the planner never cuts a
tile into more parts than the merge handles."""
from __future__ import annotations

import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = []
for N in (1, 2, 127, 128, 129, 255, 256, 257, 383, 513, 1024, 3000, 4096, 16384, 32768):
    for BH in (1, 3, 16, 32, 64):
        for causal in (0, 1):
            for G in (1, 7, 152):
                for split in (0, 1):
                    if N * BH > 64 * 4096 and G != 152:
                        continue
                    CASES.append((N, N, BH, causal, G, split, -1, 0))
# queries against a different number of keys: decode, cross attention, and
# Nq > Nkv (causal rows that see no key)
for N, Nkv in ((1, 4096), (16, 8192), (64, 3000), (127, 1000), (200, 70), (513, 200), (300, 1), (1000, 129)):
    for BH in (1, 5, 32):
        for causal in (0, 1):
            for G in (1, 7, 152):
                for split in (0, 1):
                    CASES.append((N, Nkv, BH, causal, G, split, -1, 0))
# band (sliding-window) masks: windows narrower and wider than a step, two-sided
for N, Nkv in ((1000, 1000), (4096, 4096), (300, 2000), (2000, 300), (1, 4096), (129, 129), (257, 5000)):
    for wl, wr in ((0, 0), (127, 0), (128, 0), (1000, 0), (64, 64), (300, -1), (5, 700), (0, 5), (4095, 0),
                   (-1, 128), (1 << 29, 3)):
        for BH in (1, 7):
            for G in (7, 152):
                for split in (0, 1):
                    CASES.append((N, Nkv, BH, 1, G, split, wl, wr))


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("sched") / "schedule_check")
    cmd = ["g++", "-O2", "-std=c++17", "-I", os.path.join(ROOT, "exact_attention_10_gb300", "csrc"),
           os.path.join(ROOT, "tests", "schedule_check.cpp"), "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True)
    return exe


PLAN_CASES = []
for N in (1, 2, 100, 256, 257, 513, 1000, 1024, 2048, 3000, 4096, 8192, 16384, 32768, 65536):
    for BH in (1, 2, 3, 8, 16, 32, 64, 128):
        for causal in (0, 1):
            for sms in (148, 152):
                if N * BH > 64 * 16384:
                    continue
                PLAN_CASES.append((N, N, BH, causal, sms, -1, 0))
for N, Nkv in ((1, 32768), (4, 131072), (64, 16384), (128, 4096), (513, 200), (4096, 64)):
    for BH in (1, 8, 32, 128):
        for causal in (0, 1):
            PLAN_CASES.append((N, Nkv, BH, causal, 152, -1, 0))
for N, Nkv, wl, wr in ((32768, 32768, 4096, 0), (8192, 8192, 255, 0), (1, 131072, 8192, 0), (4096, 4096, 512, 512),
                       (1500, 1500, 300, -1), (8192, 8192, 1000, -1), (3000, 3000, -1, 200), (4, 65536, 8191, 0),
                       (300, 2000, 511, 0), (513, 200, 50, 10)):
    for BH in (1, 3, 32):
        PLAN_CASES.append((N, Nkv, BH, 1, 152, wl, wr))

# the decode shapes bench.py times beside the headline, and the one-tile heads
# the GPU parity tests spread over more CTA tiles than SMs
for N, Nkv, BH in ((4, 32768, 32), (1, 8192, 256), (1, 32768, 32), (4, 131072, 8), (128, 32768, 32), (16, 2000, 160),
                   (77, 1500, 160), (1, 700, 160), (128, 900, 160)):
    for causal in (0, 1):
        PLAN_CASES.append((N, Nkv, BH, causal, 152, -1, 0))
for N, Nkv, BH, wl, wr in ((16, 2000, 160, 500, 0), (77, 1500, 160, 300, 40), (4, 131072, 8, 8191, 0)):
    PLAN_CASES.append((N, Nkv, BH, 1, 152, wl, wr))


def test_schedule_planner(checker):
    """Every schedule the planner picks covers all work once, and a balanced
    one cuts no tile into more parts than the merge handles."""
    args = ["plan"] + [str(x) for case in PLAN_CASES for x in case]
    res = subprocess.run([checker, *args], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:]
    assert f"{len(PLAN_CASES)} cases, 0 failures" in res.stdout


def test_schedule_exhaustive(checker):
    args = [str(x) for case in CASES for x in case]
    res = subprocess.run([checker, *args], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:]
    assert f"{len(CASES)} cases, 0 failures" in res.stdout


def test_no_alloc_planner_falls_back_to_whole_tiles(checker):
    """fa_fwd_noalloc's planner (sched_plan_limited): where the automatic
    plan would split tiles into more partial results than the static
    workspace holds, it runs whole tiles, which need none; otherwise, and for
    explicit requests, it plans exactly as fa_fwd_ex does.  The automatic
    plan never needs more than the real 48 MiB limit on these shapes, so the
    fallback is exercised with small limits as well."""
    cases = [(4096, 4096, 32, 0, 152, -1, 0, 64), (4096, 4096, 32, 1, 152, -1, 0, 64),
             (4, 32768, 32, 0, 152, -1, 0, 128), (1, 8192, 256, 0, 152, -1, 0, 128),
             (4, 131072, 8, 1, 152, -1, 0, 128), (3000, 3000, 16, 0, 152, -1, 0, 128),
             (16384, 16384, 32, 0, 152, -1, 0, 128), (8192, 8192, 3, 1, 152, 1000, -1, 64),
             (1024, 1024, 64, 0, 152, -1, 0, 64)]
    for limit, expect_fallbacks in ((48 << 20, False), (1 << 20, True), (0, True)):
        args = ["limit", str(limit)] + [str(x) for case in cases for x in case]
        res = subprocess.run([checker, *args], capture_output=True, text=True, timeout=600)
        assert res.returncode == 0, res.stdout[-2000:]
        assert f"{len(cases)} cases, 0 failures" in res.stdout, res.stdout
        fallbacks = int(res.stdout.split(",")[-1].split()[0])
        assert (fallbacks > 0) == expect_fallbacks, (limit, res.stdout)


TAIL_CASES = []
for N, Nkv in ((3000, 3000), (1024, 1024), (4096, 4096), (257, 257), (1, 4096), (300, 2000), (513, 129)):
    for BH in (3, 16, 32, 64, 160):
        for G in (7, 100, 152):
            for gt in (0, 3, 50):
                TAIL_CASES.append((N, Nkv, BH, G, gt))


def test_tail_split_schedules(checker):
    """The tail split (non-causal): every CTA takes its floor(T / G) whole
    tiles, and the tiles of the last partial wave are spread as units over
    the first gt CTAs; every unit is covered once, a CTA's partial parts come
    before its whole tiles, and each split tile's merge expects exactly the
    parts that hold work."""
    args = ["tail"] + [str(x) for case in TAIL_CASES for x in case]
    res = subprocess.run([checker, *args], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:]
    assert f"{len(TAIL_CASES)} cases, 0 failures" in res.stdout, res.stdout[-500:]
