"""GPU parity: the CUDA path against the fp64 oracle, through the C ABI.

Tolerances (max over every compared element), as the task states them:
  bf16: max|O - O_ref| <= 1e-2;  fp16: max|O - O_ref| <= 2e-3;  |LSE - LSE_ref| <= 1e-3.
O_ref is the unrounded fp64 oracle output, so the kernel's own output
rounding counts against the tolerance.

Workloads: the five named in exact_attention_10_gb300.inputs, compared in full
where the oracle finishes in seconds; at the long-context sizes, in the same
launch configuration bench.py times, three heads in full and 512 rows of
every other head (rows 0, 1, tile edges, N-1 and random rows).  Edge cases: N around tile edges,
one key, several heads, both dtypes and head sizes, large logits.  The
balanced schedule (tiles split into parts and merged) is forced on the full
workloads and every edge case, where its small sizes cut tiles into up to
seven parts.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_10_gb300 import fa
from exact_attention_10_gb300.inputs import WORKLOADS, make_custom, make_qkv

pytestmark = pytest.mark.gpu

TOL_O = {"bf16": 1e-2, "fp16": 2e-3}
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load()


def _run(q, k, v, causal, scale, schedule="auto"):
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale, schedule=schedule)
    rc = fa.sync_status(torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0, fa.status_string(rc)
    return o.cpu(), lse.cpu()


def _report(o, lse, o_ref, lse_ref):
    od = o.double().numpy().reshape(o_ref.shape)
    ld = lse.double().numpy().reshape(lse_ref.shape)
    err = np.abs(od - o_ref)
    lerr = np.abs(ld - lse_ref)
    return float(err.max()), float(err.mean()), float(lerr.max()), err


def _check_full(q, k, v, causal, scale, dtype, label="", schedule="auto"):
    o, lse = _run(q, k, v, causal, scale, schedule)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all(), label
    o_ref, lse_ref = oracle.forward(q, k, v, causal, scale)
    emax, emean, lmax, err = _report(o, lse, o_ref, lse_ref)
    where = np.unravel_index(int(err.argmax()), err.shape)
    print(f"{label} causal={int(causal)} {schedule}: max|dO|={emax:.3e} mean|dO|={emean:.3e} max|dLSE|={lmax:.3e} "
          f"worst at {tuple(int(i) for i in where)} (|O_ref|={abs(o_ref[where]):.3f})")
    assert emax <= TOL_O[dtype], (label, emax)
    assert lmax <= TOL_LSE, (label, lmax)
    return emax, emean, lmax


@pytest.mark.parametrize("schedule", ["auto", "balanced"])
@pytest.mark.parametrize("name", ["tiny_n256", "b4h16_n1024", "ragged_n3000_d128_fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_workload_full(name, causal, schedule):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w, seed=0)
    _check_full(q, k, v, causal, w.scale, w.dtype, name, schedule)


@pytest.mark.parametrize("seed", [1, 2])
@pytest.mark.parametrize("name", ["tiny_n256", "b4h16_n1024"])
def test_workload_extra_seeds(name, seed):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w, seed=seed)
    for causal in (False, True):
        _check_full(q, k, v, causal, w.scale, w.dtype, f"{name}/seed{seed}")


@pytest.mark.parametrize("schedule", ["auto", "whole_tiles", "balanced"])
@pytest.mark.parametrize("causal", [False, True])
def test_n4096_full_and_error_magnitude(causal, schedule):
    """The pages' N = 4096 comparison scale, compared in full.  Non-causal, the
    mean |O - O_f64| should sit near the 4.52e-5 the pages measured for a
    kernel that sums l from fp32 P and rounds P to bf16 ("How to profile and
    optimise kernels", the P cast section), and cannot beat the 2.9e-5 floor of
    bf16 output rounding."""
    w = WORKLOADS["b2h16_n4096"]
    q, k, v = make_qkv(w, seed=0)
    _, emean, _ = _check_full(q, k, v, causal, w.scale, w.dtype, w.name, schedule)
    if not causal:
        assert 2.8e-5 <= emean <= 6.0e-5, emean


def _sample_rows(BH, N, per_head, seed, full_heads=()):
    """Rows to compare: every row of the heads in ``full_heads``; in every
    other head, rows 0, 1, the 128-row tile edges around 128 and 256, N/2,
    N-2, N-1 and random distinct rows, ``per_head`` in all."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 255, 256, N // 2, N - 2, N - 1]
    bh_idx, row_idx = [], []
    for h in range(BH):
        if h in full_heads:
            rows = range(N)
        else:
            rows = set(r for r in fixed if 0 <= r < N)
            rest = np.setdiff1d(np.arange(N), np.fromiter(rows, dtype=np.int64))
            rows.update(int(r) for r in rng.choice(rest, per_head - len(rows), replace=False))
            rows = sorted(rows)
        for r in rows:
            bh_idx.append(h)
            row_idx.append(r)
    return np.array(bh_idx), np.array(row_idx)


LONG_FULL_HEADS = (0, 15, 31)


@pytest.mark.parametrize("name", ["long_n32768_d128", "long_n16384_d128"])
def test_long_context_sampled_rows(name):
    """The long-context workload in the launch configuration bench.py times:
    heads 0, 15 and 31 compared against the oracle in full, and 512 rows of
    every other head (rows 0, 1, 127, 128, N-1 among them).  Each row of the
    oracle is computed on its own, so a sampled row is checked exactly as in
    a full comparison."""
    w = WORKLOADS[name]
    q, k, v = make_qkv(w, seed=0)
    causal = w.masks[0]
    o, lse = _run(q, k, v, causal, w.scale)
    assert torch.isfinite(lse).all()
    BH = w.B * w.H
    bh_idx, row_idx = _sample_rows(BH, w.N, 512, seed=5, full_heads=LONG_FULL_HEADS)
    assert len(bh_idx) == len(LONG_FULL_HEADS) * w.N + (BH - len(LONG_FULL_HEADS)) * 512
    o_ref, lse_ref = oracle.rows(q, k, v, causal, w.scale, bh_idx, row_idx)
    of = o.reshape(BH, w.N, w.D).double().numpy()[bh_idx, row_idx]
    lf = lse.reshape(BH, w.N).double().numpy()[bh_idx, row_idx]
    err = np.abs(of - o_ref)
    emax = float(err.max())
    lmax = float(np.abs(lf - lse_ref).max())
    worst = int(err.max(axis=1).argmax())
    print(f"{name}: {len(bh_idx)} rows, max|dO|={emax:.3e} (head {bh_idx[worst]} row {row_idx[worst]}) "
          f"mean|dO|={float(err.mean()):.3e} max|dLSE|={lmax:.3e}")
    assert emax <= TOL_O[w.dtype] and lmax <= TOL_LSE
    # every output row is a convex combination of V rows: finite and bounded by max|V|
    assert torch.isfinite(o.float()).all()
    assert float(o.float().abs().max()) <= float(v.float().abs().max()) * 1.01


@pytest.mark.parametrize("D", [64, 128])
def test_tail_split_long_tiles(D):
    """B1 H8 N8192 non-causal: 256 CTA tiles of 64 key steps on the GPU's
    SMs, which the automatic schedule runs as a tail split (each CTA a whole
    tile, the last wave's 104 tiles cut into parts and merged).  Heads 0 and
    7 are compared in full, 512 rows of every other head."""
    q, k, v = make_custom(1, 8, 8192, D, "bf16", seed=8192 + D)
    scale = D ** -0.5
    o, lse = _run(q, k, v, False, scale)
    bh_idx, row_idx = _sample_rows(8, 8192, 512, seed=9, full_heads=(0, 7))
    o_ref, lse_ref = oracle.rows(q, k, v, False, scale, bh_idx, row_idx)
    of = o.reshape(8, 8192, D).double().numpy()[bh_idx, row_idx]
    lf = lse.reshape(8, 8192).double().numpy()[bh_idx, row_idx]
    emax = float(np.abs(of - o_ref).max())
    lmax = float(np.abs(lf - lse_ref).max())
    print(f"tail split D{D}: {len(bh_idx)} rows, max|dO|={emax:.3e} max|dLSE|={lmax:.3e}")
    assert emax <= TOL_O["bf16"] and lmax <= TOL_LSE


EDGE_N = [1, 2, 3, 64, 127, 128, 129, 255, 256, 257, 383, 384, 513]


@pytest.mark.parametrize("schedule", ["auto", "balanced"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("N", EDGE_N)
def test_edge_lengths(N, dtype, D, schedule):
    q, k, v = make_custom(2, 3, N, D, dtype, seed=N + D)
    for causal in (False, True):
        _check_full(q, k, v, causal, 1.0 / math.sqrt(D), dtype, f"N{N} D{D} {dtype}", schedule)


@pytest.mark.parametrize("causal", [False, True])
def test_schedules_agree(causal):
    """Whole tiles and balanced parts compute the same function.  They are not
    bit-identical: a part rounds its probabilities P to bf16 relative to its
    own running row max before the P.V product ("How to profile and optimise
    kernels", the P cast section), so the two differ at the scale of that
    rounding plus the output rounding it tips.  Each lies within a mean
    |dO| of 6e-5 of the exact result at this size (test_n4096...), so their
    mean difference is bounded by the same figure; the maximum stays far inside
    the bf16 tolerance.  (Measured: max 4.9e-4, mean 2.1e-5, LSE 1.9e-6.)"""
    q, k, v = (x.cuda() for x in make_custom(1, 8, 4096, 64, "bf16", seed=21))
    o1, l1 = fa.forward(q, k, v, causal=causal, schedule="whole_tiles")
    o2, l2 = fa.forward(q, k, v, causal=causal, schedule="balanced")
    assert fa.sync_status(torch.cuda.current_stream().cuda_stream) == 0
    d = (o1.float() - o2.float()).abs()
    dl = float((l1 - l2).abs().max())
    print(f"causal={int(causal)}: max|dO|={float(d.max()):.3e} mean|dO|={float(d.mean()):.3e} max|dLSE|={dl:.3e}")
    assert float(d.max()) <= 2e-3 and float(d.mean()) <= 6e-5
    assert dl <= 1e-4


def test_two_library_copies_in_one_process(tmp_path):
    """A second, separately loaded copy of the library launches its own
    kernels correctly (its launch set-up is private to it)."""
    import ctypes
    import shutil
    from exact_attention_10_gb300 import build as fa_build
    copy = str(tmp_path / "libfa_copy.so")
    shutil.copy(fa_build.LIB_PATH, copy)
    lib2 = fa.load(copy)
    w = WORKLOADS["b2h16_n4096"]
    q, k, v = (x.cuda() for x in make_qkv(w, seed=0))
    o1, l1 = fa.forward(q, k, v, causal=False, scale=w.scale, schedule="balanced")
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    st = torch.cuda.current_stream().cuda_stream
    for sched in (1, 2):   # whole tiles, balanced
        rc = lib2.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(), w.B, w.H, w.N,
                            w.D, 0, ctypes.c_float(w.scale), 0, sched, ctypes.c_void_p(st))
        assert rc == 0, rc
        assert lib2.fa_sync_status(ctypes.c_void_p(st)) == 0
        if sched == 2:
            assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_rejects_unknown_schedule():
    w = WORKLOADS["tiny_n256"]
    q, k, v = (x.cuda() for x in make_qkv(w, seed=0))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    rc = fa.fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 256, 64, 0,
                    0.125, 0, 0, schedule=3)
    assert rc == 1   # FA_ERR_INVALID_VALUE


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_large_logits_stay_finite(dtype):
    """Q and K amplified 4x at N = 513 ("Building a Verifiable FlashAttention
    Forward from PyTorch to Triton", Part 4: the stability case): finite
    everywhere and within tolerance.

    In bf16 this case produces outputs with |O_ref| >= 4, where the spacing of
    bf16 values is 2^-5: the exact answer rounded to bf16 can itself be more
    than 1e-2 away from O_ref (4.208 -> 4.21875 is 0.0107).  So for bf16 the
    1e-2 bound is applied strictly where |O_ref| < 4 (half a bf16 step there is
    at most 2^-8), and elsewhere to the error in excess of that unavoidable
    output-rounding floor.  fp16 is held to 2e-3 everywhere."""
    q, k, v = make_custom(1, 4, 513, 64, dtype, seed=7, qk_gain=4.0)
    for causal in (False, True):
        o, lse = _run(q, k, v, causal, 1.0 / 8)
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        o_ref, lse_ref = oracle.forward(q, k, v, causal, 1.0 / 8)
        emax, _, lmax, err = _report(o, lse, o_ref, lse_ref)
        assert lmax <= TOL_LSE
        if dtype == "fp16":
            assert emax <= TOL_O["fp16"], emax
            continue
        floor = np.abs(torch.from_numpy(o_ref).to(torch.bfloat16).double().numpy() - o_ref)
        small = np.abs(o_ref) < 4.0
        print(f"amplified bf16 causal={int(causal)}: max|dO|={emax:.3e}, "
              f"max over |O_ref|<4: {err[small].max():.3e}, max excess over rounding floor: "
              f"{(err - floor).max():.3e}")
        assert err[small].max() <= TOL_O["bf16"]
        assert (err - floor).max() <= TOL_O["bf16"]


def test_deterministic_and_no_out_of_bounds_writes():
    """Two launches give identical bits; bytes just outside O and LSE are untouched."""
    B, H, N, D = 2, 4, 777, 128
    q, k, v = (x.cuda() for x in make_custom(B, H, N, D, "bf16", seed=11))
    pad = 4096
    o_buf = torch.full((B * H * N * D + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * H * N + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[pad:pad + B * H * N * D].view(B, H, N, D)
    lse = l_buf[pad:pad + B * H * N].view(B, H, N)
    for causal, schedule in ((False, "auto"), (True, "auto"), (False, "balanced"), (True, "balanced")):
        fa.forward(q, k, v, causal=causal, out=o, lse=lse, schedule=schedule)
        first = (o.clone(), lse.clone())
        fa.forward(q, k, v, causal=causal, out=o, lse=lse, schedule=schedule)
        torch.cuda.synchronize()
        assert torch.equal(first[0], o) and torch.equal(first[1], lse)
        for buf in (o_buf, l_buf):
            assert bool((buf[:pad].float() == 7.0).all()) and bool((buf[-pad:].float() == 7.0).all())


def test_side_stream_and_status():
    w = WORKLOADS["tiny_n256"]
    q, k, v = (x.cuda() for x in make_qkv(w, seed=0))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    assert fa.sync_status(s.cuda_stream) == 0
    o_ref, _ = oracle.forward(q.cpu(), k.cpu(), v.cpu(), True, w.scale)
    assert float(np.abs(o.cpu().double().numpy() - o_ref).max()) <= TOL_O["bf16"]


def test_rejects_host_memory():
    w = WORKLOADS["tiny_n256"]
    q, k, v = make_qkv(w, seed=0)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32)
    rc = fa.fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 256, 64, 0,
                    0.125, 0, 0)
    assert rc == 1   # FA_ERR_INVALID_VALUE


# --- queries against a different number of keys (fa_fwd_qkv) ----------------

RECT = [  # (B, H, Nq, Nkv, D, dtype)
    (1, 8, 1, 4096, 64, "bf16"),        # decode: one query, long K/V
    (2, 4, 16, 2000, 128, "fp16"),
    (1, 4, 127, 1000, 64, "bf16"),
    (2, 2, 200, 70, 128, "bf16"),       # more queries than keys
    (1, 3, 513, 200, 64, "fp16"),       # causal: the first 313 rows see no key
    (1, 2, 300, 1, 64, "bf16"),
    (1, 2, 1000, 129, 128, "bf16"),
]


def _rect(B, H, Nq, Nkv, D, dtype, seed):
    q = make_custom(B, H, Nq, D, dtype, seed=seed)[0]
    _, k, v = make_custom(B, H, Nkv, D, dtype, seed=seed + 1)
    return q, k, v


@pytest.mark.parametrize("schedule", ["auto", "balanced"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nkv,D,dtype", RECT)
def test_queries_against_other_key_counts(B, H, Nq, Nkv, D, dtype, causal, schedule):
    q, k, v = _rect(B, H, Nq, Nkv, D, dtype, seed=Nq + Nkv)
    scale = D ** -0.5
    dev = torch.device("cuda:0")
    o, lse = fa.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale, schedule=schedule)
    assert fa.sync_status(torch.cuda.current_stream(dev).cuda_stream) == 0
    o_ref, lse_ref = oracle.forward_qkv(q, k, v, causal, scale)
    od = o.cpu().double().numpy()
    ld = lse.cpu().double().numpy()
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(ld), empty)
    assert (od[empty] == 0.0).all()   # rows that see no key: O = 0 exactly
    emax = float(np.abs(od - o_ref).max())
    lmax = float(np.abs(ld[~empty] - lse_ref[~empty]).max()) if (~empty).any() else 0.0
    print(f"Nq={Nq} Nkv={Nkv} D={D} {dtype} causal={int(causal)} {schedule}: max|dO|={emax:.3e} "
          f"max|dLSE|={lmax:.3e} empty rows={int(empty.sum())}")
    assert emax <= TOL_O[dtype] and lmax <= TOL_LSE


@pytest.mark.parametrize("causal", [False, True])
def test_split_kv_decode_long_context(causal):
    """Decoding 4 queries against 32768 keys over 32 heads: 32 CTA tiles of
    256 steps, which the balanced schedule cuts into parts across the SMs and
    merges by LSE (split-KV); compared in full with the oracle."""
    q, k, v = _rect(1, 32, 4, 32768, 128, "bf16", seed=9)
    dev = torch.device("cuda:0")
    outs = {}
    for schedule in ("whole_tiles", "balanced"):
        outs[schedule] = fa.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=128 ** -0.5,
                                    schedule=schedule)
    assert fa.sync_status(torch.cuda.current_stream(dev).cuda_stream) == 0
    o_ref, lse_ref = oracle.forward_qkv(q, k, v, causal, 128 ** -0.5)
    for schedule, (o, lse) in outs.items():
        emax = float(np.abs(o.cpu().double().numpy() - o_ref).max())
        lmax = float(np.abs(lse.cpu().double().numpy() - lse_ref).max())
        print(f"decode {schedule} causal={int(causal)}: max|dO|={emax:.3e} max|dLSE|={lmax:.3e}")
        assert emax <= TOL_O["bf16"] and lmax <= TOL_LSE


@pytest.mark.parametrize("schedule", ["auto", "balanced"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nkv,D", [(1, 4, 2, 131072, 64), (1, 2, 33, 65536, 128), (2, 3, 64, 40000, 64)])
def test_decode_many_parts(B, H, Nq, Nkv, D, causal, schedule):
    """Few query rows against very long key sequences: the balanced schedule
    cuts each head's key steps into up to 32 parts (heads of at most 32 rows),
    16 (at most 64 rows) or 8, and the merge stages every part's row
    statistics; compared in full with the oracle."""
    q, k, v = _rect(B, H, Nq, Nkv, D, "bf16", seed=Nq + Nkv)
    scale = D ** -0.5
    dev = torch.device("cuda:0")
    o, lse = fa.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale, schedule=schedule)
    assert fa.sync_status(torch.cuda.current_stream(dev).cuda_stream) == 0
    o_ref, lse_ref = oracle.forward_qkv(q, k, v, causal, scale)
    emax = float(np.abs(o.cpu().double().numpy() - o_ref).max())
    lmax = float(np.abs(lse.cpu().double().numpy() - lse_ref).max())
    print(f"decode Nq={Nq} Nkv={Nkv} D={D} causal={int(causal)} {schedule}: max|dO|={emax:.3e} max|dLSE|={lmax:.3e}")
    assert emax <= TOL_O["bf16"] and lmax <= TOL_LSE


@pytest.mark.parametrize("schedule", ["whole_tiles", "balanced"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nkv,dtype", [(1, 700, "bf16"), (77, 1300, "fp16"), (128, 900, "bf16")])
def test_one_tile_heads_many_per_cta(Nq, Nkv, dtype, causal, schedule):
    """D = 128 heads of at most 128 query rows run the separate-P order with
    K and V released separately; 160 heads over the SMs give CTAs several
    such tiles (whole tiles) or parts (balanced) in a row, so the producer's
    hand-over of the last V between them is exercised.  Compared in full."""
    q, k, v = _rect(2, 80, Nq, Nkv, 128, dtype, seed=Nq * 7 + Nkv)
    scale = 128 ** -0.5
    dev = torch.device("cuda:0")
    o, lse = fa.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale, schedule=schedule)
    assert fa.sync_status(torch.cuda.current_stream(dev).cuda_stream) == 0
    o_ref, lse_ref = oracle.forward_qkv(q, k, v, causal, scale)
    emax = float(np.abs(o.cpu().double().numpy() - o_ref).max())
    lmax = float(np.abs(lse.cpu().double().numpy() - lse_ref).max())
    print(f"one-tile heads Nq={Nq} Nkv={Nkv} {dtype} causal={int(causal)} {schedule}: max|dO|={emax:.3e} max|dLSE|={lmax:.3e}")
    assert emax <= TOL_O[dtype] and lmax <= TOL_LSE
