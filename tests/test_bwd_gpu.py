"""Attention backward (fa_bwd) on the GPU against the fp64 oracle's gradients.

The CUDA path takes O and LSE from the library's own forward (as a training
step would) and an upstream gradient dO; the oracle differentiates the exact
attention of the same Q, K, V.  Errors are measured normwise per gradient,
||g - g_ref|| / ||g_ref||, and row by row: each row's largest element error
against that row's own largest reference element plus the gradient's RMS
(see BOUNDS).  Cases cover D = 64 and 128, bf16 and fp16,
causal and not, one and several 128-row tiles, ragged lengths, N = 1, a
4096-row sequence compared in full, and CTAs that run several key tiles.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from exact_attention_10_gb300 import fa
from exact_attention_10_gb300.inputs import make_custom

pytestmark = pytest.mark.gpu

# Rounding in the path, per element: P and dS are rounded to the input type
# for the tensor-core products, O (an input, from the forward) and the three
# outputs are in the input type; the products accumulate in fp32.  With unit
# roundoff u (2^-8 bf16, 2^-11 fp16), each rounding contributes at most u/2
# relative to the terms it touches, and four of them stack on dK and dQ (O via
# delta, dS, the output, and P inside dS's factor), so the normwise error is
# bounded by about 2u.
#
# The bounds are set from the errors measured on a GB300 over the cases below
# (both dtypes, D = 64 and 128, causal and not, N from 128 to 4096), with a
# stated margin:
#   normwise: measured at most 0.67u on every gradient; bound 1.5u (2.2x).
#   per row r of a gradient (a query row of dQ, a key row of dK and dV):
#     max_d |g - g_ref|  <=  12u * (max_d |g_ref[r]| + rms(g_ref)).
#   A row's error scales with its own magnitude, and rows whose exact
#   gradient is (nearly) zero -- causal row 0 of dQ, where P = 1 and dS = 0,
#   and the first few causal rows -- keep an error from the fp32 cancellation
#   in dP - delta, set by the gradient's overall scale, hence the RMS term.
#   Measured at most 7.6u (dQ of the first causal rows: row 1 of a head, in
#   bf16); bound 12u (1.6x).
# A wrong term on any row of ordinary magnitude shows as an error of the
# order of that row itself, hundreds of u.
U = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}
BOUNDS = {dt: {"norm": 1.5 * u, "row": 12 * u} for dt, u in U.items()}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load()


def _inputs(B, H, N, D, dtype, seed):
    q, k, v = make_custom(B, H, N, D, dtype, seed=seed)
    do = make_custom(B, H, N, D, dtype, seed=seed + 7)[0]
    return q, k, v, do


def _gpu_grads(q, k, v, do, causal, scale, deterministic=False):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(qd, kd, vd, o, dod, lse, causal=causal, scale=scale, deterministic=deterministic)
    rc = fa.sync_status(torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0, fa.status_string(rc)
    return dq.cpu(), dk.cpu(), dv.cpu()


def _rms(x):
    return float(np.sqrt(np.mean(np.square(x)))) if x.size else 0.0


def _errors(g, ref, floor):
    """(normwise error, worst per-row error ratio, its row): the row ratio is
    max_d |g - g_ref| / (max_d |g_ref[r]| + floor) over rows r, floor being
    the gradient's RMS.  (The normwise error of an identically zero reference
    is taken against the floor.)"""
    gd = g.double().numpy().reshape(ref.shape)
    assert np.isfinite(gd).all()
    nref = float(np.linalg.norm(ref))
    norm = float(np.linalg.norm(gd - ref)) / (nref if nref > 0 else floor * np.sqrt(ref.size))
    D = ref.shape[-1]
    err = np.abs(gd - ref).reshape(-1, D).max(axis=1)
    scale = np.abs(ref).reshape(-1, D).max(axis=1) + floor
    ratio = err / scale
    worst = int(ratio.argmax())
    return norm, float(ratio[worst]), worst


def _check(grads, refs, dtype, label):
    u = U[dtype]
    # A gradient whose exact value is zero everywhere (one visible key per
    # query: P = 1, dS = 0, so dQ = dK = 0) keeps only the fp32 cancellation
    # residue of dP - delta; its floor is the RMS of all three gradients.
    rms_all = _rms(np.concatenate([r.reshape(-1) for r in refs]))
    for name, g, ref in zip(("dQ", "dK", "dV"), grads, refs):
        norm, row, where = _errors(g, ref, _rms(ref) or rms_all)
        print(f"{label} {name}: normwise {norm / u:.2f}u  worst row {row / u:.2f}u (flattened row {where})")
        assert norm <= BOUNDS[dtype]["norm"], (label, name, norm / u)
        assert row <= BOUNDS[dtype]["row"], (label, name, row / u, where)


CASES = [  # (B, H, N, D, dtype)
    (1, 2, 128, 64, "bf16"),
    (1, 2, 256, 128, "fp16"),
    (2, 3, 300, 64, "bf16"),      # ragged: 3 tiles, the last 44 rows
    (1, 2, 1000, 128, "bf16"),
    (2, 2, 777, 128, "fp16"),
    (1, 3, 513, 64, "fp16"),
    (1, 4, 129, 128, "bf16"),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,D,dtype", CASES)
def test_backward_matches_oracle(B, H, N, D, dtype, causal):
    """At D = 64 both dQ paths: the fused pass (the default) and the second
    pass (deterministic)."""
    q, k, v, do = _inputs(B, H, N, D, dtype, seed=N + D)
    scale = D ** -0.5
    refs = oracle.backward(q, k, v, do, causal, scale)
    for det in ((False, True) if D == 64 else (False,)):
        grads = _gpu_grads(q, k, v, do, causal, scale, deterministic=det)
        _check(grads, refs, dtype, f"B{B} H{H} N{N} D{D} {dtype} causal={int(causal)} deterministic={int(det)}")


@pytest.mark.parametrize("D", [64, 128])
def test_backward_single_row(D):
    """N = 1: P = 1 and dS = 0 in exact arithmetic.  P rounds to exactly 1,
    so dV = dO bit for bit; dS is left with the fp32 rounding of dP - delta
    (two sums of the same products in different orders), so dQ and dK are
    tiny rather than zero."""
    q, k, v, do = _inputs(2, 3, 1, D, "bf16", seed=D)
    for causal in (False, True):
        dq, dk, dv = _gpu_grads(q, k, v, do, causal, D ** -0.5)
        assert dq.abs().max().item() <= 1e-3 and dk.abs().max().item() <= 1e-3
        assert torch.equal(dv, do)


def test_backward_deterministic_and_invariant():
    """Two deterministic calls give identical bits (no atomics), and the key
    rows of dK sum to (nearly) zero per head, as every row of dS does."""
    B, H, N, D = 2, 4, 1000, 64
    q, k, v, do = _inputs(B, H, N, D, "bf16", seed=3)
    a = _gpu_grads(q, k, v, do, True, D ** -0.5, deterministic=True)
    b = _gpu_grads(q, k, v, do, True, D ** -0.5, deterministic=True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    dk = a[1].double()
    colsum = dk.sum(dim=2).abs().max().item()
    assert colsum <= 1e-2 * dk.abs().sum(dim=2).max().item()


@pytest.mark.parametrize("causal", [False, True])
def test_backward_fused_against_two_pass(causal):
    """The D = 64 fused pass against the two-pass path on the same inputs:
    dK and dV come from the same arithmetic in the same order (bit for bit,
    and on every call); dQ differs only by the order of its fp32 adds, so
    within a few fp32 roundings of its accumulation, far below the 16-bit
    output step (checked: at most one unit in the last place of dQ's type,
    with a floor of 2^-16 of the largest |dQ| for elements that cancel)."""
    B, H, N, D = 2, 4, 1000, 64
    q, k, v, do = _inputs(B, H, N, D, "bf16", seed=5)
    det = _gpu_grads(q, k, v, do, causal, D ** -0.5, deterministic=True)
    f1 = _gpu_grads(q, k, v, do, causal, D ** -0.5)
    f2 = _gpu_grads(q, k, v, do, causal, D ** -0.5)
    for x in (f1, f2):
        assert torch.equal(x[1], det[1]) and torch.equal(x[2], det[2])
        a, b = x[0].float(), det[0].float()
        ulp = torch.maximum(a.abs(), b.abs()) * 2.0 ** -7 + b.abs().max() * 2.0 ** -16
        assert bool(((a - b).abs() <= ulp).all()), float(((a - b).abs() / ulp).max())


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_long_sequence(causal, D):
    """N = 4096 over two heads (32 key tiles per head, every combination of
    diagonal and full tiles), compared in full; at D = 64 the fused pass, whose
    dQ sums 32 key tiles' products in the fp32 accumulator."""
    q, k, v, do = _inputs(1, 2, 4096, D, "bf16", seed=11)
    scale = D ** -0.5
    grads = _gpu_grads(q, k, v, do, causal, scale)
    refs = oracle.backward(q, k, v, do, causal, scale)
    _check(grads, refs, "bf16", f"N4096 D{D} causal={int(causal)}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_several_tiles_per_cta(causal, D):
    """B4 H16 N1024: 512 key tiles over the SMs, so every CTA runs several
    (of uneven length when causal) and the passes' hand-over from one key tile
    to the next -- the resident tiles reloaded, the accumulators read out and
    restarted, the next tile's first S and dP -- is exercised on every CTA.
    Four heads spread over the batch are compared in full."""
    B, H, N = 4, 16, 1024
    q, k, v, do = _inputs(B, H, N, D, "bf16", seed=23)
    scale = D ** -0.5
    grads = _gpu_grads(q, k, v, do, causal, scale)
    for b, h in ((0, 0), (1, 5), (2, 10), (3, 15)):
        sl = lambda x: x[b:b + 1, h:h + 1]
        refs = oracle.backward(sl(q), sl(k), sl(v), sl(do), causal, scale)
        _check(tuple(sl(g) for g in grads), refs, "bf16", f"B4 H16 N1024 D{D} causal={int(causal)} b{b} h{h}")


BAND = [  # (B, H, Nq, Nkv, D, dtype, (left, right))
    (1, 2, 1000, 1000, 64, "bf16", (255, 0)),     # causal sliding window
    (1, 2, 777, 777, 128, "fp16", (100, 100)),    # two-sided, narrower than a tile
    (1, 2, 300, 2000, 64, "bf16", (511, 0)),      # the last 300 positions of a longer sequence
    (1, 2, 513, 200, 128, "bf16", (50, 10)),      # more queries than keys: rows without keys, keys without queries
    (2, 2, 600, 600, 64, "bf16", (-1, 0)),        # causal through the band entry point
    (1, 3, 129, 1000, 128, "bf16", (-1, 0)),      # Nq != Nkv, bottom-right causal
    (1, 2, 1500, 1500, 64, "fp16", (300, -1)),    # bounded on the left only
    (1, 2, 1000, 1000, 128, "bf16", (-1, -1)),    # no mask through the band entry point
    (1, 2, 2048, 2048, 64, "bf16", (0, 0)),       # the diagonal alone
]


@pytest.mark.parametrize("B,H,Nq,Nkv,D,dtype,window", BAND)
def test_backward_band_matches_oracle(B, H, Nq, Nkv, D, dtype, window):
    """fa_bwd_band against the oracle's band gradients, from the forward's own
    O and LSE under the same window."""
    q = make_custom(B, H, Nq, D, dtype, seed=Nq)[0]
    _, k, v = make_custom(B, H, Nkv, D, dtype, seed=Nkv + 1)
    do = make_custom(B, H, Nq, D, dtype, seed=Nq + 7)[0]
    scale = D ** -0.5
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, scale=scale, window=window)
    grads = fa.backward(qd, kd, vd, o, dod, lse, scale=scale, window=window)
    rc = fa.sync_status(torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0, fa.status_string(rc)
    refs = oracle.backward_band(q, k, v, do, window[0], window[1], scale)
    _check([g.cpu() for g in grads], refs, dtype, f"Nq{Nq} Nkv{Nkv} D{D} {dtype} window={window}")
    # Rows the band leaves empty are exactly zero: queries that see no key
    # (dQ) and keys that no query sees (dK, dV).
    ii = np.arange(Nq)[:, None] + (Nkv - Nq)
    jj = np.arange(Nkv)[None, :]
    vis = np.ones((Nq, Nkv), dtype=bool)
    if window[0] >= 0:
        vis &= jj >= ii - window[0]
    if window[1] >= 0:
        vis &= jj <= ii + window[1]
    for g, empty in zip(grads, (~vis.any(axis=1), ~vis.any(axis=0), ~vis.any(axis=0))):
        got = g.cpu()
        assert (got[:, :, empty] == 0).all()
