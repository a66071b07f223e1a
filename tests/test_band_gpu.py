"""Sliding-window (band) masks through fa_fwd_band on the GPU, compared in
full with the oracle's band definition.

With i' = i + (Nkv - Nq), query i sees keys j in [i' - left, i' + right]; a
negative bound is unbounded.  Cases cover windows narrower than one 128-key
tile, windows that straddle tile edges, one-sided and two-sided bands, bands
wider than the sequence (which must give the unmasked result), rows whose
band holds no key (O = 0, LSE = -inf), Nq != Nkv, decode against a long
windowed context (split-KV), both dtypes and both head dimensions, and the
whole-tile and balanced schedules.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from exact_attention_10_gb300 import fa
from exact_attention_10_gb300.inputs import make_custom

pytestmark = pytest.mark.gpu

TOL_O = {"bf16": 1e-2, "fp16": 2e-3}
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load()


def _inputs(B, H, Nq, Nkv, D, dtype, seed):
    q = make_custom(B, H, Nq, D, dtype, seed=seed)[0]
    _, k, v = make_custom(B, H, Nkv, D, dtype, seed=seed + 1)
    return q, k, v


def _band(q, k, v, window, scale, schedule):
    dev = torch.device("cuda:0")
    o, lse = fa.forward(q.to(dev), k.to(dev), v.to(dev), scale=scale, schedule=schedule, window=window)
    rc = fa.sync_status(torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0, fa.status_string(rc)
    return o.cpu(), lse.cpu()


def _compare(o, lse, o_ref, lse_ref, dtype, label):
    od = o.double().numpy()
    ld = lse.double().numpy()
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(ld), empty), label
    assert (od[empty] == 0.0).all(), label   # rows whose band is empty: O = 0 exactly
    assert np.isfinite(od).all() and np.isfinite(ld[~empty]).all(), label
    emax = float(np.abs(od - o_ref).max())
    lmax = float(np.abs(ld[~empty] - lse_ref[~empty]).max()) if (~empty).any() else 0.0
    print(f"{label}: max|dO|={emax:.3e} max|dLSE|={lmax:.3e} empty rows={int(empty.sum())}")
    assert emax <= TOL_O[dtype], (label, emax)
    assert lmax <= TOL_LSE, (label, lmax)


SQUARE = [  # (B, H, N, D, dtype, (left, right))
    (1, 4, 1000, 64, "bf16", (255, 0)),      # causal sliding window of 256 keys
    (1, 4, 1000, 128, "fp16", (100, 100)),   # two-sided, narrower than a tile
    (2, 2, 777, 64, "bf16", (0, 0)),         # the diagonal alone
    (1, 3, 1500, 128, "bf16", (-1, 50)),     # bounded on the right only
    (1, 3, 1500, 64, "fp16", (300, -1)),     # bounded on the left only
    (1, 2, 2048, 64, "bf16", (127, 0)),      # window = one tile, tile-aligned length
    (1, 2, 2049, 128, "bf16", (128, 129)),   # edges one past a tile boundary
    (1, 2, 513, 64, "bf16", (600, 600)),     # wider than the sequence: no mask
    (1, 2, 300, 128, "fp16", (0, 5)),        # looking ahead only: keys i..i+5
    # unbounded on the left at D = 64: the causal kernels, whose masked steps
    # hide keys in TMEM before S is read; right edges off the 32-column chunks
    (1, 3, 1500, 64, "bf16", (-1, 50)),
    (1, 2, 777, 64, "fp16", (-1, 5)),
    (2, 2, 1000, 64, "bf16", (-1, 31)),
]


@pytest.mark.parametrize("schedule", ["whole_tiles", "balanced"])
@pytest.mark.parametrize("B,H,N,D,dtype,window", SQUARE)
def test_band_square(B, H, N, D, dtype, window, schedule):
    q, k, v = _inputs(B, H, N, N, D, dtype, seed=N + D + window[0])
    scale = D ** -0.5
    o, lse = _band(q, k, v, window, scale, schedule)
    o_ref, lse_ref = oracle.forward_band(q, k, v, window[0], window[1], scale)
    _compare(o, lse, o_ref, lse_ref, dtype, f"N={N} D={D} {dtype} window={window} {schedule}")


RECT = [  # (B, H, Nq, Nkv, D, dtype, (left, right))
    (1, 4, 300, 2000, 128, "fp16", (511, 0)),   # last 300 positions of a 2000-token windowed sequence
    (1, 3, 513, 200, 64, "bf16", (50, 10)),     # more queries than keys: the first rows see nothing
    (2, 2, 64, 5000, 64, "bf16", (1023, 0)),
    (1, 2, 1000, 129, 128, "bf16", (-1, 3)),
    (1, 2, 1, 4096, 64, "bf16", (1000, 0)),     # decode with a window
]


@pytest.mark.parametrize("schedule", ["auto", "whole_tiles", "balanced"])
@pytest.mark.parametrize("B,H,Nq,Nkv,D,dtype,window", RECT)
def test_band_other_key_counts(B, H, Nq, Nkv, D, dtype, window, schedule):
    q, k, v = _inputs(B, H, Nq, Nkv, D, dtype, seed=Nq + Nkv)
    scale = D ** -0.5
    o, lse = _band(q, k, v, window, scale, schedule)
    o_ref, lse_ref = oracle.forward_band(q, k, v, window[0], window[1], scale)
    _compare(o, lse, o_ref, lse_ref, dtype, f"Nq={Nq} Nkv={Nkv} D={D} {dtype} window={window} {schedule}")


def test_band_decode_long_windowed_context():
    """Four queries against 65536 keys over 16 heads with a window of 8192:
    each head's 64 visible key tiles are split across CTAs (split-KV) and
    merged by LSE; compared in full with the oracle."""
    q, k, v = _inputs(1, 16, 4, 65536, 128, "bf16", seed=21)
    scale = 128 ** -0.5
    o_ref, lse_ref = oracle.forward_band(q, k, v, 8191, 0, scale)
    for schedule in ("whole_tiles", "balanced", "auto"):
        o, lse = _band(q, k, v, (8191, 0), scale, schedule)
        _compare(o, lse, o_ref, lse_ref, "bf16", f"decode window=8192 {schedule}")


@pytest.mark.parametrize("schedule", ["whole_tiles", "balanced"])
@pytest.mark.parametrize("Nq,Nkv,window,dtype", [(16, 2000, (500, 0), "bf16"), (77, 1500, (300, 40), "fp16")])
def test_band_one_tile_heads_many_per_cta(Nq, Nkv, window, dtype, schedule):
    """D = 128 heads of at most 128 query rows under a band run the one-tile
    order (K and V released separately); 160 heads give CTAs several such
    tiles (whole tiles) or parts (balanced), so the producer hands a part's
    last V over from a band's first key step on.  Compared in full."""
    q, k, v = _inputs(2, 80, Nq, Nkv, 128, dtype, seed=Nq * 5 + Nkv)
    scale = 128 ** -0.5
    o, lse = _band(q, k, v, window, scale, schedule)
    o_ref, lse_ref = oracle.forward_band(q, k, v, window[0], window[1], scale)
    _compare(o, lse, o_ref, lse_ref, dtype, f"one-tile band Nq={Nq} Nkv={Nkv} window={window} {dtype} {schedule}")


@pytest.mark.parametrize("D", [64, 128])
def test_band_reduces_to_the_plain_masks(D):
    """The band (-1, 0) is fa_fwd_qkv's causal mask and (-1, -1) no mask: same
    kernels, bit-identical results.  A finite band wider than the sequence
    runs the masked kernel but sees every key, so it equals the unmasked
    result bit for bit when both run whole tiles (same key order per row)."""
    q, k, v = _inputs(1, 4, 1500, 1500, D, "bf16", seed=D)
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    scale = D ** -0.5
    for causal, window in ((True, (-1, 0)), (False, (-1, -1))):
        ref = fa.forward(qd, kd, vd, causal=causal, scale=scale)
        got = fa.forward(qd, kd, vd, scale=scale, window=window)
        assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1])
    ref = fa.forward(qd, kd, vd, causal=False, scale=scale, schedule="whole_tiles")
    got = fa.forward(qd, kd, vd, scale=scale, window=(1500, 1500), schedule="whole_tiles")
    assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1])
    assert fa.sync_status(torch.cuda.current_stream(dev).cuda_stream) == 0


def test_band_long_sequence_sampled_rows():
    """N = 32768 with a causal window of 4096 (the workload shape of
    sliding-window long-context attention), checked on sampled rows: row i
    needs only keys [i - 4095, i], so the oracle's band call on that slice
    (one query against 4096 keys, window (4095, 0)) is the exact row."""
    B, H, N, D = 1, 8, 32768, 128
    q, k, v = _inputs(B, H, N, N, D, "bf16", seed=5)
    scale = D ** -0.5
    o, lse = _band(q, k, v, (4095, 0), scale, "auto")
    rng = np.random.default_rng(7)
    rows = np.concatenate([[0, 1, 127, 128, 4095, 4096, 4097, N - 1], rng.integers(0, N, 24)])
    for h in range(H):
        for i in rows:
            lo = max(0, int(i) - 4095)
            o_ref, lse_ref = oracle.forward_band(q[0, h, i:i + 1], k[0, h, lo:i + 1], v[0, h, lo:i + 1], 4095, 0, scale)
            e = float(np.abs(o[0, h, i].double().numpy() - o_ref[0]).max())
            le = abs(float(lse[0, h, i]) - float(lse_ref[0]))
            assert e <= TOL_O["bf16"] and le <= TOL_LSE, (h, int(i), e, le)
