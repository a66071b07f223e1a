"""Attention backward (fa_bwd) on the GPU against the fp64 oracle's gradients.

The CUDA path takes O and LSE from the library's own forward (as a training
step would) and an upstream gradient dO; the oracle differentiates the exact
attention of the same Q, K, V.  Errors are measured normwise per gradient,
||g - g_ref|| / ||g_ref||, plus the largest element error relative to the
largest reference element, against bounds derived from the rounding the
path performs (see BOUNDS).  Cases cover D = 64 and 128, bf16 and fp16,
causal and not, one and several 128-row tiles, ragged lengths, N = 1, and a
4096-row sequence compared in full.
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
# bounded by about 2u; the bounds below allow 4u normwise and 16u on the
# largest element relative to the largest reference element.
U = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}
BOUNDS = {dt: {"norm": 4 * u, "max": 16 * u} for dt, u in U.items()}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load()


def _inputs(B, H, N, D, dtype, seed):
    q, k, v = make_custom(B, H, N, D, dtype, seed=seed)
    do = make_custom(B, H, N, D, dtype, seed=seed + 7)[0]
    return q, k, v, do


def _gpu_grads(q, k, v, do, causal, scale):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    rc = fa.sync_status(torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0, fa.status_string(rc)
    return dq.cpu(), dk.cpu(), dv.cpu()


def _errors(g, ref):
    gd = g.double().numpy().reshape(ref.shape)
    assert np.isfinite(gd).all()
    nref = float(np.linalg.norm(ref))
    norm = float(np.linalg.norm(gd - ref)) / nref if nref > 0 else float(np.linalg.norm(gd))
    mref = float(np.abs(ref).max())
    mx = float(np.abs(gd - ref).max()) / mref if mref > 0 else float(np.abs(gd).max())
    return norm, mx


def _check(grads, refs, dtype, label):
    for name, g, ref in zip(("dQ", "dK", "dV"), grads, refs):
        norm, mx = _errors(g, ref)
        print(f"{label} {name}: normwise {norm:.2e}  max/max|ref| {mx:.2e}")
        assert norm <= BOUNDS[dtype]["norm"], (label, name, norm)
        assert mx <= BOUNDS[dtype]["max"], (label, name, mx)


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
    q, k, v, do = _inputs(B, H, N, D, dtype, seed=N + D)
    scale = D ** -0.5
    grads = _gpu_grads(q, k, v, do, causal, scale)
    refs = oracle.backward(q, k, v, do, causal, scale)
    _check(grads, refs, dtype, f"B{B} H{H} N{N} D{D} {dtype} causal={int(causal)}")


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
    """Two calls give identical bits (no atomics), and the key rows of dK sum
    to (nearly) zero per head, as every row of dS does."""
    B, H, N, D = 2, 4, 1000, 64
    q, k, v, do = _inputs(B, H, N, D, "bf16", seed=3)
    a = _gpu_grads(q, k, v, do, True, D ** -0.5)
    b = _gpu_grads(q, k, v, do, True, D ** -0.5)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    dk = a[1].double()
    colsum = dk.sum(dim=2).abs().max().item()
    assert colsum <= 1e-2 * dk.abs().sum(dim=2).max().item()


@pytest.mark.parametrize("causal", [False, True])
def test_backward_long_sequence(causal):
    """N = 4096, D = 128 over two heads (32 key tiles per head, every
    combination of diagonal and full tiles), compared in full."""
    q, k, v, do = _inputs(1, 2, 4096, 128, "bf16", seed=11)
    scale = 128 ** -0.5
    grads = _gpu_grads(q, k, v, do, causal, scale)
    refs = oracle.backward(q, k, v, do, causal, scale)
    _check(grads, refs, "bf16", f"N4096 D128 causal={int(causal)}")
