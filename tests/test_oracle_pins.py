"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: a closed form, an
invariant the pages state, an independent library routine (PyTorch's fp64 CPU
scaled-dot-product attention, scipy's softmax, torch's dtype conversion), a
brute-force equivalence on tiny inputs, or a figure the pages print.  The
pins are chosen so that a plausible slip anywhere in the oracle (a dropped
scale, a wrong causal index, V swapped for K, a missing normalisation, an
inverted rescale, log2 for ln) fails at least one of them;
``test_oracle_mutants.py`` plants such slips and checks exactly that.

Every test takes the oracle library handle as a parameter so the mutant test
can rerun them against a deliberately broken build.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# Every scale used below is exactly representable in float32: the oracle, like
# the library, takes the softmax scale as a float32 value.

def _rand(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


# ---------------------------------------------------------------------------
# Individual pins (each a plain function of the library handle)
# ---------------------------------------------------------------------------

def pin_decode(lib):
    """bf16/fp16 decoding equals torch's exact widening, for every bit pattern."""
    bits = np.arange(65536, dtype=np.uint16)
    for name, tdt in (("bf16", torch.bfloat16), ("fp16", torch.float16)):
        ours = oracle.decode(bits, name, lib=lib)
        ref = torch.from_numpy(bits.view(np.int16).copy()).view(tdt).to(torch.float64).numpy()
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(ours), nan), name
        assert np.array_equal(ours[~nan], ref[~nan]), name


def pin_rows_sum_to_one(lib):
    """Each row of softmax(S) sums to 1; masked entries (j > i under causal) are 0.

    "Triton: FlashAttention-2 Forward Pass", Verification checklist / Bugs
    found: check that each softmax row sums to 1."""
    for causal in (False, True):
        for N, D in ((1, 1), (5, 3), (17, 8)):
            q, k = _rand((N, D), 1), _rand((N, D), 2)
            P = oracle.probs(q, k, causal, 0.6875, lib=lib)
            assert np.all(P >= 0.0)
            assert np.allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
            if causal:
                assert np.all(P[np.triu_indices(N, 1)] == 0.0)


def pin_probs_vs_scipy(lib):
    """softmax(S) equals scipy.special.softmax of the scaled scores with a -inf causal mask."""
    from scipy.special import softmax
    for causal in (False, True):
        q, k = _rand((9, 6), 3), _rand((9, 6), 4)
        s = 0.375
        S = s * (q @ k.T)
        if causal:
            S = np.where(np.triu(np.ones((9, 9), bool), 1), -np.inf, S)
        ref = softmax(S, axis=1)
        P = oracle.probs(q, k, causal, s, lib=lib)
        assert np.allclose(P, ref, rtol=0, atol=1e-14)


def pin_constant_v(lib):
    """Constant V gives constant O: O is a convex combination of V rows.

    "A09 - Advanced Triton & FlashAttention", 3. Deep Dive: acc / l is
    softmax(s) @ V, an exact identity."""
    for causal in (False, True):
        q, k = _rand((2, 13, 5), 5), _rand((2, 13, 5), 6)
        v = np.full((2, 13, 5), 0.0)
        v[..., :] = np.array([1.5, -2.0, 0.25, 3.0, -0.125])
        O, _ = oracle.forward(q, k, v, causal, 0.875, lib=lib)
        assert np.allclose(O, v, rtol=0, atol=1e-14)


def pin_identical_keys(lib):
    """All keys equal: uniform weights, O = mean of the visible V rows and
    LSE = x + log|J| with x the common scaled score (closed form)."""
    N, D = 11, 4
    q = _rand((N, D), 7)
    k = np.tile(_rand((1, D), 8), (N, 1))
    v = _rand((N, D), 9)
    s = 0.625
    for causal in (False, True):
        O, L = oracle.forward(q, k, v, causal, s, lib=lib)
        x = s * (q @ k[0])
        for i in range(N):
            n = i + 1 if causal else N
            assert np.allclose(O[i], v[:n].mean(axis=0), rtol=0, atol=1e-14)
            assert abs(L[i] - (x[i] + math.log(n))) < 1e-13


def pin_zero_query(lib):
    """Q = 0 makes every score 0: O = mean of visible V, LSE = log|J|."""
    N, D = 9, 3
    q = np.zeros((N, D))
    k, v = _rand((N, D), 10), _rand((N, D), 11)
    for causal in (False, True):
        O, L = oracle.forward(q, k, v, causal, 1.25, lib=lib)
        for i in range(N):
            n = i + 1 if causal else N
            assert np.allclose(O[i], v[:n].mean(axis=0), rtol=0, atol=1e-14)
            assert abs(L[i] - math.log(n)) < 1e-14


def pin_causal_row0(lib):
    """Under the causal mask row 0 sees only key 0: O[0] = V[0], LSE[0] = s q0.k0."""
    q, k, v = _rand((3, 7, 6), 12), _rand((3, 7, 6), 13), _rand((3, 7, 6), 14)
    s = 0.4375
    O, L = oracle.forward(q, k, v, True, s, lib=lib)
    assert np.array_equal(O[:, 0], v[:, 0])
    assert np.allclose(L[:, 0], s * np.einsum("bd,bd->b", q[:, 0], k[:, 0]), rtol=0, atol=1e-14)


def pin_one_hot(lib):
    """One key whose score leads all others by > 60 takes all the weight: O = that V row."""
    N, D = 8, 4
    q = np.zeros((N, D)); q[:, 0] = 10.0
    k = _rand((N, D), 15) * 0.1
    k[5, 0] = 10.0            # score of key 5 is ~ 100 * s higher than the others
    v = _rand((N, D), 16)
    O, L = oracle.forward(q, k, v, False, 1.0, lib=lib)
    assert np.allclose(O, np.tile(v[5], (N, 1)), rtol=0, atol=1e-20 + 1e-15)
    assert np.allclose(L, q @ k[5], rtol=0, atol=1e-12)


def pin_vs_torch_sdpa(lib):
    """Full forward equals PyTorch's fp64 CPU scaled_dot_product_attention (an
    independent implementation), and LSE equals torch.logsumexp of the masked
    scaled scores."""
    for causal in (False, True):
        for (B, H, N, D, s) in ((2, 3, 37, 16, 0.25), (1, 2, 130, 64, 1.0 / 8)):
            q = torch.from_numpy(_rand((B, H, N, D), 17))
            k = torch.from_numpy(_rand((B, H, N, D), 18))
            v = torch.from_numpy(_rand((B, H, N, D), 19))
            ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=s)
            S = s * (q @ k.transpose(-1, -2))
            if causal:
                S = S.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
            lse_ref = torch.logsumexp(S, dim=-1)
            O, L = oracle.forward(q, k, v, causal, s, lib=lib)
            assert np.allclose(O, ref.numpy(), rtol=0, atol=1e-13)
            assert np.allclose(L, lse_ref.numpy(), rtol=0, atol=1e-12)


def pin_tiled_equals_explicit(lib):
    """The tiled online-softmax recurrence equals the explicit softmax on
    brute-force tiny inputs: ragged tails, BM != BN, one key, causal skip.

    "Building a Verifiable FlashAttention Forward from PyTorch to Triton",
    Part 2 (tiled PyTorch validates the recurrence) and Part 4 (lengths 127,
    128, 129); "Triton: FlashAttention-2 Forward Pass", Verification checklist."""
    seed = 20
    for N in (1, 2, 3, 15, 16, 17, 37, 53):
        for D in (1, 4, 64):
            q, k, v = _rand((2, N, D), seed), _rand((2, N, D), seed + 1), _rand((2, N, D), seed + 2)
            seed += 3
            for causal in (False, True):
                O_ref, L_ref = oracle.forward(q, k, v, causal, 0.5, lib=lib)
                for BM, BN in ((16, 16), (16, 32), (32, 16), (7, 5), (64, 64), (1, 3)):
                    O, L = oracle.tiled(q, k, v, causal, 0.5, BM, BN, lib=lib)
                    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
                    assert np.max(np.abs(O - O_ref)) <= 1e-12, (N, D, causal, BM, BN)
                    assert np.max(np.abs(L - L_ref)) <= 1e-12, (N, D, causal, BM, BN)


def pin_unbalanced_magnitudes(lib):
    """Keys scaled up tile by tile so every new tile raises the running max: a
    missing or inverted rescale shows up.  ("A09 - Advanced Triton &
    FlashAttention", pitfalls: unbalanced magnitudes expose a missing rescale.)"""
    N, D, BN = 64, 8, 8
    q = _rand((N, D), 40)
    k = _rand((N, D), 41)
    for t in range(N // BN):
        k[t * BN:(t + 1) * BN] *= 1.0 + 2.0 * t
    v = _rand((N, D), 42)
    for causal in (False, True):
        O_ref, L_ref = oracle.forward(q, k, v, causal, 0.5, lib=lib)
        O, L = oracle.tiled(q, k, v, causal, 0.5, 16, BN, lib=lib)
        assert np.max(np.abs(O - O_ref)) <= 1e-12
        assert np.max(np.abs(L - L_ref)) <= 1e-11
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=causal, scale=0.5)
        assert np.allclose(O_ref, ref.numpy(), rtol=0, atol=1e-12)


def pin_first_step_rescale(lib):
    """m_old = -inf on the first tile gives alpha = exp(-inf) = 0, not NaN
    ("FlashAttention 2 from PyTorch to Triton", Step 1 notes; "Triton:
    FlashAttention-2 Forward Pass", rescale direction): a single key tile of a
    single key reproduces the key's V row exactly."""
    q, k, v = _rand((1, 1, 5), 43), _rand((1, 1, 5), 44), _rand((1, 1, 5), 45)
    for causal in (False, True):
        O, L = oracle.tiled(q, k, v, causal, 0.3125, 1, 1, lib=lib)
        assert np.array_equal(O, v)
        assert abs(L[0, 0] - 0.3125 * float(q[0, 0] @ k[0, 0])) < 1e-15


def _masked_sdpa(q, k, v, causal, s):
    """PyTorch fp64 reference for Nq queries against Nkv keys with an explicit
    bottom-right causal mask; rows that see no key are defined as O = 0,
    LSE = -inf (the empty sum)."""
    Nq, Nkv = q.shape[-2], k.shape[-2]
    S = s * (q @ k.transpose(-1, -2))
    if causal:
        i = torch.arange(Nq).unsqueeze(1)
        j = torch.arange(Nkv).unsqueeze(0)
        S = S.masked_fill(j > i + (Nkv - Nq), float("-inf"))
    lse = torch.logsumexp(S, dim=-1)
    empty = torch.isinf(lse) & (lse < 0)
    P = torch.softmax(S.masked_fill(empty.unsqueeze(-1), 0.0), dim=-1)
    O = (P @ v).masked_fill(empty.unsqueeze(-1), 0.0)
    return O.numpy(), lse.numpy()


def pin_qkv_vs_torch(lib):
    """Nq queries against Nkv keys (cross attention, decode, Nq > Nkv with
    empty rows) equal PyTorch's fp64 softmax under an explicit bottom-right
    mask (an independent route), including O = 0, LSE = -inf for rows that
    see no key."""
    for causal in (False, True):
        for (B, H, Nq, Nkv, D, s) in ((1, 2, 1, 200, 16, 0.25), (2, 1, 37, 130, 8, 0.5), (1, 3, 70, 20, 4, 1.0)):
            q = torch.from_numpy(_rand((B, H, Nq, D), 31))
            k = torch.from_numpy(_rand((B, H, Nkv, D), 32))
            v = torch.from_numpy(_rand((B, H, Nkv, D), 33))
            O, L = oracle.forward_qkv(q, k, v, causal, s, lib=lib)
            O_ref, L_ref = _masked_sdpa(q, k, v, causal, s)
            assert np.array_equal(np.isneginf(L), np.isneginf(L_ref))
            fin = ~np.isneginf(L_ref)
            assert np.allclose(L[fin], L_ref[fin], rtol=0, atol=1e-12)
            assert np.allclose(O, O_ref, rtol=0, atol=1e-13)
            if causal and Nq > Nkv:
                assert np.isneginf(L[..., : Nq - Nkv]).all() and (O[..., : Nq - Nkv, :] == 0.0).all()


def pin_qkv_is_the_suffix_of_square_causal(lib):
    """Decoding the last Nq positions of a sequence of Nkv gives the last Nq
    rows of the square causal attention over the whole sequence (the
    bottom-right alignment), checked against the square oracle, itself pinned
    to PyTorch above."""
    Nkv, D, s = 67, 8, 0.375
    q_all = _rand((2, Nkv, D), 41)
    k, v = _rand((2, Nkv, D), 42), _rand((2, Nkv, D), 43)
    O_sq, L_sq = oracle.forward(q_all, k, v, True, s, lib=lib)
    for Nq in (1, 5, 64, 67):
        O, L = oracle.forward_qkv(np.ascontiguousarray(q_all[:, Nkv - Nq:]), k, v, True, s, lib=lib)
        assert np.allclose(O, O_sq[:, Nkv - Nq:], rtol=0, atol=1e-14)
        assert np.allclose(L, L_sq[:, Nkv - Nq:], rtol=0, atol=1e-13)


def _band_sdpa(q, k, v, left, right, s):
    """PyTorch fp64 reference under an explicit band mask (empty rows O = 0, LSE = -inf)."""
    Nq, Nkv = q.shape[-2], k.shape[-2]
    S = s * (q @ k.transpose(-1, -2))
    ii = torch.arange(Nq).unsqueeze(1) + (Nkv - Nq)
    j = torch.arange(Nkv).unsqueeze(0)
    hide = torch.zeros(Nq, Nkv, dtype=torch.bool)
    if left >= 0:
        hide |= j < ii - left
    if right >= 0:
        hide |= j > ii + right
    S = S.masked_fill(hide, float("-inf"))
    lse = torch.logsumexp(S, dim=-1)
    empty = torch.isinf(lse) & (lse < 0)
    P = torch.softmax(S.masked_fill(empty.unsqueeze(-1), 0.0), dim=-1)
    O = (P @ v).masked_fill(empty.unsqueeze(-1), 0.0)
    return O.numpy(), lse.numpy()


def pin_band_vs_torch(lib):
    """Band (sliding-window) masks -- causal windows, two-sided windows, windows
    wider than the sequence, Nq != Nkv -- equal PyTorch's fp64 softmax under an
    explicit mask (an independent route), including empty rows."""
    for (Nq, Nkv, left, right) in ((37, 37, 5, 0), (40, 70, 9, 3), (70, 40, 0, 0), (33, 33, -1, -1), (33, 33, -1, 0),
                                   (50, 20, 2, 0), (16, 300, 100, -1)):
        q = torch.from_numpy(_rand((2, Nq, 8), 51))
        k = torch.from_numpy(_rand((2, Nkv, 8), 52))
        v = torch.from_numpy(_rand((2, Nkv, 8), 53))
        O, L = oracle.forward_band(q, k, v, left, right, 0.5, lib=lib)
        O_ref, L_ref = _band_sdpa(q, k, v, left, right, 0.5)
        assert np.array_equal(np.isneginf(L), np.isneginf(L_ref)), (Nq, Nkv, left, right)
        fin = ~np.isneginf(L_ref)
        assert np.allclose(L[fin], L_ref[fin], rtol=0, atol=1e-12)
        assert np.allclose(O, O_ref, rtol=0, atol=1e-13)


def pin_band_closed_forms(lib):
    """A band of width one (left = right = 0) gives O = V[i'] and LSE = the one
    score; an unbounded band equals the oracle's full attention; (unbounded, 0)
    equals its causal attention."""
    Nq = Nkv = 29
    q, k, v = _rand((3, Nq, 4), 61), _rand((3, Nkv, 4), 62), _rand((3, Nkv, 4), 63)
    O, L = oracle.forward_band(q, k, v, 0, 0, 0.25, lib=lib)
    assert np.allclose(O, v, rtol=0, atol=1e-15)
    assert np.allclose(L, 0.25 * np.einsum("bid,bid->bi", q, k), rtol=0, atol=1e-13)
    for causal, (left, right) in ((False, (-1, -1)), (True, (-1, 0))):
        O1, L1 = oracle.forward_band(q, k, v, left, right, 0.25, lib=lib)
        O2, L2 = oracle.forward(q, k, v, causal, 0.25, lib=lib)
        assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


# --- backward -----------------------------------------------------------------

BWD_SHAPES = ((5, 5, -1, -1), (5, 5, -1, 0), (4, 7, 2, 1), (6, 3, -1, 0), (7, 7, 1, 1))   # (Nq, Nkv, left, right)


def pin_backward_finite_differences(lib):
    """The gradients of loss = sum(O * dO) by central differences of the
    oracle's own (separately pinned) forward, element by element, on tiny fp64
    inputs: unmasked, causal, a band with Nq != Nkv, rows that see no key, and
    a two-sided band.  Pins every term of the backward without restating it."""
    h = 1e-6
    for n, (Nq, Nkv, left, right) in enumerate(BWD_SHAPES):
        D = 3
        q, k, v = _rand((2, Nq, D), 71 + n), _rand((2, Nkv, D), 81 + n), _rand((2, Nkv, D), 91 + n)
        do = _rand((2, Nq, D), 101 + n)
        dq, dk, dv = oracle.backward_band(q, k, v, do, left, right, 0.5, lib=lib)

        def loss(qq, kk, vv):
            O, _ = oracle.forward_band(qq, kk, vv, left, right, 0.5, lib=lib)
            return float((O * do).sum())

        for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
            num = np.empty_like(x)
            for idx in np.ndindex(*x.shape):
                args = [q.copy(), k.copy(), v.copy()]
                args[which][idx] += h
                up = loss(*args)
                args[which][idx] -= 2 * h
                num[idx] = (up - loss(*args)) / (2 * h)
            assert np.allclose(g, num, rtol=0, atol=1e-7), (Nq, Nkv, left, right, which, float(np.abs(g - num).max()))


def _band_autograd(q, k, v, do, left, right, s):
    """PyTorch fp64 autograd through softmax(s Q K^T) V under an explicit band
    mask (rows that see no key give O = 0)."""
    q, k, v = (torch.from_numpy(x).clone().requires_grad_(True) for x in (q, k, v))
    Nq, Nkv = q.shape[-2], k.shape[-2]
    ii = torch.arange(Nq).unsqueeze(1) + (Nkv - Nq)
    j = torch.arange(Nkv).unsqueeze(0)
    hide = torch.zeros(Nq, Nkv, dtype=torch.bool)
    if left >= 0:
        hide |= j < ii - left
    if right >= 0:
        hide |= j > ii + right
    empty = hide.all(dim=-1, keepdim=True)
    S = (s * (q @ k.transpose(-1, -2))).masked_fill(hide, float("-inf")).masked_fill(empty, 0.0)
    O = (torch.softmax(S, dim=-1) @ v).masked_fill(empty, 0.0)
    O.backward(torch.from_numpy(do))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def pin_backward_vs_torch_autograd(lib):
    """dQ, dK, dV equal PyTorch's fp64 autograd through the explicit softmax
    formula (an independent route), for unmasked, causal, band, Nq != Nkv and
    empty-row cases at moderate sizes."""
    for n, (Nq, Nkv, left, right) in enumerate(((33, 33, -1, -1), (33, 33, -1, 0), (40, 70, 9, 3), (70, 40, 0, 0),
                                                (50, 20, 2, 0), (16, 300, 100, -1))):
        q, k, v = _rand((2, Nq, 8), 111 + n), _rand((2, Nkv, 8), 121 + n), _rand((2, Nkv, 8), 131 + n)
        do = _rand((2, Nq, 8), 141 + n)
        got = oracle.backward_band(q, k, v, do, left, right, 0.5, lib=lib)
        ref = _band_autograd(q, k, v, do, left, right, 0.5)
        for a, b in zip(got, ref):
            assert np.allclose(a, b, rtol=0, atol=1e-12), (Nq, Nkv, left, right, float(np.abs(a - b).max()))


def pin_backward_invariants(lib):
    """Each row of dS = P (dP - delta) sums to zero, so the key rows of dK sum
    to zero; each visible row of P sums to one, so the key rows of dV sum to the
    dO rows of queries that see a key.  (bf16 inputs, causal and band masks.)"""
    from exact_attention_10_gb300.inputs import make_custom
    for (Nq, Nkv, left, right) in ((64, 64, -1, 0), (40, 70, 7, 3), (70, 40, -1, 0)):
        q = make_custom(1, 2, Nq, 16, "bf16", seed=Nq)[0]
        _, k, v = make_custom(1, 2, Nkv, 16, "bf16", seed=Nkv + 1)
        do = make_custom(1, 2, Nq, 16, "bf16", seed=Nq + 2)[0]
        dq, dk, dv = oracle.backward_band(q, k, v, do, left, right, 0.25, lib=lib)
        _, L = oracle.forward_band(q, k, v, left, right, 0.25, lib=lib)
        seen = ~np.isneginf(L)
        dod = oracle.decode(do.view(torch.int16).numpy().view(np.uint16), "bf16", lib=lib).reshape(do.shape)
        assert np.allclose(dk.sum(axis=-2), 0.0, rtol=0, atol=1e-12)
        assert np.allclose(dv.sum(axis=-2), (dod * seen[..., None]).sum(axis=-2), rtol=0, atol=1e-12)
        assert (dq[~seen] == 0).all()


def pin_backward_constant_v(lib):
    """With every V row equal, O does not depend on Q or K: dQ = dK = 0, and
    dV = P^T dO with P from the oracle's (separately pinned) probabilities."""
    N, D = 24, 5
    q, k = _rand((1, N, D), 151), _rand((1, N, D), 152)
    v = np.repeat(_rand((1, 1, D), 153), N, axis=1)
    do = _rand((1, N, D), 154)
    for causal in (False, True):
        dq, dk, dv = oracle.backward(q, k, v, do, causal, 0.5, lib=lib)
        assert np.allclose(dq, 0.0, rtol=0, atol=1e-13) and np.allclose(dk, 0.0, rtol=0, atol=1e-13)
        P = oracle.probs(q[0], k[0], causal, 0.5, lib=lib)
        assert np.allclose(dv[0], P.T @ do[0], rtol=0, atol=1e-13)


def pin_backward_delta_is_rowsum_do_o(lib):
    """The softmax Jacobian's delta_i = sum_j P_ij dP_ij equals the pages'
    D = rowsum(dO o O) with O from the oracle's forward."""
    for (Nq, Nkv, left, right) in ((33, 33, -1, 0), (40, 70, 9, 3), (70, 40, 0, 0)):
        q, k, v = _rand((2, Nq, 8), 161), _rand((2, Nkv, 8), 162), _rand((2, Nkv, 8), 163)
        do = _rand((2, Nq, 8), 164)
        *_, delta = oracle.backward_band(q, k, v, do, left, right, 0.5, with_delta=True, lib=lib)
        O, _ = oracle.forward_band(q, k, v, left, right, 0.5, lib=lib)
        assert np.allclose(delta, (do * O).sum(axis=-1), rtol=0, atol=1e-12)


PINS = [pin_decode, pin_rows_sum_to_one, pin_probs_vs_scipy, pin_constant_v, pin_identical_keys,
        pin_zero_query, pin_causal_row0, pin_one_hot, pin_vs_torch_sdpa, pin_tiled_equals_explicit,
        pin_unbalanced_magnitudes, pin_first_step_rescale, pin_qkv_vs_torch, pin_qkv_is_the_suffix_of_square_causal,
        pin_band_vs_torch, pin_band_closed_forms, pin_backward_finite_differences, pin_backward_vs_torch_autograd,
        pin_backward_invariants, pin_backward_constant_v, pin_backward_delta_is_rowsum_do_o]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


# ---------------------------------------------------------------------------
# Consistency of the entry points with each other on low-precision inputs
# ---------------------------------------------------------------------------

def test_bf16_inputs_are_decoded_exactly(oracle_lib):
    """Forward on bf16 tensors equals forward on the same values widened to fp64 (bit for bit)."""
    from exact_attention_10_gb300.inputs import make_custom
    q, k, v = make_custom(1, 2, 40, 16, "bf16", seed=3)
    O1, L1 = oracle.forward(q, k, v, True, 0.25, lib=oracle_lib)
    O2, L2 = oracle.forward(q.double(), k.double(), v.double(), True, 0.25, lib=oracle_lib)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_rows_equal_forward(oracle_lib):
    """A sampled row is exactly the row of the full forward (rows are independent)."""
    from exact_attention_10_gb300.inputs import make_custom
    q, k, v = make_custom(2, 2, 77, 32, "fp16", seed=4, qk_gain=4.0)
    for causal in (False, True):
        O, L = oracle.forward(q, k, v, causal, 0.1875, lib=oracle_lib)
        bh = np.array([0, 0, 1, 2, 3, 3])
        ri = np.array([0, 76, 5, 40, 1, 76])
        Or, Lr = oracle.rows(q, k, v, causal, 0.1875, bh, ri, lib=oracle_lib)
        Of, Lf = O.reshape(4, 77, 32), L.reshape(4, 77)
        assert np.array_equal(Or, Of[bh, ri]) and np.array_equal(Lr, Lf[bh, ri])


def test_rows_rejects_bad_indices(oracle_lib):
    q = torch.zeros(1, 2, 4, 2, dtype=torch.float64)
    with pytest.raises(ValueError):
        oracle.rows(q, q, q, False, 1.0, [0], [4], lib=oracle_lib)      # row out of range
    with pytest.raises(ValueError):
        oracle.rows(q, q, q, False, 1.0, [1, 0], [0, 1], lib=oracle_lib)  # heads not non-decreasing


# ---------------------------------------------------------------------------
# A figure the pages print
# ---------------------------------------------------------------------------

def _golden(name):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split("=", 1)
                vals[key.strip()] = val.strip()
    return vals


@pytest.mark.slow
def test_bf16_output_rounding_floor_matches_page(oracle_lib):
    """At B*H = 32, N = 4096, D = 64, bf16 N(0,1) inputs, non-causal, scale 1/8,
    rounding the exact output to bf16 costs a mean absolute error of 2.9e-5
    ("How to profile and optimise kernels", the P cast section).  The oracle's
    exact output, rounded to bf16, must show that figure: a dropped scale or a
    wrong normalisation changes the output magnitudes and moves it."""
    g = _golden("bf16_rounding_floor.txt")
    from exact_attention_10_gb300.inputs import WORKLOADS, make_qkv
    w = WORKLOADS["b2h16_n4096"]
    q, k, v = make_qkv(w, seed=0)
    heads = int(g["heads_sampled"])
    qs, ks, vs = (x.reshape(32, w.N, w.D)[:heads] for x in (q, k, v))
    O, _ = oracle.forward(qs, ks, vs, False, w.scale, lib=oracle_lib)
    Ob = torch.from_numpy(O).to(torch.bfloat16).to(torch.float64).numpy()
    mean_err = float(np.mean(np.abs(Ob - O)))
    lo, hi = float(g["accept_low"]), float(g["accept_high"])
    assert lo <= mean_err <= hi, mean_err
