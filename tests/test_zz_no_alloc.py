"""fa_fwd_noalloc -- the entry point that allocates no memory -- called
through the C ABI on the GPU.  (Named to be collected last, so that it runs
both after every other test, against whatever state they leave, and alone.)

It must give exactly what fa_fwd_ex gives (same kernels, same schedule: the
only difference is where the balanced schedule's partial results live), on
consecutive calls; it must not allocate device memory; and it must reject a
call that needs more than its static workspace before anything is enqueued.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from exact_attention_10_gb300 import fa
from exact_attention_10_gb300.inputs import make_custom

pytestmark = pytest.mark.gpu

AUTO, WHOLE, BALANCED = 0, 1, 2
FA_ERR_NO_ALLOC_LIMIT = 6


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return fa.load()


def _call(fn, q, k, v, o, lse, causal, schedule, scale):
    B, H, N, D = q.shape
    dtype = 0 if q.dtype == torch.bfloat16 else 1
    st = torch.cuda.current_stream().cuda_stream
    return fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, D, int(causal),
              ctypes.c_float(scale), dtype, schedule, ctypes.c_void_p(st))


@pytest.mark.parametrize("B,H,N,D,dtype", [(2, 16, 4096, 64, "bf16"), (2, 8, 3000, 128, "fp16"), (1, 3, 513, 64, "bf16")])
@pytest.mark.parametrize("schedule", [AUTO, BALANCED])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_fa_fwd_ex_on_two_calls_in_a_row(lib, B, H, N, D, dtype, schedule, causal):
    q, k, v = (x.cuda() for x in make_custom(B, H, N, D, dtype, seed=N + D))
    scale = D ** -0.5
    o_ref, l_ref = torch.empty_like(q), torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    assert _call(lib.fa_fwd_ex, q, k, v, o_ref, l_ref, causal, schedule, scale) == 0
    outs = []
    for _ in range(2):   # two calls in a row, the second reusing the workspace the first left
        o, lse = torch.full_like(q, 7.0), torch.full(q.shape[:-1], 7.0, dtype=torch.float32, device="cuda")
        assert _call(lib.fa_fwd_noalloc, q, k, v, o, lse, causal, schedule, scale) == 0
        outs.append((o, lse))
    assert lib.fa_sync_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    for o, lse in outs:
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_allocates_no_device_memory(lib):
    q, k, v = (x.cuda() for x in make_custom(2, 16, 4096, 64, "bf16", seed=3))
    o, lse = torch.empty_like(q), torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    assert _call(lib.fa_fwd_noalloc, q, k, v, o, lse, False, BALANCED, 0.125) == 0   # set-up call
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch0 = torch.cuda.memory_allocated()
    for causal in (False, True, False):
        assert _call(lib.fa_fwd_noalloc, q, k, v, o, lse, causal, BALANCED, 0.125) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == torch0


def test_rejects_a_call_beyond_its_workspace(lib):
    """Four million one-row heads: each head is one CTA tile with its own merge
    counters (8 bytes), 32 MB of counters on top of 20.5 MB of partial-result
    slots (D = 64, 152 CTAs), more than FA_NOALLOC_WORKSPACE_BYTES (48 MiB),
    while each tensor stays at 512 MB."""
    B, H, N, D = 2000, 2000, 1, 64
    q = torch.randn(B, H, N, D, device="cuda").to(torch.bfloat16)   # Q, K and V may alias
    o = torch.full_like(q, 7.0)
    lse = torch.full((B, H, N), 7.0, dtype=torch.float32, device="cuda")
    rc = _call(lib.fa_fwd_noalloc, q, q, q, o, lse, False, BALANCED, 0.125)
    assert rc == FA_ERR_NO_ALLOC_LIMIT, fa.status_string(rc)
    assert "static workspace" in fa.status_string(rc)
    torch.cuda.synchronize()
    assert bool((o.float() == 7.0).all()) and bool((lse == 7.0).all())   # nothing was enqueued
    # the same call with whole tiles needs no workspace
    assert _call(lib.fa_fwd_noalloc, q, q, q, o, lse, False, WHOLE, 0.125) == 0
    assert lib.fa_sync_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    ref = torch.empty_like(o)
    ref_lse = torch.empty_like(lse)
    assert _call(lib.fa_fwd_ex, q, q, q, ref, ref_lse, False, WHOLE, 0.125) == 0
    torch.cuda.synchronize()
    assert torch.equal(o, ref) and torch.equal(lse, ref_lse)
    # the automatic schedule never fails on the limit: where its plan would
    # not fit it runs whole tiles (its planner is checked on the CPU in
    # tests/test_schedule.py with smaller limits)
    o.fill_(7.0)
    assert _call(lib.fa_fwd_noalloc, q, q, q, o, lse, False, AUTO, 0.125) == 0
    assert lib.fa_sync_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    assert torch.equal(o, ref) and torch.equal(lse, ref_lse)
