"""Plant plausible slips in the oracle (on the CPU) and check a pin catches each.

Each mutant is the oracle's C source with one textual change, compiled into a
temporary library.  The pins of ``test_oracle_pins.py`` are rerun against it;
at least one must fail.  This shows the pins constrain every part of the
oracle: the scale, the causal index, the operands, the normalisation, the
LSE's log base and shift, the rescale direction of the recurrence, its causal
loop bound, the bf16/fp16 decoders, and the backward's terms (delta, scales,
operands, normalisation, band).  No mutant indexes outside its arrays.
"""
from __future__ import annotations

import os

import pytest

import oracle
from oracle.build import SRC, build
from test_oracle_pins import PINS

MUTANTS = {
    "drop_scale": ("        x[j] = s * dot;", "        x[j] = dot;"),
    "ignore_causal": ("ref_row_vis(q, Kh, Vh, causal ? i + 1 : N,", "ref_row_vis(q, Kh, Vh, causal ? N : N,"),
    "causal_off_by_one": ("ref_row_vis(q, Kh, Vh, causal ? i + 1 : N,", "ref_row_vis(q, Kh, Vh, causal ? i + (i == 0) : N,"),
    "wrong_key_index": ("dot += q[d] * Kh[j * D + d];", "dot += q[d] * Kh[(nvis - 1 - j) * D + d];"),
    "qkv_top_left_causal": ("long last = i + Nkv - Nq;", "long last = i;"),
    "band_left_off_by_one": ("long lo = left < 0 ? 0 : ii - left,", "long lo = left < 0 ? 0 : ii - left + 1,"),
    "band_ignores_right": ("hi = right < 0 ? Nkv - 1 : ii + right;", "hi = Nkv - 1;"),
    "qkv_empty_row_lse": ("        *lse = -INFINITY;\n        return;", "        *lse = 0.0;\n        return;"),
    "k_instead_of_v": ("o[d] += w * Vh[j * D + d];", "o[d] += w * Kh[j * D + d];"),
    "no_normalisation": ("        o[d] /= l;", "        o[d] /= 1.0;"),
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "lse_no_shift": ("*lse = m + log(l);", "*lse = log(l);"),
    "exp_sign": ("double w = exp(x[j] - m);", "double w = exp(m - x[j]);"),
    "probs_unnormalised": ("            P[i * N + j] /= l;", "            P[i * N + j] /= 1.0;"),
    "tiled_inverse_rescale": ("double alpha = exp(m[r] - shift);", "double alpha = exp(shift - m[r]);"),
    "tiled_no_acc_rescale": ("acc[r * D + d] = alpha * acc[r * D + d] + pv;", "acc[r * D + d] = acc[r * D + d] + pv;"),
    "tiled_skips_diagonal": ("hi = (q0 + BM < N) ? q0 + BM : N;", "hi = q0;"),
    "tiled_no_key_mask": ("if (kj >= N || (causal && kj > qi)) {", "if (kj >= N) {"),
    "bwd_dq_drops_delta": ("const double ds = p * (dot_d(dOh + i * D, Vh + j * D, D) - delta);",
                           "const double ds = p * (dot_d(dOh + i * D, Vh + j * D, D) - 0.0);"),
    "bwd_dk_drops_delta": ("const double ds = p * (dot_d(dOh + i * D, Vh + j * D, D) - Dr[i]);",
                           "const double ds = p * (dot_d(dOh + i * D, Vh + j * D, D) - 0.0);"),
    "bwd_dk_no_scale": ("dk[d] += s * ds * Qh[i * D + d];", "dk[d] += ds * Qh[i * D + d];"),
    "bwd_dv_uses_ds": ("dv[d] += p * dOh[i * D + d];", "dv[d] += ds * dOh[i * D + d];"),
    "bwd_dq_uses_v": ("dq[d] += s * ds * Kh[j * D + d];", "dq[d] += s * ds * Vh[j * D + d];"),
    "bwd_p_unnormalised": ("            const double p = exp(x[j] - L);", "            const double p = exp(x[j] - m);"),
    "bwd_delta_uses_k": ("delta += exp(x[j] - L) * dot_d(dOh + i * D, Vh + j * D, D);",
                         "delta += exp(x[j] - L) * dot_d(dOh + i * D, Kh + j * D, D);"),
    "bwd_keys_ignore_band": ("                if (j < lo || j > hi)\n                    continue;",
                             "                if (j < 0)\n                    continue;"),
    "bf16_shift": ("uint32_t u = ((uint32_t)h) << 16;", "uint32_t u = ((uint32_t)h) << 15;"),
    "fp16_bias": ("v = ldexp((double)(f + 1024), e - 25);", "v = ldexp((double)(f + 1024), e - 24);"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"mutation site for {name} not found in the oracle source"
    src = tmp_path / f"mut_{name}.c"
    src.write_text(source.replace(old, new, 1))
    so = build(str(src), str(tmp_path / f"mut_{name}.so"))
    lib = oracle._load(so)
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except Exception as e:  # an assertion, or a NaN that breaks a closed form
            caught.append(f"{pin.__name__}: {type(e).__name__}")
    assert caught, f"mutant {name} passed every pin"


def test_unmutated_source_passes_all_pins(source, tmp_path):
    """Control: the same build route with no change passes every pin."""
    src = tmp_path / "same.c"
    src.write_text(source)
    lib = oracle._load(build(str(src), str(tmp_path / "same.so")))
    for pin in PINS:
        pin(lib)
