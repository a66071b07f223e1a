"""The bench's FLOP and byte accounting against counts the pages print."""
from __future__ import annotations

import os

import pytest

from exact_attention_10_gb300 import accounting as acc


def _golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "flop_and_byte_counts.txt")
    vals = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split("=", 1)
            vals[k.strip()] = float(v)
    return vals


def test_flops_match_page_counts():
    g = _golden()
    assert acc.flops(4, 8, 4096, 64, False) == pytest.approx(g["flops_noncausal_b4h8_n4096_d64"], rel=1e-3)
    assert acc.flops(4, 8, 4096, 64, True) == pytest.approx(g["flops_causal_b4h8_n4096_d64"], rel=1e-3)
    # the exact causal count includes the diagonal: a little above half
    assert acc.flops(4, 8, 4096, 64, True) < acc.flops_causal_exact(4, 8, 4096, 64) < \
        acc.flops(4, 8, 4096, 64, True) * 1.001


def test_fused_bytes_match_page_table():
    g = _golden()
    for n in (1024, 4096, 16384):
        assert acc.fused_bytes(1, 1, n, 128, with_lse=False) == g[f"fused_bytes_per_head_d128_n{n}"]
        assert round(acc.unfused_bytes_per_head(n, 128) / acc.fused_bytes(1, 1, n, 128, with_lse=False)) == \
            g[f"unfused_ratio_d128_n{n}"]
        assert acc.unfused_ratio(n, 128) == g[f"unfused_ratio_d128_n{n}"]


def test_l2_operand_bytes_causal_is_about_half():
    nc = acc.l2_operand_bytes(2, 16, 4096, 64, False)
    c = acc.l2_operand_bytes(2, 16, 4096, 64, True)
    assert nc == 2 * 16 * 16 * 32 * 2 * 128 * 64 * 2
    assert 0.5 < c / nc < 0.56
