"""CPU-only checks of the C-ABI library: it loads, exports every function the
header declares, and rejects bad arguments before touching any device.

No test here launches work: without a GPU the library can only be loaded and
its host-side validation exercised.
"""
from __future__ import annotations

import os
import re

import pytest

from exact_attention_10_gb300 import build as fa_build
from exact_attention_10_gb300 import fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

OK, INVALID, MISALIGNED, UNSUPPORTED = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa_build.LIB_PATH):
        fa_build.build()
    return fa.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    assert _declared_functions() == sorted(fa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(lib):
    """Built with hidden visibility: the dynamic symbol table holds the ABI
    functions only, so no internal symbol (a launcher's once-per-device flags,
    say) can be unified with another copy of the library in the process."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", fa_build.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    names = sorted(line.split()[-1] for line in out.splitlines() if line.strip())
    assert names == _declared_functions(), names


def test_status_strings(lib):
    for code in range(7):
        s = fa.status_string(code)
        assert s and s != "unknown status"
    assert fa.status_string(99) == "unknown status"


# Fake, never-dereferenced addresses: validation must reject the call first.
A = 0x10000000
GOOD = dict(q=A, k=A + 0x1000000, v=A + 0x2000000, o=A + 0x3000000, lse=A + 0x4000000,
            B=1, H=2, N=256, D=64, causal=0, scale=0.125, dtype=0)


def _call(**over):
    a = dict(GOOD, **over)
    return fa.fwd_raw(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"], a["causal"],
                      a["scale"], a["dtype"], 0)


@pytest.mark.parametrize("over", [
    dict(D=32), dict(D=96), dict(D=256), dict(B=0), dict(H=-1), dict(N=0), dict(causal=2), dict(dtype=2),
    dict(scale=0.0), dict(scale=-0.125), dict(scale=float("inf")), dict(scale=float("nan")),
    dict(q=0), dict(k=0), dict(v=0), dict(o=0), dict(lse=0),
    dict(B=1 << 16, H=1 << 10, N=4),                                   # B*H*N >= 2^31
    dict(o=A),                                                          # O aliases Q
    dict(o=A + 0x1000000 + 64),                                         # O overlaps K
    dict(lse=A + 0x3000000 + 128),                                      # LSE overlaps O
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_invalid_arguments_rejected(lib, over):
    assert _call(**over) == INVALID


@pytest.mark.parametrize("field", ["q", "k", "v", "o", "lse"])
def test_misaligned_pointer_rejected(lib, field):
    assert _call(**{field: GOOD[field] + 8}) == MISALIGNED


def test_valid_arguments_without_device(lib):
    """Sound arguments on a machine with no GPU: unsupported device, nothing launched."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert _call() == UNSUPPORTED
    assert _call(causal=1, D=128, dtype=1) == UNSUPPORTED


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(OSError):
        fa.load(str(tmp_path / "nope.so"))


def test_no_oracle_on_the_product_path():
    """The product package and the CUDA sources never reference the oracle."""
    pkg = os.path.join(ROOT, "exact_attention_10_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "attn_ref" not in text, f


def test_qkv_invalid_arguments_rejected(lib):
    """fa_fwd_qkv validates Nq and Nkv before touching any device."""
    import ctypes
    a = GOOD
    for nq, nkv in ((0, 16), (16, 0), (-1, 16), (1, 1 << 31 - 1)):
        rc = lib.fa_fwd_qkv(a["q"], a["k"], a["v"], a["o"], a["lse"], 1, 2, nq, nkv, 64, 0, ctypes.c_float(0.125), 0,
                            0, None)
        assert rc == INVALID, (nq, nkv, rc)



def test_band_arguments(lib):
    """fa_fwd_band validates its sizes like fa_fwd_qkv; any window bound is
    valid (a negative one is unbounded), so sound sizes reach the device check."""
    import ctypes
    a = GOOD
    for nq, nkv in ((0, 16), (16, 0), (-1, 16)):
        rc = lib.fa_fwd_band(a["q"], a["k"], a["v"], a["o"], a["lse"], 1, 2, nq, nkv, 64, 3, 0,
                             ctypes.c_float(0.125), 0, 0, None)
        assert rc == INVALID, (nq, nkv, rc)
    rc = lib.fa_fwd_band(a["q"], a["k"], a["v"], a["o"], a["lse"], 1, 2, 16, 16, 64, 3, 0, ctypes.c_float(0.0), 0, 0,
                         None)
    assert rc == INVALID
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        for window in ((-1, -1), (-1, 0), (0, 0), (5, -7), (1 << 30, 1 << 30)):
            rc = lib.fa_fwd_band(a["q"], a["k"], a["v"], a["o"], a["lse"], 1, 2, 16, 300, 64, window[0], window[1],
                                 ctypes.c_float(0.125), 0, 0, None)
            assert rc == UNSUPPORTED, (window, rc)


def test_bwd_invalid_arguments_rejected(lib):
    """fa_bwd validates everything before touching a device: sizes, flags,
    scale, NULL and misaligned pointers, and outputs overlapping an input or
    each other."""
    import ctypes
    base = dict(q=A, k=A + 0x1000000, v=A + 0x2000000, o=A + 0x3000000, do=A + 0x4000000, lse=A + 0x5000000,
                dq=A + 0x6000000, dk=A + 0x7000000, dv=A + 0x8000000, B=1, H=2, N=256, D=64, causal=0, scale=0.125,
                dtype=0)

    def call(**over):
        a = dict(base, **over)
        return lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"], a["B"],
                          a["H"], a["N"], a["D"], a["causal"], ctypes.c_float(a["scale"]), a["dtype"], None)

    for over in (dict(D=96), dict(B=0), dict(N=0), dict(causal=2), dict(dtype=3), dict(scale=0.0),
                 dict(scale=float("nan")), dict(q=0), dict(do=0), dict(lse=0), dict(dv=0),
                 dict(B=1 << 16, H=1 << 8, N=129),                   # B*H*Npad >= 2^31
                 dict(dq=A + 0x1000000),                              # dQ aliases K
                 dict(dk=A + 0x6000000 + 64),                         # dK overlaps dQ
                 dict(dv=A + 0x5000000)):                             # dV overlaps LSE
        assert call(**over) == INVALID, over
    for f in ("q", "do", "lse", "dk"):
        assert call(**{f: base[f] + 8}) == MISALIGNED, f
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert call() == UNSUPPORTED
        assert call(causal=1, D=128, dtype=1) == UNSUPPORTED


def test_bwd_band_arguments(lib):
    """fa_bwd_band validates its sizes like fa_bwd; any window bound is valid."""
    import ctypes
    a = [A + i * 0x1000000 for i in range(9)]
    for nq, nkv in ((0, 16), (16, 0), (-1, 16)):
        rc = lib.fa_bwd_band(*a, 1, 2, nq, nkv, 64, 3, 0, ctypes.c_float(0.125), 0, None)
        assert rc == INVALID, (nq, nkv, rc)
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        for window in ((-1, -1), (-1, 0), (0, 0), (5, -7)):
            rc = lib.fa_bwd_band(*a, 1, 2, 16, 300, 64, window[0], window[1], ctypes.c_float(0.125), 0, None)
            assert rc == UNSUPPORTED, (window, rc)
