"""The C-ABI library loads, exports every entry point include/bws.h declares,
and rejects bad arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"\b(bws_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    import bit_weight_streaming_gb300 as bws
    return bws.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 12
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_error_string(lib):
    assert lib.bws_version() >= 100
    assert isinstance(lib.bws_last_error(), bytes)


def test_argument_checks_without_gpu(lib):
    from bit_weight_streaming_gb300._lib import SIGNATURES
    f = lib.bws_nvfp4_gemv
    # null codes
    rc = f(None, None, None, None, 1, 64, 64, None, None, 0, None)
    assert rc == 1 and b"null" in lib.bws_last_error()
    # N out of range
    rc = f(16, 16, 16, 16, 9, 64, 64, 16, 256, 1 << 20, None)
    assert rc == 1
    # d_in not a multiple of 32
    rc = f(16, 16, 16, 16, 1, 64, 48, 16, 256, 1 << 20, None)
    assert rc == 2
    # misaligned codes
    rc = f(17, 16, 16, 16, 1, 64, 64, 16, 256, 1 << 20, None)
    assert rc == 3
    # empty: nothing to do
    assert f(None, None, None, None, 0, 64, 64, None, None, 0, None) == 0
    assert f(None, None, None, None, 1, 0, 64, None, None, 0, None) == 0
    # workspace too small
    rc = f(16, 16, 16, 16, 1, 64, 64, 16, 256, 16, None)
    assert rc == 7
    # quantizer shape checks
    assert lib.bws_nvfp4_quantize(16, 4, 24, 16, 16, 16, 16, 256, None) == 2
    assert lib.bws_mxfp4_quantize(16, 4, 48, 16, 16, None) == 2


def test_workspace_size_monotone(lib):
    a = lib.bws_gemv_workspace_size(1, 17408, 5120)
    b = lib.bws_gemv_workspace_size(8, 17408, 5120)
    assert 0 < a < b
    assert lib.bws_gemv_workspace_size(0, 10, 10) == 0
