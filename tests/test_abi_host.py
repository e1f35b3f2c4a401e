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


def test_router_argument_checks_without_gpu(lib):
    f = lib.bws_moe_router_topk
    ws = 1 << 20

    # (W, x, N, n_experts, d, topk, logits, ids, route_w, workspace, workspace_bytes, stream)
    def call(W=16, x=16, N=1, E=8, d=64, k=2, logits=None, ids=16, w=16, buf=256, nbytes=ws):
        return f(W, x, N, E, d, k, logits, ids, w, buf, nbytes, None)

    assert call(W=None) == 1 and b"null" in lib.bws_last_error()
    assert call(N=0) == 1 and call(N=9) == 1
    assert call(k=0) == 1 and call(k=9) == 1
    assert call(E=4, k=5) == 1                      # more experts chosen than exist
    assert call(E=0) == 2 and call(E=2049) == 2
    assert call(d=60) == 2 and call(d=7176) == 2
    assert call(W=24) == 3 and call(x=40) == 3      # 16-byte alignment
    assert call(ids=None) == 1 and call(w=None) == 1
    assert call(ids=18) == 3 and call(logits=18) == 3
    assert call(nbytes=16) == 7 and call(buf=None) == 7
    assert call(buf=260) == 3                       # 256-byte aligned workspace
    assert lib.bws_moe_router_workspace_size(1, 512) == 256 + 2048
    assert lib.bws_moe_router_workspace_size(8, 512) == 256 + 16384
    assert lib.bws_moe_router_workspace_size(0, 512) == 0
    assert lib.bws_moe_router_workspace_size(1, 4096) == 0


def test_w4a8_argument_checks_without_gpu(lib):
    f = lib.bws_mxfp4_w4a8_gemv
    ws = 1 << 24

    # (codes, scales, x, N, d_out, d_in, y, workspace, workspace_bytes, stream)
    def call(c=32, s=32, x=32, N=1, d_out=64, d_in=256, y=32, buf=256, nbytes=ws):
        return f(c, s, x, N, d_out, d_in, y, buf, nbytes, None)

    assert call(N=0) == 0 and call(d_out=0) == 0           # no-ops
    assert call(c=None) == 1 and b"null" in lib.bws_last_error()
    assert call(N=9) == 1
    assert call(d_in=128) == 2 and call(d_in=320) == 2
    assert call(c=48) == 3 and call(s=36) == 3 and call(x=33) == 3
    assert call(nbytes=256) == 7 and call(buf=None) == 7
    assert call(buf=272) == 3
    assert lib.bws_w4a8_workspace_size(9, 64, 256) == 0
    assert lib.bws_w4a8_workspace_size(1, 64, 320) == 0
    assert 0 < lib.bws_w4a8_workspace_size(1, 64, 256) < lib.bws_w4a8_workspace_size(8, 17408, 5120)
    q = lib.bws_mxfp8_quantize
    assert q(None, 0, 32, None, None, None) == 0
    assert q(None, 1, 32, 16, 16, None) == 1
    assert q(16, 1, 48, 16, 16, None) == 2 and q(17, 1, 32, 16, 16, None) == 3
