"""The no-allocation NVFP4 GEMV entry point, called through the C ABI.

bws_nvfp4_gemv_noalloc serves callers that cannot allocate device memory; it
uses the library's static device scratch instead of a caller workspace. Two
calls in a row (different activations, so stale scratch contents would show)
must each match the workspace entry point within the product tolerance, and
sizes beyond the static scratch must be refused with a message. This file is
collected last so that a run stopping at the first failure has already run
every other test."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import quant as Q, products as P, tolerance as T
from tests.gpu_util import device, bws, f64
import synth

pytestmark = pytest.mark.gpu


def _call(lib, c, s, t, x, y):
    return lib.bws_nvfp4_gemv_noalloc(c.data_ptr(), s.data_ptr(), t.data_ptr(), x.data_ptr(), x.shape[0],
                                      c.shape[0], x.shape[1], y.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_twice():
    m = bws()
    lib = m.lib()
    dev = device()
    d_out, d_in, N = 3000, 2560, 3
    W = synth.weight_fp32((d_out, d_in), seed=41).numpy()
    cq, sq, tq = Q.nvfp4_quantize(W)
    c, s = torch.from_numpy(cq).to(dev), torch.from_numpy(sq).to(dev)
    t = torch.tensor([float(tq)], dtype=torch.float32, device=dev)
    for call in range(2):
        x = synth.activation_bf16(N, d_in, seed=100 + call, device=dev)
        y_ws = m.nvfp4_gemv(c, s, t, x)
        y = torch.full((N, d_out), float("nan"), dtype=torch.bfloat16, device=dev)
        rc = _call(lib, c, s, t, x, y)
        assert rc == 0, lib.bws_last_error()
        torch.cuda.synchronize()
        y_ref, A = P.nvfp4_gemv(cq, sq, tq, f64(x))
        ok, worst, at = T.check(f64(y_ws), f64(y), A)      # against the workspace entry point
        assert ok, (call, worst, at)
        ok, worst, at = T.check(y_ref, f64(y), A)          # and against the oracle
        assert ok, (call, worst, at)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """A size whose activations alone (N * d_in * 8 bytes) exceed the scratch.
    Every buffer is allocated at its full declared size, so that a refusal
    that stopped working would show as a wrong status, not as accesses past
    the end of a buffer."""
    m = bws()
    lib = m.lib()
    dev = device()
    d_out, d_in, N = 32, 262144, 8
    c = torch.zeros((d_out, d_in // 2), dtype=torch.uint8, device=dev)
    s = torch.zeros((d_out, d_in // 16), dtype=torch.uint8, device=dev)
    t = torch.ones(1, dtype=torch.float32, device=dev)
    x = torch.zeros((N, d_in), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((N, d_out), dtype=torch.bfloat16, device=dev)
    rc = lib.bws_nvfp4_gemv_noalloc(c.data_ptr(), s.data_ptr(), t.data_ptr(), x.data_ptr(), N, d_out, d_in,
                                    y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 7
    assert b"static scratch" in lib.bws_last_error()
