"""The device status paths, through the C ABI: a bounded wait that runs out
returns an error status instead of hanging, and an activation too small for
the two f16 bands is reported.

* bws_debug_wait_flag runs the library's bounded flag wait on a flag that
  nothing sets: the kernel must give up after its poll limit, set
  BWS_STATUS_WAIT_TIMEOUT and return; bws_status_word then returns
  BWS_ERR_TIMEOUT, and the context stays usable for the next product.
* x = [1, 2^-60, 0, ...]: 2^-60 lies below both f16 bands of its token
  (2^-57 of the largest magnitude), so the product treats it as zero and sets
  BWS_STATUS_X_FLUSHED; the result stays within the product bound plus the
  flushed elements' largest contribution 2^-57 * max|x| * sum_j |w_ij| (the
  reading the library documents for this status bit)."""
import ctypes
import time

import numpy as np
import pytest
import torch

from oracle import quant as Q, products as P, tolerance as T
from tests.gpu_util import device, bws, f64
import synth

pytestmark = pytest.mark.gpu

BWS_ERR_TIMEOUT = 6
WAIT_TIMEOUT = 0x100


def _wait(lib, flag, polls, ws):
    return lib.bws_debug_wait_flag(flag.data_ptr(), polls, ws.data_ptr(), ws.numel(),
                                   torch.cuda.current_stream().cuda_stream)


def test_bounded_wait_runs_out_and_reports_timeout():
    m = bws()
    lib = m.lib()
    dev = device()
    ws = torch.zeros(int(lib.bws_gemv_workspace_size(1, 1, 32)), dtype=torch.uint8, device=dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)       # nothing ever sets it
    torch.cuda.synchronize()
    t0 = time.time()
    assert _wait(lib, flag, 4000, ws) == 0, lib.bws_last_error()
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    st = ctypes.c_uint32(0)
    rc = lib.bws_status_word(ws.data_ptr(), ctypes.addressof(st), torch.cuda.current_stream().cuda_stream)
    assert rc == BWS_ERR_TIMEOUT, (rc, lib.bws_last_error())
    assert st.value & WAIT_TIMEOUT
    # a flag that is set: the same wait returns at once and reports nothing
    flag.fill_(1)
    assert _wait(lib, flag, 4000, ws) == 0
    rc = lib.bws_status_word(ws.data_ptr(), ctypes.addressof(st), torch.cuda.current_stream().cuda_stream)
    assert rc == 0 and not (st.value & WAIT_TIMEOUT)
    # the context is still usable
    W = synth.weight_fp32((64, 256), seed=9).numpy()
    c, s, t = Q.nvfp4_quantize(W)
    x = synth.activation_bf16(1, 256, seed=9, device=dev)
    y = m.nvfp4_gemv(torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev),
                     torch.tensor([float(t)], device=dev), x)
    torch.cuda.synchronize()
    y_ref, A = P.nvfp4_gemv(c, s, t, f64(x))
    assert T.check(y_ref, f64(y), A)[0]


@pytest.mark.parametrize("d_in", [256, 4096])
def test_activation_below_both_bands_is_flagged(d_in):
    m = bws()
    dev = device()
    W = synth.weight_fp32((48, d_in), seed=10).numpy()
    W[:, 0] = 0.0                     # no weight on the large element: the tiny one is all there is
    c, s, t = Q.nvfp4_quantize(W)
    x = torch.zeros((1, d_in), dtype=torch.float32)
    x[0, 0] = 1.0
    x[0, 1] = 2.0 ** -60
    x = x.to(torch.bfloat16).to(dev)
    ws = m.Workspace(dev)
    y = m.nvfp4_gemv(torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev),
                     torch.tensor([float(t)], device=dev), x, ws=ws)
    torch.cuda.synchronize()
    assert m.status_word(ws) & m.BWS_STATUS_X_FLUSHED
    y_ref, A = P.nvfp4_gemv(c, s, t, f64(x))
    w_abs = np.abs(P.nvfp4_dequantize(c, s, t)).sum(axis=1)
    ok, worst, at = T.check(y_ref, f64(y), A, extra=2.0 ** -57 * 1.0 * w_abs[None, :])
    assert ok, (worst, at)
