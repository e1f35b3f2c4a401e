"""Python names of the C entry points (argument marshalling only)."""
import torch

from ._lib import lib, check, BwsError


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device=None):
    return torch.cuda.current_stream(device).cuda_stream


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise BwsError("tensors must be contiguous CUDA tensors")


class Workspace:
    """A caller-owned scratch buffer, grown on demand (256-byte aligned)."""

    def __init__(self, device="cuda"):
        self.device = torch.device(device)
        self.buf = None

    def get(self, nbytes):
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)
        return self.buf

    @property
    def ptr(self):
        return self.buf.data_ptr()

    @property
    def nbytes(self):
        return self.buf.numel()


def _ws(ws, nbytes, device):
    if ws is None:
        ws = Workspace(device)
    buf = ws.get(nbytes) if isinstance(ws, Workspace) else ws
    return buf


def nvfp4_quantize(W, ws=None):
    """W fp32 [d_out, d_in] -> (codes u8 [d_out, d_in/2], scales u8 [d_out, d_in/16], s_t fp32 [1])."""
    _need_cuda(W)
    d_out, d_in = W.shape
    codes = torch.empty((d_out, d_in // 2), dtype=torch.uint8, device=W.device)
    scales = torch.empty((d_out, d_in // 16), dtype=torch.uint8, device=W.device)
    ts = torch.empty((1,), dtype=torch.float32, device=W.device)
    buf = _ws(ws, lib().bws_nvfp4_quantize_workspace_size(d_out, d_in), W.device)
    check(lib().bws_nvfp4_quantize(_ptr(W), d_out, d_in, _ptr(codes), _ptr(scales), _ptr(ts),
                                   _ptr(buf), buf.numel(), _stream(W.device)), "bws_nvfp4_quantize")
    return codes, scales, ts


def mxfp4_quantize(W):
    """W fp32 [rows, d_in] -> (codes u8 [rows, d_in/2], scales u8 [rows, d_in/32])."""
    _need_cuda(W)
    rows, d_in = W.shape
    codes = torch.empty((rows, d_in // 2), dtype=torch.uint8, device=W.device)
    scales = torch.empty((rows, d_in // 32), dtype=torch.uint8, device=W.device)
    check(lib().bws_mxfp4_quantize(_ptr(W), rows, d_in, _ptr(codes), _ptr(scales), _stream(W.device)),
          "bws_mxfp4_quantize")
    return codes, scales


def fp8_rowwise_quantize(W):
    """W fp32 [rows, cols] -> (codes u8 [rows, cols], row_scale fp32 [rows])."""
    _need_cuda(W)
    rows, cols = W.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=W.device)
    rs = torch.empty((rows,), dtype=torch.float32, device=W.device)
    check(lib().bws_fp8_rowwise_quantize(_ptr(W), rows, cols, _ptr(codes), _ptr(rs), _stream(W.device)),
          "bws_fp8_rowwise_quantize")
    return codes, rs


def gemv_workspace_size(N, d_out_total, d_in):
    return int(lib().bws_gemv_workspace_size(N, d_out_total, d_in))


def nvfp4_gemv(codes, scales, ts, x, y=None, ws=None):
    """y bf16 [N, d_out] = x bf16 [N, d_in] times the NVFP4 matrix, transposed."""
    _need_cuda(codes, scales, ts, x, y)
    N, d_in = x.shape
    d_out = codes.shape[0]
    if y is None:
        y = torch.empty((N, d_out), dtype=torch.bfloat16, device=x.device)
    buf = _ws(ws, gemv_workspace_size(N, d_out, d_in), x.device)
    check(lib().bws_nvfp4_gemv(_ptr(codes), _ptr(scales), _ptr(ts), _ptr(x), N, d_out, d_in, _ptr(y),
                               _ptr(buf), buf.numel(), _stream(x.device)), "bws_nvfp4_gemv")
    return y


def nvfp4_gate_up_silu(gate, up, x, h=None, ws=None):
    """gate, up: (codes, scales, ts) NVFP4 [d_inter, d_in]; h bf16 [N, d_inter]."""
    _need_cuda(*gate, *up, x, h)
    N, d_in = x.shape
    d_inter = gate[0].shape[0]
    if h is None:
        h = torch.empty((N, d_inter), dtype=torch.bfloat16, device=x.device)
    buf = _ws(ws, gemv_workspace_size(N, 2 * d_inter, d_in), x.device)
    check(lib().bws_nvfp4_gate_up_silu(_ptr(gate[0]), _ptr(gate[1]), _ptr(gate[2]), _ptr(up[0]), _ptr(up[1]),
                                       _ptr(up[2]), _ptr(x), N, d_inter, d_in, _ptr(h), _ptr(buf),
                                       buf.numel(), _stream(x.device)), "bws_nvfp4_gate_up_silu")
    return h


def fp8_lmhead_gemv(W, row_scale, x, logits=None, ws=None):
    """logits fp32 [N, V] for an FP8 row-scaled head W u8 [V, d]."""
    _need_cuda(W, row_scale, x, logits)
    N, d = x.shape
    V = W.shape[0]
    if logits is None:
        logits = torch.empty((N, V), dtype=torch.float32, device=x.device)
    buf = _ws(ws, gemv_workspace_size(N, V, d), x.device)
    check(lib().bws_fp8_lmhead_gemv(_ptr(W), _ptr(row_scale), _ptr(x), N, V, d, _ptr(logits), _ptr(buf),
                                    buf.numel(), _stream(x.device)), "bws_fp8_lmhead_gemv")
    return logits


def status_word(ws):
    """OR of the status bits set by the last product call that used ws."""
    import ctypes
    buf = ws.buf if isinstance(ws, Workspace) else ws
    out = ctypes.c_uint32(0)
    check(lib().bws_status_word(_ptr(buf), ctypes.addressof(out), _stream(buf.device)), "bws_status_word")
    return out.value


def hbm_read_probe(src, out):
    _need_cuda(src, out)
    check(lib().bws_hbm_read_probe(_ptr(src), src.numel() * src.element_size(), _ptr(out),
                                   _stream(src.device)), "bws_hbm_read_probe")


def l2_flush(buf):
    _need_cuda(buf)
    check(lib().bws_l2_flush(_ptr(buf), buf.numel() * buf.element_size(), _stream(buf.device)), "bws_l2_flush")
