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


def nvfp4_prepare(x, d_out_max, ws):
    """Prepares x bf16 [N, d_in] in ws for nvfp4_gemv_prepared calls with
    d_out <= d_out_max (the activation prep of nvfp4_gemv, run once)."""
    _need_cuda(x)
    N, d_in = x.shape
    buf = _ws(ws, gemv_workspace_size(N, d_out_max, d_in), x.device)
    check(lib().bws_nvfp4_prepare(_ptr(x), N, d_in, d_out_max, _ptr(buf), buf.numel(), _stream(x.device)),
          "bws_nvfp4_prepare")
    return ws


def nvfp4_gemv_prepared(codes, scales, ts, N, d_in, ws, y=None):
    """y bf16 [N, d_out] = the activations last prepared in ws times the NVFP4
    matrix, transposed (the product kernel of nvfp4_gemv alone)."""
    _need_cuda(codes, scales, ts, y)
    d_out = codes.shape[0]
    if y is None:
        y = torch.empty((N, d_out), dtype=torch.bfloat16, device=codes.device)
    buf = _ws(ws, gemv_workspace_size(N, d_out, d_in), codes.device)
    check(lib().bws_nvfp4_gemv_prepared(_ptr(codes), _ptr(scales), _ptr(ts), N, d_out, d_in, _ptr(y), _ptr(buf),
                                        buf.numel(), _stream(codes.device)), "bws_nvfp4_gemv_prepared")
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


def fp8_lmhead_argmax(W, row_scale, x, logits=False, row_token=None, ws=None):
    """Greedy next-token choice fused into the FP8 output layer: int32 [N]
    rows of the largest logit (lowest row on ties), through row_token when
    given. logits=True also returns the fp32 [N, V] logits (a tensor may be
    passed to store them into)."""
    _need_cuda(W, row_scale, x)
    N, d = x.shape
    V = W.shape[0]
    if logits is True:
        logits = torch.empty((N, V), dtype=torch.float32, device=x.device)
    tok = torch.empty(N, dtype=torch.int32, device=x.device)
    buf = _ws(ws, gemv_workspace_size(N, V, d), x.device)
    check(lib().bws_fp8_lmhead_argmax(_ptr(W), _ptr(row_scale), _ptr(x), N, V, d,
                                      _ptr(logits) if logits is not False else None, _ptr(row_token), _ptr(tok),
                                      _ptr(buf), buf.numel(), _stream(x.device)), "bws_fp8_lmhead_argmax")
    return (tok, logits) if logits is not False else tok


def moe_router_topk(W_router, x, topk, logits=False, ws=None):
    """MoE routing on the device: the top-k experts of each token by the
    logits z = W_router x (BF16 operands, FP32 sums; lower id first on equal
    logits) and their softmax-renormalised weights. Returns (ids int32 [N, k],
    route_w fp32 [N, k]), largest logit first, plus the fp32 [N, E] logits
    when logits=True (a tensor may be passed to store them into)."""
    _need_cuda(W_router, x)
    N, d = x.shape
    E = W_router.shape[0]
    if logits is True:
        logits = torch.empty((N, E), dtype=torch.float32, device=x.device)
    ids = torch.empty((N, topk), dtype=torch.int32, device=x.device)
    w = torch.empty((N, topk), dtype=torch.float32, device=x.device)
    buf = _ws(ws, lib().bws_moe_router_workspace_size(N, E), x.device)
    check(lib().bws_moe_router_topk(_ptr(W_router), _ptr(x), N, E, d, topk,
                                    _ptr(logits) if logits is not False else None, _ptr(ids), _ptr(w),
                                    _ptr(buf), buf.numel(), _stream(x.device)), "bws_moe_router_topk")
    return (ids, w, logits) if logits is not False else (ids, w)


def mxfp8_quantize(x):
    """MXFP8 activations: x bf16 [N, d] -> (codes u8 [N, d] E4M3, scales u8
    [N, d/32] E8M0), one power-of-two scale per 32 values."""
    _need_cuda(x)
    N, d = x.shape
    codes = torch.empty((N, d), dtype=torch.uint8, device=x.device)
    scales = torch.empty((N, d // 32), dtype=torch.uint8, device=x.device)
    check(lib().bws_mxfp8_quantize(_ptr(x), N, d, _ptr(codes), _ptr(scales), _stream(x.device)),
          "bws_mxfp8_quantize")
    return codes, scales


def mxfp4_w4a8_gemv(codes, scales, x, y=None, ws=None):
    """W4A8 on the tensor cores: MXFP4 weights (codes u8 [d_out, d_in/2],
    E8M0 scales u8 [d_out, d_in/32]) times the MXFP8 quantization of x bf16
    [N, d_in] (N <= 8), FP32 accumulation; returns y bf16 [N, d_out]."""
    _need_cuda(codes, scales, x)
    N, d_in = x.shape
    d_out = codes.shape[0]
    if y is None:
        y = torch.empty((N, d_out), dtype=torch.bfloat16, device=x.device)
    buf = _ws(ws, lib().bws_w4a8_workspace_size(N, d_out, d_in), x.device)
    check(lib().bws_mxfp4_w4a8_gemv(_ptr(codes), _ptr(scales), _ptr(x), N, d_out, d_in, _ptr(y), _ptr(buf),
                                    buf.numel(), _stream(x.device)), "bws_mxfp4_w4a8_gemv")
    return y


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


# ---- MoE -------------------------------------------------------------------

import ctypes as _C


class MoeLayer(_C.Structure):
    """Mirror of struct bws_moe_layer (include/bws.h)."""
    _fields_ = [
        ("n_experts", _C.c_int), ("hidden", _C.c_int), ("inter", _C.c_int),
        ("gate_up_codes", _C.c_void_p), ("gate_up_codes_stride", _C.c_size_t),
        ("gate_up_scales", _C.c_void_p), ("gate_up_scales_stride", _C.c_size_t),
        ("down_codes", _C.c_void_p), ("down_codes_stride", _C.c_size_t),
        ("down_scales", _C.c_void_p), ("down_scales_stride", _C.c_size_t),
        ("shared_gate_up_codes", _C.c_void_p), ("shared_gate_up_scales", _C.c_void_p),
        ("shared_down_codes", _C.c_void_p), ("shared_down_scales", _C.c_void_p),
    ]


class MoeWeights:
    """Device tensors of one MXFP4 MoE layer, laid out as bws_moe_layer wants:
    gate_up codes [E, 2*inter, hidden/2], scales [E, 2*inter, hidden/32],
    down codes [E, hidden, inter/2], scales [E, hidden, inter/32], and the
    shared expert's four tensors (or None)."""

    def __init__(self, gate_up_codes, gate_up_scales, down_codes, down_scales, shared=None):
        self.gu_c, self.gu_s, self.dn_c, self.dn_s = gate_up_codes, gate_up_scales, down_codes, down_scales
        self.shared = shared
        E, two_i, _ = gate_up_codes.shape
        self.n_experts, self.inter, self.hidden = E, two_i // 2, down_codes.shape[1]

    def descriptor(self):
        d = MoeLayer()
        d.n_experts, d.hidden, d.inter = self.n_experts, self.hidden, self.inter
        d.gate_up_codes, d.gate_up_codes_stride = self.gu_c.data_ptr(), self.gu_c[0].numel()
        d.gate_up_scales, d.gate_up_scales_stride = self.gu_s.data_ptr(), self.gu_s[0].numel()
        d.down_codes, d.down_codes_stride = self.dn_c.data_ptr(), self.dn_c[0].numel()
        d.down_scales, d.down_scales_stride = self.dn_s.data_ptr(), self.dn_s[0].numel()
        if self.shared is not None:
            sgc, sgs, sdc, sds = self.shared
            d.shared_gate_up_codes, d.shared_gate_up_scales = sgc.data_ptr(), sgs.data_ptr()
            d.shared_down_codes, d.shared_down_scales = sdc.data_ptr(), sds.data_ptr()
        return d


def mxfp4_moe_workspace_size(layer, N, topk):
    d = layer.descriptor()
    return int(lib().bws_mxfp4_moe_workspace_size(_C.addressof(d), N, topk))


def mxfp4_moe_gemv(layer, ids, route_w, x, y=None, ws=None):
    """y bf16 [N, hidden] = shared(x) + sum_k route_w[:, k] * expert_{ids[:, k]}(x)."""
    _need_cuda(ids, route_w, x, y)
    N, hidden = x.shape
    topk = ids.shape[1]
    if y is None:
        y = torch.empty((N, hidden), dtype=torch.bfloat16, device=x.device)
    d = layer.descriptor()
    buf = _ws(ws, lib().bws_mxfp4_moe_workspace_size(_C.addressof(d), N, topk), x.device)
    check(lib().bws_mxfp4_moe_gemv(_C.addressof(d), _ptr(ids), _ptr(route_w), N, topk, _ptr(x), _ptr(y),
                                   _ptr(buf), buf.numel(), _stream(x.device)), "bws_mxfp4_moe_gemv")
    return y


def mxfp4_moe_inspect(layer, ws, N, topk):
    """(n_slots, slot experts, h bf16 [slots, N, inter], status) of the last call."""
    import numpy as np
    d = layer.descriptor()
    buf = ws.buf if isinstance(ws, Workspace) else ws
    max_slots = N * topk + (1 if layer.shared is not None else 0)
    n_slots = _C.c_int(0)
    status = _C.c_uint32(0)
    experts = np.zeros(max_slots, dtype=np.int32)
    h = np.zeros((max_slots, N, layer.inter), dtype=np.uint16)
    check(lib().bws_mxfp4_moe_inspect(_ptr(buf), _C.addressof(d), N, topk, _C.addressof(n_slots),
                                      experts.ctypes.data, h.ctypes.data, _C.addressof(status),
                                      _stream(buf.device)), "bws_mxfp4_moe_inspect")
    return n_slots.value, experts, h, status.value
