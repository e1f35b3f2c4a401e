"""Python side of the whole-decode-step ABI: ctypes mirrors of bws_matrix,
bws_layer and bws_stack, and a runner that owns the plan and the workspace."""
import ctypes as C

import torch

from ._lib import lib, check, BwsError
from .api import MoeLayer, MoeWeights, Workspace, _ptr, _stream

FMT_NVFP4, FMT_MXFP4, FMT_FP8_ROW = 1, 2, 3
LAYER_MIXER_MLP, LAYER_MLP, LAYER_MOE = 1, 2, 3


class Matrix(C.Structure):
    _fields_ = [("format", C.c_int), ("d_out", C.c_int), ("d_in", C.c_int),
                ("codes", C.c_void_p), ("scales", C.c_void_p), ("scale32", C.c_void_p)]


class Layer(C.Structure):
    _fields_ = [("kind", C.c_int), ("n_mixer_in", C.c_int), ("mixer_in", Matrix * 4),
                ("mixer_out", Matrix), ("gate", Matrix), ("up", Matrix), ("down", Matrix),
                ("moe", MoeLayer), ("ids", C.c_void_p), ("route_w", C.c_void_p), ("topk", C.c_int),
                ("router", C.c_void_p)]


class Stack(C.Structure):
    _fields_ = [("hidden", C.c_int), ("n_layers", C.c_int), ("layers", C.POINTER(Layer)),
                ("head", Matrix), ("rms_eps", C.c_float)]


class QMatrix:
    """A quantized matrix on the device: format, codes, block scales, FP32 scale."""

    def __init__(self, fmt, codes, scales=None, scale32=None):
        self.fmt, self.codes, self.scales, self.scale32 = fmt, codes, scales, scale32
        self.d_out = codes.shape[0]
        self.d_in = codes.shape[1] * (2 if fmt in (FMT_NVFP4, FMT_MXFP4) else 1)

    def nbytes(self):
        b = self.codes.numel()
        if self.scales is not None:
            b += self.scales.numel()
        if self.fmt == FMT_FP8_ROW:
            b += self.scale32.numel() * 4
        return b

    def struct(self):
        return Matrix(self.fmt, self.d_out, self.d_in, _ptr(self.codes), _ptr(self.scales), _ptr(self.scale32))


class DecodeStack:
    """Layers: dicts with kind 'mixer_mlp' (mixer_in: [QMatrix], mixer_out,
    gate, up, down), 'mlp' (gate, up, down) or 'moe' (moe: MoeWeights, ids,
    route_w device tensors [N][topk]; optional 'router': bf16 [n_experts]
    [hidden], with which the step routes the layer itself and writes the
    chosen ids and weights into ids / route_w). head: QMatrix (FP8)."""

    def __init__(self, hidden, layers, head, N, rms_eps=1e-6, device="cuda"):
        self.hidden, self.layers_py, self.head, self.N = hidden, layers, head, N
        self.device = torch.device(device)
        arr = (Layer * max(1, len(layers)))()
        for i, L in enumerate(layers):
            s = arr[i]
            if L["kind"] == "mixer_mlp":
                s.kind = LAYER_MIXER_MLP
                s.n_mixer_in = len(L["mixer_in"])
                for j, m in enumerate(L["mixer_in"]):
                    s.mixer_in[j] = m.struct()
                s.mixer_out = L["mixer_out"].struct()
            elif L["kind"] == "mlp":
                s.kind = LAYER_MLP
            elif L["kind"] == "moe":
                s.kind = LAYER_MOE
                s.moe = L["moe"].descriptor()
                s.ids, s.route_w, s.topk = _ptr(L["ids"]), _ptr(L["route_w"]), L["ids"].shape[1]
                if L.get("router") is not None:
                    r = L["router"]
                    assert r.dtype == torch.bfloat16 and r.is_contiguous() and tuple(r.shape) == (L["moe"].n_experts, hidden)
                    s.router = _ptr(r)
            else:
                raise BwsError(f"unknown layer kind {L['kind']}")
            if L["kind"] in ("mixer_mlp", "mlp"):
                s.gate, s.up, s.down = L["gate"].struct(), L["up"].struct(), L["down"].struct()
        self._arr = arr
        self._stack = Stack(hidden, len(layers), C.cast(arr, C.POINTER(Layer)), head.struct(), rms_eps)
        plan = C.c_void_p()
        check(lib().bws_decode_step_plan_create(C.addressof(self._stack), N, C.byref(plan)),
              "bws_decode_step_plan_create")
        self.plan = plan
        self.ws = Workspace(self.device)
        self.ws.get(lib().bws_decode_step_workspace_size(plan))

    @property
    def kernel_count(self):
        return int(lib().bws_decode_step_kernel_count(self.plan))

    @property
    def workspace_bytes(self):
        return int(lib().bws_decode_step_workspace_size(self.plan))

    def step(self, x0, logits=None):
        if logits is None:
            logits = torch.empty((self.N, self.head.d_out), dtype=torch.float32, device=self.device)
        check(lib().bws_decode_step_stream(self.plan, _ptr(x0), _ptr(logits), self.ws.ptr, self.ws.nbytes,
                                           _stream(self.device)), "bws_decode_step_stream")
        return logits

    def step_greedy(self, x0, tokens=None, logits=None, row_token=None):
        """One step with the greedy next-token choice fused into the output
        layer: returns tokens int32 [N] (logits are stored too when a tensor
        is passed)."""
        if tokens is None:
            tokens = torch.empty(self.N, dtype=torch.int32, device=self.device)
        check(lib().bws_decode_step_greedy(self.plan, _ptr(x0), _ptr(logits), _ptr(row_token), _ptr(tokens),
                                           self.ws.ptr, self.ws.nbytes, _stream(self.device)),
              "bws_decode_step_greedy")
        return tokens

    def tap_size(self):
        return int(lib().bws_decode_step_tap_size(self.plan))

    def step_tap(self, x0, logits=None):
        """One step through bws_decode_step_tap: returns (logits, records),
        records being the list of device tensors (views of one tap buffer)
        in the order the C ABI writes them (see tap_layout)."""
        if logits is None:
            logits = torch.empty((self.N, self.head.d_out), dtype=torch.float32, device=self.device)
        n = self.tap_size()
        if n == 0:
            raise BwsError("this plan has no tap (persistent step kernel)")
        buf = torch.empty(n, dtype=torch.uint8, device=self.device)
        check(lib().bws_decode_step_tap(self.plan, _ptr(x0), _ptr(logits), self.ws.ptr, self.ws.nbytes, _ptr(buf), n,
                                        _stream(self.device)), "bws_decode_step_tap")
        recs, off = [], 0
        for kind, dtype, shape in self.tap_layout():
            nbytes = int(torch.Size(shape).numel()) * torch.tensor([], dtype=dtype).element_size()
            recs.append((kind, buf[off:off + nbytes].view(dtype).view(shape)))
            off += (nbytes + 255) // 256 * 256
        assert off == n, (off, n)
        return logits, recs

    def tap_layout(self):
        """(kind, dtype, shape) of each tap record, in order."""
        N, H = self.N, self.hidden
        out = []
        for L in self.layers_py:
            if L["kind"] == "mixer_mlp":
                out += [("a", torch.bfloat16, (N, H)), ("r", torch.float32, (N, H)),
                        ("v", torch.bfloat16, (N, L["mixer_out"].d_in))]
            if L["kind"] in ("mixer_mlp", "mlp"):
                out += [("m", torch.bfloat16, (N, H)), ("r", torch.float32, (N, H)),
                        ("h", torch.bfloat16, (N, L["gate"].d_out))]
            if L["kind"] == "moe":
                w = L["moe"]
                S = N * L["ids"].shape[1] + (1 if w.shared is not None else 0)
                out += [("m", torch.bfloat16, (N, H)), ("r", torch.float32, (N, H))]
                if L.get("router") is not None:
                    k = L["ids"].shape[1]
                    out += [("z", torch.float32, (N, w.n_experts)), ("ids", torch.int32, (N, k)),
                            ("route_w", torch.float32, (N, k))]
                out += [("n_slots", torch.int32, (1,)), ("slot_expert", torch.int32, (S,)),
                        ("cw", torch.float32, (S, N)), ("h_slots", torch.bfloat16, (S, N, w.inter)),
                        ("y_slots", torch.float32, (S, N, H))]
        out += [("x_head", torch.bfloat16, (N, H)), ("r", torch.float32, (N, H))]
        return out

    def weight_bytes(self, distinct_experts=None):
        """Algorithmic bytes of one step (codes + block/row scales, and the
        BF16 routers). For MoE layers pass the number of distinct routed
        experts per MoE layer."""
        b = self.head.nbytes()
        k = 0
        for L in self.layers_py:
            if L["kind"] == "mixer_mlp":
                b += sum(m.nbytes() for m in L["mixer_in"]) + L["mixer_out"].nbytes()
            if L["kind"] in ("mixer_mlp", "mlp"):
                b += L["gate"].nbytes() + L["up"].nbytes() + L["down"].nbytes()
            if L["kind"] == "moe":
                w = L["moe"]
                per = (w.gu_c[0].numel() + w.gu_s[0].numel() + w.dn_c[0].numel() + w.dn_s[0].numel())
                n = distinct_experts[k] + (1 if w.shared is not None else 0)
                b += n * per
                if L.get("router") is not None:
                    b += L["router"].numel() * 2
                k += 1
        return b

    def __del__(self):
        try:
            lib().bws_decode_step_plan_destroy(self.plan)
        except Exception:
            pass
