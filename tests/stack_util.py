"""Shared by the stack tests: oracle-quantized device stacks and the oracle's
view of them."""
import numpy as np
import torch

from oracle import quant as Q, products as P, model as M, formats as F

FMT_NVFP4, FMT_MXFP4, FMT_FP8_ROW = 1, 2, 3


def oracle_quantizers(device):
    """Quantizers for workloads.make_matrix that run the oracle on the CPU and
    upload its codes: device weights then carry no CUDA-path output."""
    def nv(W):
        c, s, t = Q.nvfp4_quantize(W.cpu().numpy())
        return (torch.from_numpy(c).to(device), torch.from_numpy(s).to(device),
                torch.tensor([float(t)], dtype=torch.float32, device=device))

    def mx(W):
        c, s = Q.mxfp4_quantize(W.cpu().numpy())
        return torch.from_numpy(c).to(device), torch.from_numpy(s).to(device)

    def f8(W):
        c, r = Q.fp8_rowwise_quantize(W.cpu().numpy())
        return torch.from_numpy(c).to(device), torch.from_numpy(r).to(device)
    return {FMT_NVFP4: nv, FMT_MXFP4: mx, FMT_FP8_ROW: f8}


def dequant(qm):
    c = qm.codes.cpu().numpy()
    if qm.fmt == FMT_NVFP4:
        return P.nvfp4_dequantize(c, qm.scales.cpu().numpy(), np.float32(qm.scale32.item()))
    if qm.fmt == FMT_MXFP4:
        return P.mxfp4_dequantize(c, qm.scales.cpu().numpy())
    return P.fp8_dequantize(c, qm.scale32.cpu().numpy())


def oracle_layers(stack):
    out = []
    for L in stack.layers_py:
        if L["kind"] == "mixer_mlp":
            out.append({"kind": "mixer_mlp", "in": [dequant(m) for m in L["mixer_in"]], "out": dequant(L["mixer_out"]),
                        "gate": dequant(L["gate"]), "up": dequant(L["up"]), "down": dequant(L["down"])})
        elif L["kind"] == "mlp":
            out.append({"kind": "mlp", "gate": dequant(L["gate"]), "up": dequant(L["up"]), "down": dequant(L["down"])})
        else:
            w = L["moe"]
            cache = {}

            def expert(e, w=w, cache=cache):
                if e not in cache:
                    if e < 0:
                        gc, gs, dc, ds = w.shared
                    else:
                        gc, gs, dc, ds = w.gu_c[e], w.gu_s[e], w.dn_c[e], w.dn_s[e]
                    gu = P.mxfp4_dequantize(gc.cpu().numpy(), gs.cpu().numpy())
                    dn = P.mxfp4_dequantize(dc.cpu().numpy(), ds.cpu().numpy())
                    cache[e] = (gu[: w.inter], gu[w.inter:], dn)
                return cache[e]
            out.append({"kind": "moe", "moe": {"ids": L["ids_host"].numpy(), "route_w": L["route_w_host"].numpy(),
                                               "expert": expert, "shared": expert(-1) if w.shared is not None else None}})
    return out


def oracle_layer_fn(r, L):
    if L["kind"] == "mixer_mlp":
        return M.dense_layer(r, L)
    return M.moe_layer(r, L)


def oracle_logits(stack, x0):
    layers = oracle_layers(stack)
    head = dequant(stack.head)
    return M.decode_stack(x0, layers, head, layer_fn=oracle_layer_fn)


# End-to-end slack for activation roundings: BF16 activations at stage
# boundaries may legitimately differ by one ulp when the FP32 (GPU) and FP64
# (oracle) values straddle a rounding boundary; their propagated effect on the
# logits is allowed up to 2^-6 of the logits' RMS. The CPU test
# test_oracle_stack_sensitivity pins that the oracle's own response to such
# flips stays well inside this slack.
STACK_SLACK = 2.0 ** -6
