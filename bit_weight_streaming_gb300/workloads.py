"""Synthetic weight-stream workloads built on the device.

Weights are drawn by the seeded generators in ``synth`` (W ~ N(0, 0.02) in
FP32, one stream per tensor) and quantized by this library's GPU quantizers;
a caller may inject other quantizers (the tests inject the oracle's, so that
the oracle never consumes a CUDA-path output).

Shapes follow the workloads the pages describe:
* the 27B-shape dense stack: 64 layers of hidden 5120, MLP 17408, every
  fourth layer full attention (Wq 12288x5120, Wk, Wv 1024x5120, Wo 5120x6144),
  the other 48 a linear-attention block whose fused input projection
  (46336x5120) and output projection (5120x6144) are sized so that the stack
  totals 17.82 GB, plus a 248320x5120 FP8 output layer;
* the MoE stack: hidden 2560, 2 dense MLP layers (intermediate 6912), 40 MoE
  layers of 512 experts (intermediate 768, top-8 + 1 shared) in MXFP4, and a
  157184x2560 FP8 output layer.
"""
import torch

import synth
from . import api
from .stack import QMatrix, DecodeStack, FMT_NVFP4, FMT_MXFP4, FMT_FP8_ROW


def gpu_quantizers():
    return {
        FMT_NVFP4: lambda W: api.nvfp4_quantize(W),
        FMT_MXFP4: lambda W: api.mxfp4_quantize(W),
        FMT_FP8_ROW: lambda W: api.fp8_rowwise_quantize(W),
    }


def make_matrix(fmt, shape, seed, index, quant=None, device="cuda"):
    quant = quant or gpu_quantizers()
    W = synth.weight_fp32(shape, seed=seed, index=index, device=device)
    out = quant[fmt](W)
    del W
    if fmt == FMT_NVFP4:
        c, s, t = out
        return QMatrix(fmt, c, s, t)
    if fmt == FMT_MXFP4:
        c, s = out
        return QMatrix(fmt, c, s, None)
    c, r = out
    return QMatrix(fmt, c, None, r)


# ---- the dense 27B-shape stack ------------------------------------------------

def dense_layer_shapes(i, hidden=5120, inter=17408, attn=(12288, 1024, 1024, 6144), gdn=(46336, 6144)):
    """(mixer_in shapes, mixer_out shape, mlp shapes) of layer i."""
    if i % 4 == 3:
        q, k, v, dv = attn
        mixer_in = [(q, hidden), (k, hidden), (v, hidden)]
        mixer_out = (hidden, dv)
    else:
        d_in_proj, dv = gdn
        mixer_in = [(d_in_proj, hidden)]
        mixer_out = (hidden, dv)
    return mixer_in, mixer_out, {"gate": (inter, hidden), "up": (inter, hidden), "down": (hidden, inter)}


def dense_stack_layers(n_layers, seed=0, hidden=5120, inter=17408, attn=(12288, 1024, 1024, 6144),
                       gdn=(46336, 6144), fmt=FMT_NVFP4, quant=None, device="cuda"):
    """fmt: one format for every matrix, or fmt(layer, part) with part
    'mixer' or 'mlp'."""
    fmt_of = fmt if callable(fmt) else (lambda i, part: fmt)
    layers = []
    idx = 0
    for i in range(n_layers):
        mixer_in, mixer_out, mlp = dense_layer_shapes(i, hidden, inter, attn, gdn)
        L = {"kind": "mixer_mlp", "mixer_in": []}
        fm, fl = fmt_of(i, "mixer"), fmt_of(i, "mlp")
        for s in mixer_in:
            L["mixer_in"].append(make_matrix(fm, s, seed, idx, quant, device)); idx += 1
        L["mixer_out"] = make_matrix(fm, mixer_out, seed, idx, quant, device); idx += 1
        for name in ("gate", "up", "down"):
            L[name] = make_matrix(fl, mlp[name], seed, idx, quant, device); idx += 1
        layers.append(L)
    return layers


# The pages' mixed checkpoint ([Spark27B] "Fewer bytes per weight: NVFP4"):
# FP8 attention and linear-attention projections in every layer, NVFP4 MLPs
# in layers 0-55 and FP8 MLPs in the last eight; the MLPs are 59 % of the
# layer bytes. With FP8 mixers the linear-attention projections are sized
# down to 14336x5120 in and 5120x8192 out so that the layers total 17.77 GB
# (the pages: 17.83 GB).
MIXED_GDN = (14336, 8192)
MIXED_FP8_MLP_FROM = 56


def mixed_fmt(n_fp8_from=MIXED_FP8_MLP_FROM):
    return lambda i, part: FMT_FP8_ROW if (part == "mixer" or i >= n_fp8_from) else FMT_NVFP4


def dense_27b_mixed(N, seed=0, n_layers=64, hidden=5120, inter=17408, vocab=248320, attn=(12288, 1024, 1024, 6144),
                    gdn=MIXED_GDN, n_fp8_from=MIXED_FP8_MLP_FROM, quant=None, device="cuda"):
    layers = dense_stack_layers(n_layers, seed, hidden, inter, attn, gdn, mixed_fmt(n_fp8_from), quant, device)
    head = make_matrix(FMT_FP8_ROW, (vocab, hidden), seed, 100000, quant, device)
    return DecodeStack(hidden, layers, head, N, device=device)


def dense_27b(N, seed=0, n_layers=64, hidden=5120, inter=17408, vocab=248320, attn=(12288, 1024, 1024, 6144),
              gdn=(46336, 6144), quant=None, device="cuda"):
    layers = dense_stack_layers(n_layers, seed, hidden, inter, attn, gdn, FMT_NVFP4, quant, device)
    head = make_matrix(FMT_FP8_ROW, (vocab, hidden), seed, 100000, quant, device)
    return DecodeStack(hidden, layers, head, N, device=device)


# ---- the MoE stack ------------------------------------------------------------------

def moe_weights(n_experts, hidden, inter, seed, layer, with_shared=True, quant=None, device="cuda",
                batch=64):
    """Stacked MXFP4 expert tensors of one MoE layer (gate rows then up rows).
    Experts are drawn and quantized `batch` at a time (one FP32 draw per
    batch and tensor kind; MXFP4 rows are independent, so quantizing the
    stacked rows equals quantizing each expert)."""
    quant = quant or gpu_quantizers()
    n = n_experts + (1 if with_shared else 0)
    gu_c = torch.empty((n, 2 * inter, hidden // 2), dtype=torch.uint8, device=device)
    gu_s = torch.empty((n, 2 * inter, hidden // 32), dtype=torch.uint8, device=device)
    dn_c = torch.empty((n, hidden, inter // 2), dtype=torch.uint8, device=device)
    dn_s = torch.empty((n, hidden, inter // 32), dtype=torch.uint8, device=device)
    for e0 in range(0, n, batch):
        nb = min(batch, n - e0)
        for k, (shape, c_dst, s_dst) in enumerate([((2 * inter, hidden), gu_c, gu_s), ((hidden, inter), dn_c, dn_s)]):
            W = synth.weight_fp32((nb * shape[0], shape[1]), seed=seed, index=1000000 + 4096 * layer + 2 * e0 + k,
                                  device=device)
            c, s = quant[FMT_MXFP4](W)
            c_dst[e0:e0 + nb].copy_(c.view(nb, shape[0], -1))
            s_dst[e0:e0 + nb].copy_(s.view(nb, shape[0], -1))
            del W
    shared = (gu_c[n_experts], gu_s[n_experts], dn_c[n_experts], dn_s[n_experts]) if with_shared else None
    return api.MoeWeights(gu_c[:n_experts], gu_s[:n_experts], dn_c[:n_experts], dn_s[:n_experts], shared)


def router_weights(n_experts, hidden, seed, layer, device="cuda"):
    """A BF16 [n_experts][hidden] router: seeded N(0, 0.02) FP32 rounded to
    BF16 (nearest, ties to even)."""
    return synth.weight_fp32((n_experts, hidden), seed=seed, index=3000000 + layer, device=device).to(torch.bfloat16)


def moe_stack_layers(N, seed=0, n_dense=2, n_moe=40, hidden=2560, inter=768, n_experts=512, topk=8,
                     dense_inter=6912, quant=None, device="cuda", router=False):
    """router=False: seeded expert ids and combine weights (inputs); True: a
    BF16 router per MoE layer, the step choosing ids and weights itself and
    writing them into the layer's ids / route_w tensors."""
    layers = []
    for i in range(n_dense):
        L = {"kind": "mlp"}
        for k, (name, shape) in enumerate([("gate", (dense_inter, hidden)), ("up", (dense_inter, hidden)),
                                           ("down", (hidden, dense_inter))]):
            L[name] = make_matrix(FMT_MXFP4, shape, seed, 2000000 + 8 * i + k, quant, device)
        layers.append(L)
    for j in range(n_moe):
        li = n_dense + j
        w = moe_weights(n_experts, hidden, inter, seed, li, True, quant, device)
        if router:
            layers.append({"kind": "moe", "moe": w, "router": router_weights(n_experts, hidden, seed, li, device),
                           "ids": torch.zeros((N, topk), dtype=torch.int32, device=device),
                           "route_w": torch.zeros((N, topk), dtype=torch.float32, device=device)})
            continue
        ids = synth.expert_ids(N, topk, n_experts, seed=seed, layer=li)
        rw = synth.route_weights(N, topk, seed=seed, layer=li)
        layers.append({"kind": "moe", "moe": w, "ids": ids.to(device), "route_w": rw.to(device), "ids_host": ids,
                       "route_w_host": rw})
    return layers


def moe_ling(N, seed=0, n_dense=2, n_moe=40, hidden=2560, inter=768, n_experts=512, topk=8, dense_inter=6912,
             vocab=157184, quant=None, device="cuda", router=False):
    layers = moe_stack_layers(N, seed, n_dense, n_moe, hidden, inter, n_experts, topk, dense_inter, quant, device,
                              router)
    head = make_matrix(FMT_FP8_ROW, (vocab, hidden), seed, 100001, quant, device)
    return DecodeStack(hidden, layers, head, N, device=device)


def distinct_per_moe_layer(stack):
    """Distinct routed experts per MoE layer (a routed stack: those of the
    ids its last step wrote)."""
    return [len(set((L["ids_host"] if "ids_host" in L else L["ids"].cpu()).reshape(-1).tolist()))
            for L in stack.layers_py if L["kind"] == "moe"]
