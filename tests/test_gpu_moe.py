"""GPU MXFP4 mixture-of-experts layer against the oracle.

Checked: the slot table (bit-exact: shared expert first, then the distinct
routed experts in ascending order), the SwiGLU activations of every slot, and
y. Every expected value and every bound comes from the oracle alone. The y
bound adds to the product bound the largest legitimate difference in h: h is
BF16-rounded on both sides from values that may differ by the h bound e_h,
so |dh| <= e_h + ulp_bf16(|h| + e_h), which moves y by |W_down| |dh|:
|dy| <= sum_s cw_s (1e-4 sum|D h| + sum_j |D_ij| dh_j) + 1e-6 sum_s cw_s |ys|
+ 1/2 ulp(y).
"""
import numpy as np
import pytest
import torch

from oracle import quant as Q, products as P, model as M, formats as F, tolerance as T
from tests.gpu_util import device, bws, np_, f64
import synth


def _build(E, hidden, inter, seed, with_shared, gpu_quant=False, used=None, layer=0):
    """Expert weights for the GPU and the oracle's dequantized view of each
    expert. The oracle's view always comes from the oracle's own quantizer
    run on the CPU. The device tensors hold the same oracle codes, or, with
    gpu_quant (the full-size shape), the GPU quantizer's codes of the same
    FP32 weights, checked bit-exact against the oracle's for every expert in
    `used` (only those are read); the other experts stay zero."""
    dev = device()
    n = E + (1 if with_shared else 0)
    gu_c = torch.zeros((n, 2 * inter, hidden // 2), dtype=torch.uint8, device=dev)
    gu_s = torch.zeros((n, 2 * inter, hidden // 32), dtype=torch.uint8, device=dev)
    dn_c = torch.zeros((n, hidden, inter // 2), dtype=torch.uint8, device=dev)
    dn_s = torch.zeros((n, hidden, inter // 32), dtype=torch.uint8, device=dev)
    want = range(n) if used is None else sorted(set(E if e < 0 else e for e in used))
    oracle_codes = {}
    for e in want:
        Wgu = synth.weight_fp32((2 * inter, hidden), seed=seed, index=1000 * layer + 2 * e)
        Wd = synth.weight_fp32((hidden, inter), seed=seed, index=1000 * layer + 2 * e + 1)
        cg, sg = Q.mxfp4_quantize(Wgu.numpy())
        cd, sd = Q.mxfp4_quantize(Wd.numpy())
        oracle_codes[e] = (cg, sg, cd, sd)
        if gpu_quant:
            c, s_ = bws().mxfp4_quantize(Wgu.to(dev))
            assert np.array_equal(np_(c), cg) and np.array_equal(np_(s_), sg)
            gu_c[e].copy_(c); gu_s[e].copy_(s_)
            c, s_ = bws().mxfp4_quantize(Wd.to(dev))
            assert np.array_equal(np_(c), cd) and np.array_equal(np_(s_), sd)
            dn_c[e].copy_(c); dn_s[e].copy_(s_)
        else:
            gu_c[e].copy_(torch.from_numpy(cg)); gu_s[e].copy_(torch.from_numpy(sg))
            dn_c[e].copy_(torch.from_numpy(cd)); dn_s[e].copy_(torch.from_numpy(sd))
    shared = (gu_c[E], gu_s[E], dn_c[E], dn_s[E]) if with_shared else None
    layer_w = bws().MoeWeights(gu_c[:E], gu_s[:E], dn_c[:E], dn_s[:E], shared)
    cache = {}

    def expert(e):
        if e not in cache:
            cg, sg, cd, sd = oracle_codes[E if e < 0 else e]
            gu = P.mxfp4_dequantize(cg, sg)
            dn = P.mxfp4_dequantize(cd, sd)
            cache[e] = (gu[:inter], gu[inter:], dn)
        return cache[e]
    return layer_w, expert


def _check_moe(layer_w, expert, ids, rw, x, with_shared, rows=None):
    dev = device()
    N, topk = ids.shape
    ws = bws().Workspace(dev)
    y = bws().mxfp4_moe_gemv(layer_w, ids.to(dev), rw.to(dev), x, ws=ws)
    n_slots, slot_exp, h_bits, status = bws().mxfp4_moe_inspect(layer_w, ws, N, topk)
    ids_np = ids.numpy()
    valid = (ids_np >= 0) & (ids_np < layer_w.n_experts)
    want_slots = ([-1] if with_shared else []) + sorted(set(ids_np[valid].tolist()))
    assert n_slots == len(want_slots)
    assert slot_exp[:n_slots].tolist() == want_slots
    assert bool(status & 4) == (not valid.all())
    X = f64(x)
    rwn = rw.numpy().astype(np.float64)
    Y = np.zeros((N, layer_w.hidden))
    bound = np.zeros((N, layer_w.hidden))
    cw_abs_ys = np.zeros((N, layer_w.hidden))
    for s, e in enumerate(want_slots):
        wg, wu, wd = expert(e)
        g, Ag = P.matvec(wg, X)
        u, Au = P.matvec(wu, X)
        h_exact = M.silu(g) * u
        h_gpu = F.bf16_bits_to_float(h_bits[s])
        sig = 1.0 / (1.0 + np.exp(-g))
        dsilu = np.abs(sig * (1.0 + g * (1.0 - sig)))
        tg, tu = 1e-4 * Ag, 1e-4 * Au
        extra = dsilu * np.abs(u) * tg + np.abs(M.silu(g)) * tu + 1.1 * tg * tu + 1e-6 * np.abs(h_exact)
        ok, worst, at = T.check(h_exact, h_gpu, np.zeros_like(h_exact), extra=extra)
        assert ok, ("h", e, worst, at)
        h_ref = F.round_bf16(h_exact)
        ys, A = P.matvec(wd, h_ref)
        e_h = extra + 0.5 * F.bf16_ulp(np.abs(h_exact) + extra)   # the h bound checked above
        dh = e_h + F.bf16_ulp(np.abs(h_exact) + e_h)
        cw = np.ones(N) if e < 0 else np.array([rwn[t][ids_np[t] == e].sum() for t in range(N)])
        Y += cw[:, None] * ys
        bound += np.abs(cw)[:, None] * (1e-4 * A + dh @ np.abs(wd).T)
        cw_abs_ys += np.abs(cw)[:, None] * np.abs(ys)
    # the oracle's own MoE (its BF16 h) must agree with the per-slot sum above
    Yo = M.moe(X, np.where(valid, ids_np, 0), np.where(valid, rwn, 0.0), expert,
               shared=expert(-1) if with_shared else None)
    assert np.allclose(Yo, Y, rtol=1e-12, atol=1e-30)
    yg = f64(y)
    if rows is not None:
        yg, Y, bound, cw_abs_ys = yg[:, rows], Y[:, rows], bound[:, rows], cw_abs_ys[:, rows]
    ok, worst, at = T.check(Y, yg, np.zeros_like(Y), extra=bound + 1e-6 * cw_abs_ys)
    assert ok, ("y", worst, at)


@pytest.mark.gpu
@pytest.mark.parametrize("N", [1, 3, 8])
def test_moe_small(N):
    E, hidden, inter, topk = 16, 256, 128, 4
    layer_w, expert = _build(E, hidden, inter, seed=31, with_shared=True)
    ids = synth.expert_ids(N, topk, E, seed=N)
    rw = synth.route_weights(N, topk, seed=N)
    x = synth.activation_bf16(N, hidden, seed=N, device=device())
    _check_moe(layer_w, expert, ids, rw, x, with_shared=True)


@pytest.mark.gpu
@pytest.mark.parametrize("N,hidden,inter", [(1, 512, 256), (3, 512, 256), (8, 512, 256), (2, 256, 96),
                                            (1, 768, 512), (5, 1024, 768)])
def test_moe_stream_shapes(N, hidden, inter):
    """Shapes that take the TMA expert kernels (hidden and, for down, the
    intermediate size a multiple of 256), with several tiles per slot, a
    ragged last gate/up tile, and fewer units than CTAs."""
    E, topk = 24, 4
    layer_w, expert = _build(E, hidden, inter, seed=hidden + inter, with_shared=True)
    ids = synth.expert_ids(N, topk, E, seed=40 + N)
    rw = synth.route_weights(N, topk, seed=40 + N)
    x = synth.activation_bf16(N, hidden, seed=40 + N, device=device())
    _check_moe(layer_w, expert, ids, rw, x, with_shared=True)


@pytest.mark.gpu
def test_moe_no_shared_and_bad_id():
    E, hidden, inter, topk = 12, 320, 96, 3
    layer_w, expert = _build(E, hidden, inter, seed=5, with_shared=False)
    ids = synth.expert_ids(2, topk, E, seed=7)
    ids[1, 2] = E + 3                      # out of range: skipped and flagged
    rw = synth.route_weights(2, topk, seed=7)
    x = synth.activation_bf16(2, hidden, seed=7, device=device())
    _check_moe(layer_w, expert, ids, rw, x, with_shared=False)


@pytest.mark.gpu
def test_moe_single_expert_reduces_to_mlp():
    E, hidden, inter = 8, 256, 64
    layer_w, expert = _build(E, hidden, inter, seed=9, with_shared=False)
    ids = torch.tensor([[5]], dtype=torch.int32)
    rw = torch.tensor([[1.0]], dtype=torch.float32)
    x = synth.activation_bf16(1, hidden, seed=9, device=device())
    _check_moe(layer_w, expert, ids, rw, x, with_shared=False)


@pytest.mark.gpu
@pytest.mark.parametrize("N", [1, 4])
def test_moe_full_size_ling_shape(N):
    """512 experts, hidden 2560, intermediate 768, top-8 plus a shared expert,
    at one token and at the four-token verify width; device codes from the GPU
    quantizer (bit-exact against the oracle's for every expert the tokens
    use); every h value and every one of the 2560 output rows compared."""
    E, hidden, inter, topk = 512, 2560, 768, 8
    ids = synth.expert_ids(N, topk, E, seed=0, layer=2)
    rw = synth.route_weights(N, topk, seed=0, layer=2)
    used = sorted(set(ids.numpy().reshape(-1).tolist())) + [-1]
    layer_w, expert = _build(E, hidden, inter, seed=0, with_shared=True, gpu_quant=True, used=used)
    x = synth.activation_bf16(N, hidden, seed=0, device=device())
    _check_moe(layer_w, expert, ids, rw, x, with_shared=True)
