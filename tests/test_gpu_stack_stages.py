"""Every stage of a whole decode step, checked on its own against the oracle
from the GPU's own input to that stage (bws_decode_step_tap), at the product
bound |dy| <= 1e-4 sum|w x| + 1/2 ulp (see tests/stage_check.py).

* small dense and MoE stacks (every row of every stage; weights quantized
  by the oracle and uploaded);
* the 27B-shape dense stack at full size (64 layers, 48 linear-attention with
  a 46336x5120 input projection, 16 full-attention, MLP 17408x5120, FP8
  248320x5120 output layer) at N = 1 and N = 8;
* the Ling-shape MoE stack at full size (2 dense MLP layers, 40 MoE layers of
  512 experts with top-8 routing and a shared expert, FP8 157184x2560 output
  layer) at N = 1 and N = 4.

At full size the weights are quantized on the GPU (the oracle would take
hours over 19 GB); the checks then sample rows of each product: for every
sampled row the oracle quantizes the seeded FP32 weights itself, the GPU's
codes and scales of that row must equal the oracle's bit for bit, and the
stage is compared with the oracle's product over those rows. The per-tensor
NVFP4 scale needs the whole matrix's largest magnitude: it is taken by
torch.amax over the device copy of the seeded weights (a maximum is exact in
any order), then the oracle forms s_t from it. Element-wise stages (RMSNorm
inputs, residual updates of the MoE combine) are checked on every element."""
import numpy as np
import pytest
import torch

from oracle import quant as Q, products as P
from tests.gpu_util import device, bws
from tests.stack_util import oracle_quantizers
from tests import stage_check as SC
import synth

pytestmark = pytest.mark.gpu


# ---- providers -----------------------------------------------------------------

def _device_rows(qm):
    return lambda rows: SC.dequant_rows(qm, rows)


def _dense_rows_of(stack):
    def rows_of(li, name):
        if li is None:
            return _device_rows(stack.head)
        L = stack.layers_py[li]
        if name == "mixer_in":
            return SC.concat_provider([_device_rows(m) for m in L["mixer_in"]], [m.d_out for m in L["mixer_in"]])
        return _device_rows(L[name])
    return rows_of


def _expert_rows_small(stack):
    def expert_rows(li, e, name):
        w = stack.layers_py[li]["moe"]
        if e < 0:
            gc, gs, dc, ds = w.shared
        else:
            gc, gs, dc, ds = w.gu_c[e], w.gu_s[e], w.dn_c[e], w.dn_s[e]
        I = w.inter

        def rows(idx):
            idx = np.asarray(idx)
            if name == "down":
                return P.mxfp4_dequantize(dc[idx].cpu().numpy(), ds[idx].cpu().numpy())
            off = 0 if name == "gate" else I
            return P.mxfp4_dequantize(gc[idx + off].cpu().numpy(), gs[idx + off].cpu().numpy())
        return rows
    return expert_rows


class SeededRows:
    """Rows of a matrix the GPU quantized from the seeded FP32 weights: the
    oracle quantizes the same rows of the same FP32 weights itself, the GPU's
    codes and scales must match them exactly, and the oracle's rows are
    returned (FP64, dequantized)."""

    def __init__(self, fmt, shape, seed, index, qm, row_offset=0, rows_total=None, rep=None, what=""):
        self.fmt, self.shape, self.seed, self.index, self.qm = fmt, shape, seed, index, qm
        self.row_offset = row_offset          # rows of this matrix within a generated batch
        self.rows_total = rows_total or shape[0]
        self.rep, self.what = rep, what
        self.cache = {}

    def _w(self):
        return synth.weight_fp32((self.rows_total, self.shape[1]), seed=self.seed, index=self.index, device=device())

    def __call__(self, idx):
        idx = np.asarray(idx, dtype=np.int64)
        key = tuple(idx.tolist())
        if key in self.cache:
            return self.cache[key]
        W = self._w()
        sel = torch.from_numpy(idx + self.row_offset).to(W.device)
        rows = W.index_select(0, sel).cpu().numpy()
        if self.fmt == 1:
            amax = float(W.abs().amax().item())
            del W
            s_t = Q.nvfp4_tensor_scale(np.array([[amax]], dtype=np.float32))
            c, s, t = Q.nvfp4_quantize(rows, s_t=s_t)
            gc, gs = self.qm[0][idx].cpu().numpy(), self.qm[1][idx].cpu().numpy()
            ok = np.array_equal(gc, c) and np.array_equal(gs, s) and np.float32(self.qm[2].item()) == np.float32(t)
            out = P.nvfp4_dequantize(c, s, t)
        elif self.fmt == 2:
            del W
            c, s = Q.mxfp4_quantize(rows)
            gc, gs = self.qm[0][idx].cpu().numpy(), self.qm[1][idx].cpu().numpy()
            ok = np.array_equal(gc, c) and np.array_equal(gs, s)
            out = P.mxfp4_dequantize(c, s)
        else:
            del W
            c, r = Q.fp8_rowwise_quantize(rows)
            gc, gr = self.qm[0][idx].cpu().numpy(), self.qm[1][idx].cpu().numpy()
            ok = np.array_equal(gc, c) and np.array_equal(gr.view(np.uint32), r.view(np.uint32))
            out = P.fp8_dequantize(c, r)
        if self.rep is not None:
            self.rep.add("codes_bit_exact", self.what, ok, 0.0 if ok else float("inf"), None)
        self.cache[key] = out
        return out


def _qm_tuple(qm):
    return (qm.codes, qm.scales, qm.scale32) if qm.fmt == 1 else (
        (qm.codes, qm.scales, None) if qm.fmt == 2 else (qm.codes, qm.scale32, None))


def _dense_seeded(stack, seed, rep):
    """Providers for a stack built by workloads.dense_27b (matrix indices in
    that order: each layer's mixer inputs, mixer output, gate, up, down; the
    output layer at index 100000)."""
    from bit_weight_streaming_gb300 import workloads as W
    prov, idx = {}, 0
    for li, L in enumerate(stack.layers_py):
        ins = []
        for m in L["mixer_in"]:
            ins.append(SeededRows(m.fmt, (m.d_out, m.d_in), seed, idx, _qm_tuple(m), rep=rep, what=(li, "in", idx)))
            idx += 1
        prov[(li, "mixer_in")] = SC.concat_provider(ins, [m.d_out for m in L["mixer_in"]])
        for name in ("mixer_out", "gate", "up", "down"):
            m = L[name]
            prov[(li, name)] = SeededRows(m.fmt, (m.d_out, m.d_in), seed, idx, _qm_tuple(m), rep=rep, what=(li, name))
            idx += 1
    h = stack.head
    prov[(None, "head")] = SeededRows(h.fmt, (h.d_out, h.d_in), seed, 100000, _qm_tuple(h), rep=rep, what="head")
    return lambda li, name: prov[(li, name)]


def _moe_seeded(stack, seed, rep, n_dense):
    """Providers for a stack built by workloads.moe_ling (dense layer matrices
    at 2000000 + 8 i + k; expert tensors drawn 64 experts at a time at
    1000000 + 4096 layer + 2 e0 + k; the output layer at 100001)."""
    prov = {}
    for li in range(n_dense):
        L = stack.layers_py[li]
        for k, name in enumerate(("gate", "up", "down")):
            m = L[name]
            prov[(li, name)] = SeededRows(m.fmt, (m.d_out, m.d_in), seed, 2000000 + 8 * li + k, _qm_tuple(m),
                                          rep=rep, what=(li, name))
    h = stack.head
    prov[(None, "head")] = SeededRows(h.fmt, (h.d_out, h.d_in), seed, 100001, _qm_tuple(h), rep=rep, what="head")
    cache = {}

    def expert_rows(li, e, name):
        key = (li, e, name)
        if key not in cache:
            w = stack.layers_py[li]["moe"]
            E, I, H = w.n_experts, w.inter, w.hidden
            ee = E if e < 0 else e           # the shared expert is drawn after the routed ones
            e0 = ee // 64 * 64
            nb = min(64, E + 1 - e0)
            if e < 0:
                gc, gs, dc, ds = w.shared
            else:
                gc, gs, dc, ds = w.gu_c[e], w.gu_s[e], w.dn_c[e], w.dn_s[e]
            if name == "down":
                cache[key] = SeededRows(2, (H, I), seed, 1000000 + 4096 * li + 2 * e0 + 1, (dc, ds, None),
                                        row_offset=(ee - e0) * H, rows_total=nb * H, rep=rep, what=(li, e, name))
            else:
                off = 0 if name == "gate" else I
                base = SeededRows(2, (2 * I, H), seed, 1000000 + 4096 * li + 2 * e0, (gc, gs, None),
                                  row_offset=(ee - e0) * 2 * I, rows_total=nb * 2 * I, rep=rep, what=(li, e, name))
                cache[key] = lambda idx, base=base, off=off: base(np.asarray(idx) + off)
        return cache[key]
    return (lambda li, name: prov[(li, name)]), expert_rows


# ---- small stacks: every row ------------------------------------------------------

@pytest.mark.parametrize("N", [1, 3, 8])
def test_dense_stages_every_row(N):
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    stack = W.dense_27b(N, seed=5, n_layers=4, hidden=1024, inter=2048, vocab=1500, attn=(1536, 256, 256, 1024),
                        gdn=(2560, 1024), quant=oracle_quantizers(device()), device=device())
    x0 = synth.activation_bf16(N, 1024, seed=40 + N, device=device())
    logits, recs = stack.step_tap(x0)
    torch.cuda.synchronize()
    ref_logits = stack.step(x0)
    torch.cuda.synchronize()
    assert torch.equal(logits, ref_logits), "the tap must not change the step"
    rep = SC.Report()
    SC.check_dense_stack(rep, stack, recs, logits, x0, _dense_rows_of(stack))
    print(rep.summary())
    rep.assert_ok(expect=("rmsnorm", "mixer_in", "mixer_out", "swiglu", "down", "head"))


@pytest.mark.parametrize("N", [1, 4, 8])
def test_moe_stages_every_row(N):
    from bit_weight_streaming_gb300 import workloads as W
    m = bws()
    layers = W.moe_stack_layers(N, seed=6, n_dense=1, n_moe=3, hidden=512, inter=256, n_experts=64, topk=8,
                                dense_inter=768, quant=oracle_quantizers(device()), device=device())
    head = W.make_matrix(3, (1200, 512), 6, 9, oracle_quantizers(device()), device())
    stack = m.stack.DecodeStack(512, layers, head, N, device=device())
    x0 = synth.activation_bf16(N, 512, seed=50 + N, device=device())
    logits, recs = stack.step_tap(x0)
    torch.cuda.synchronize()
    rep = SC.Report()
    SC.check_moe_stack(rep, stack, recs, logits, x0, _dense_rows_of(stack), _expert_rows_small(stack))
    print(rep.summary())
    rep.assert_ok(expect=("slot_table", "rmsnorm", "swiglu", "expert_down", "combine", "down", "head"))


@pytest.mark.parametrize("N", [1, 4, 8])
def test_routed_moe_stages_every_row(N):
    # the MoE layers route themselves: a BF16 router per layer, the step
    # writing the chosen ids and weights that the experts then use
    from bit_weight_streaming_gb300 import workloads as W
    m = bws()
    layers = W.moe_stack_layers(N, seed=7, n_dense=1, n_moe=3, hidden=512, inter=256, n_experts=64, topk=8,
                                dense_inter=768, quant=oracle_quantizers(device()), device=device(), router=True)
    head = W.make_matrix(3, (1200, 512), 7, 9, oracle_quantizers(device()), device())
    stack = m.stack.DecodeStack(512, layers, head, N, device=device())
    x0 = synth.activation_bf16(N, 512, seed=90 + N, device=device())
    logits, recs = stack.step_tap(x0)
    torch.cuda.synchronize()
    assert torch.equal(logits, stack.step(x0)), "the tap must not change the step"
    # the ids and weights the step wrote into each layer's tensors are the ones its tap recorded
    tap_ids = [t for k, t in recs if k == "ids"]
    tap_w = [t for k, t in recs if k == "route_w"]
    assert len(tap_ids) == len(tap_w) == 3
    for L, i, w in zip(layers[1:], tap_ids, tap_w):
        assert torch.equal(L["ids"], i) and torch.equal(L["route_w"], w)
    rep = SC.Report()
    SC.check_moe_stack(rep, stack, recs, logits, x0, _dense_rows_of(stack), _expert_rows_small(stack))
    print(rep.summary())
    rep.assert_ok(expect=("router", "router_topk", "slot_table", "rmsnorm", "swiglu", "expert_down", "combine",
                          "down", "head"))
    assert rep.count["router_topk"] == 3 and rep.count["router_oracle_set"] == 3 * N


# ---- full size ---------------------------------------------------------------------

@pytest.fixture(scope="module")
def stack27b():
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    s = W.dense_27b(1, seed=0, device=device())
    torch.cuda.synchronize()
    yield s
    del s
    torch.cuda.empty_cache()


@pytest.mark.parametrize("N", [1, 8])
def test_27b_shape_stack_stages_full_size(stack27b, N):
    m = bws()
    stack = stack27b if N == 1 else m.stack.DecodeStack(stack27b.hidden, stack27b.layers_py, stack27b.head, N,
                                                        device=device())
    x0 = synth.activation_bf16(N, stack.hidden, seed=60 + N, device=device())
    logits, recs = stack.step_tap(x0)
    torch.cuda.synchronize()
    rep = SC.Report()
    SC.check_dense_stack(rep, stack, recs, logits, x0, _dense_seeded(stack, 0, rep), k_rows=16, seed=N)
    print(N, rep.summary())
    rep.assert_ok(expect=("codes_bit_exact", "rmsnorm", "mixer_in", "mixer_out", "swiglu", "down", "head"))
    # per layer the first mixer input projection (the stand-in mixer reads its first d_v outputs), the mixer
    # output, gate, up and down were sampled, and the output layer
    assert rep.count["codes_bit_exact"] == 5 * len(stack.layers_py) + 1


@pytest.mark.parametrize("N", [1, 4])
def test_ling_shape_moe_stack_stages_full_size(N):
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    stack = W.moe_ling(N, seed=0, device=device())
    torch.cuda.synchronize()
    x0 = synth.activation_bf16(N, stack.hidden, seed=70 + N, device=device())
    logits, recs = stack.step_tap(x0)
    torch.cuda.synchronize()
    rep = SC.Report()
    rows_of, expert_rows = _moe_seeded(stack, 0, rep, n_dense=2)
    SC.check_moe_stack(rep, stack, recs, logits, x0, rows_of, expert_rows, k_rows=24, seed=N)
    print(N, rep.summary())
    rep.assert_ok(expect=("codes_bit_exact", "slot_table", "rmsnorm", "swiglu", "expert_down", "combine", "down",
                          "head"))
    assert rep.count["slot_table"] == 40 and rep.count["combine"] == 40
    del stack
    torch.cuda.empty_cache()


@pytest.mark.parametrize("N", [1, 4])
def test_routed_ling_shape_moe_stack_stages_full_size(N):
    # the Ling-shape stack with a 512 x 2560 BF16 router in each of its 40 MoE layers
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    stack = W.moe_ling(N, seed=0, device=device(), router=True)
    torch.cuda.synchronize()
    x0 = synth.activation_bf16(N, stack.hidden, seed=75 + N, device=device())
    logits, recs = stack.step_tap(x0)
    torch.cuda.synchronize()
    rep = SC.Report()
    rows_of, expert_rows = _moe_seeded(stack, 0, rep, n_dense=2)
    SC.check_moe_stack(rep, stack, recs, logits, x0, rows_of, expert_rows, k_rows=24, seed=N)
    print(N, rep.summary())
    rep.assert_ok(expect=("codes_bit_exact", "router", "router_topk", "slot_table", "rmsnorm", "swiglu",
                          "expert_down", "combine", "down", "head"))
    assert rep.count["router_topk"] == 40 and rep.count["combine"] == 40
    assert rep.count["router_oracle_set"] == 40 * N
    del stack
    torch.cuda.empty_cache()


@pytest.mark.parametrize("N", [1, 8])
def test_mixer_input_rows_the_stand_in_discards(N):
    """The stand-in mixer reads only the first d_v outputs of the mixer input
    projections, so the stage checks above never see the other rows. They are
    checked here through bws_nvfp4_gemv (the same product kernel) at full
    size: the 46336x5120 linear-attention input projection on 64 rows spread
    over all of it, and the 1024x5120 key projection on every row."""
    from bit_weight_streaming_gb300 import workloads as W
    m = bws()
    rep = SC.Report()
    for shape, index, k_rows in (((46336, 5120), 9000, 60), ((1024, 5120), 9001, None)):
        qm = W.make_matrix(1, shape, 0, index, device=device())
        x = synth.activation_bf16(N, shape[1], seed=80 + N, device=device())
        y = m.nvfp4_gemv(qm.codes, qm.scales, qm.scale32, x)
        torch.cuda.synchronize()
        rows = np.arange(shape[0]) if k_rows is None else SC.sample_rows(shape[0], k_rows, index + N)
        prov = SeededRows(1, shape, 0, index, _qm_tuple(qm), rep=rep, what=shape)
        SC.check_product(rep, "product", shape, prov(rows), SC.f64(x), SC.f64(y)[:, rows])
        del qm
    print(N, rep.summary())
    rep.assert_ok(expect=("codes_bit_exact", "product"))


# ---- the mixed checkpoint: FP8 mixers, NVFP4 MLPs then FP8 in the last layers --------------

@pytest.mark.parametrize("N", [1, 8])
def test_mixed_checkpoint_stages_every_row(N):
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    stack = W.dense_27b_mixed(N, seed=9, n_layers=4, hidden=1024, inter=2048, vocab=1500,
                              attn=(1536, 256, 256, 1024), gdn=(1792, 1024), n_fp8_from=2,
                              quant=oracle_quantizers(device()), device=device())
    fmts = [(L["mixer_out"].fmt, L["down"].fmt) for L in stack.layers_py]
    assert fmts == [(3, 1), (3, 1), (3, 3), (3, 3)]
    x0 = synth.activation_bf16(N, 1024, seed=120 + N, device=device())
    logits, recs = stack.step_tap(x0)
    torch.cuda.synchronize()
    assert torch.equal(logits, stack.step(x0))
    rep = SC.Report()
    SC.check_dense_stack(rep, stack, recs, logits, x0, _dense_rows_of(stack))
    print(rep.summary())
    rep.assert_ok(expect=("rmsnorm", "mixer_in", "mixer_out", "swiglu", "down", "head"))


@pytest.mark.parametrize("N", [1, 8])
def test_mixed_checkpoint_stages_full_size(N):
    from bit_weight_streaming_gb300 import workloads as W
    bws()
    stack = W.dense_27b_mixed(N, seed=0, device=device())
    torch.cuda.synchronize()
    x0 = synth.activation_bf16(N, stack.hidden, seed=130 + N, device=device())
    logits, recs = stack.step_tap(x0)
    torch.cuda.synchronize()
    rep = SC.Report()
    SC.check_dense_stack(rep, stack, recs, logits, x0, _dense_seeded(stack, 0, rep), k_rows=16, seed=N)
    print(N, rep.summary())
    rep.assert_ok(expect=("codes_bit_exact", "rmsnorm", "mixer_in", "mixer_out", "swiglu", "down", "head"))
    assert rep.count["codes_bit_exact"] == 5 * len(stack.layers_py) + 1
    del stack
    torch.cuda.empty_cache()
