"""The greedy next-token choice fused into the FP8 output layer
(bws_fp8_lmhead_argmax, bws_decode_step_greedy), through the C ABI.

* Against the oracle on the reduced-vocabulary head's 100,032 rows (d = 256,
  weights quantized by the oracle; tiles split across CTAs): the token must
  be an acceptable greedy choice for the oracle's exact logits within the
  product bound (tests/argmax_rule.py), the stored logits within the bound.
* Against the GPU's own logits: the token is the lowest index of the largest
  stored logit, with and without storing the logits, and through a row ->
  token map.
* A planted exact tie (a row copied into a lower row): the lower row wins.
* Full size, 100032x5120 and 248320x5120 (GPU-quantized from the seeded
  weights): the token agrees with the stored logits, and sampled rows plus
  the chosen row are compared with the oracle (codes bit-exact).
* The decode step: bws_decode_step_greedy picks the same tokens as the
  argmax of its logits, on the kernel chain and in graph replay."""
import numpy as np
import pytest
import torch

from oracle import products as P, tolerance as T
from tests.gpu_util import device, bws, f64
from tests.stack_util import oracle_quantizers
from tests.argmax_rule import acceptable
from tests import stage_check as SC
import synth

pytestmark = pytest.mark.gpu


def _lowest_argmax(v):
    m = v.max(axis=1, keepdims=True)
    return np.argmax(v == m, axis=1)


def _head(V, d, seed, index, quant=None):
    from bit_weight_streaming_gb300 import workloads as W
    return W.make_matrix(3, (V, d), seed, index, quant, device())


@pytest.mark.parametrize("N", [1, 4])
def test_reduced_head_argmax_against_the_oracle(N):
    m = bws()
    V, d = 100032, 256
    h = _head(V, d, 3, 500, oracle_quantizers(device()))
    x = synth.activation_bf16(N, d, seed=90 + N, device=device())
    tok, logits = m.fp8_lmhead_argmax(h.codes, h.scale32, x, logits=True)
    torch.cuda.synchronize()
    y, A = P.fp8_gemv(h.codes.cpu().numpy(), h.scale32.cpu().numpy(), f64(x))
    ok, worst, at = T.check(y, f64(logits), A)
    assert ok, (worst, at)
    b = T.bound(y, f64(logits), A)
    tk = tok.cpu().numpy()
    for n in range(N):
        assert acceptable(y[n], b[n], int(tk[n])), (n, int(tk[n]), int(np.argmax(y[n])))
    assert np.array_equal(tk, _lowest_argmax(f64(logits)))
    # without storing the logits, and through a row -> token map
    tok2 = m.fp8_lmhead_argmax(h.codes, h.scale32, x)
    perm = torch.randperm(V, generator=torch.Generator().manual_seed(1)).to(torch.int32).to(device())
    tok3 = m.fp8_lmhead_argmax(h.codes, h.scale32, x, row_token=perm)
    torch.cuda.synchronize()
    assert torch.equal(tok2, tok) and torch.equal(tok3, perm[tok.long()])


def test_exact_tie_goes_to_the_lower_row():
    m = bws()
    V, d = 4096, 512
    h = _head(V, d, 4, 501, oracle_quantizers(device()))
    x = synth.activation_bf16(1, d, seed=7, device=device())
    top = int(m.fp8_lmhead_argmax(h.codes, h.scale32, x)[0])
    lower = 17 if top > 17 else V - 1
    h.codes[lower].copy_(h.codes[top])
    h.scale32[lower].copy_(h.scale32[top])
    tok, logits = m.fp8_lmhead_argmax(h.codes, h.scale32, x, logits=True)
    torch.cuda.synchronize()
    assert logits[0, lower].item() == logits[0, top].item()
    assert int(tok[0]) == min(lower, top)


@pytest.mark.parametrize("V", [100032, 248320])
def test_full_size_heads(V):
    from tests.test_gpu_stack_stages import SeededRows, _qm_tuple
    m = bws()
    d = 5120
    h = _head(V, d, 0, 502)
    rep = SC.Report()
    for N in (1, 8):
        x = synth.activation_bf16(N, d, seed=100 + N, device=device())
        tok, logits = m.fp8_lmhead_argmax(h.codes, h.scale32, x, logits=True)
        tok2 = m.fp8_lmhead_argmax(h.codes, h.scale32, x)
        torch.cuda.synchronize()
        L = f64(logits)
        tk = tok.cpu().numpy()
        assert np.array_equal(tk, _lowest_argmax(L)) and torch.equal(tok, tok2)
        rows = np.unique(np.concatenate([SC.sample_rows(V, 40, V + N), tk]))
        prov = SeededRows(3, (V, d), 0, 502, _qm_tuple(h), rep=rep, what=(V, N))
        SC.check_product(rep, "head", (V, N), prov(rows), f64(x), L[:, rows])
    print(V, rep.summary())
    rep.assert_ok(expect=("codes_bit_exact", "head"))


@pytest.mark.parametrize("N", [1, 3])
def test_decode_step_greedy(N):
    from bit_weight_streaming_gb300 import workloads as W
    m = bws()
    stack = W.dense_27b(N, seed=8, n_layers=2, hidden=512, inter=1024, vocab=3000, attn=(768, 256, 256, 512),
                        gdn=(1280, 512), quant=oracle_quantizers(device()), device=device())
    x0 = synth.activation_bf16(N, 512, seed=110 + N, device=device())
    logits = stack.step(x0)
    tok_direct = stack.step_greedy(x0)                   # default stream: direct launches
    s = torch.cuda.Stream()
    lg2 = torch.empty_like(logits)
    with torch.cuda.stream(s):
        t1 = stack.step_greedy(x0, logits=lg2).clone()   # records a graph
        t2 = stack.step_greedy(x0, logits=lg2).clone()   # replays it
    s.synchronize()
    torch.cuda.synchronize()
    want = _lowest_argmax(f64(logits))
    assert np.array_equal(tok_direct.cpu().numpy(), want)
    assert torch.equal(t1, tok_direct) and torch.equal(t2, tok_direct) and torch.equal(lg2, logits)
