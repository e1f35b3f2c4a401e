"""The MoE router on the GPU (bws_moe_router_topk) against the oracle's
router_topk: logits at the product bound |dz| <= 1e-4 sum|w x| + 1/2 ulp,
each token's chosen experts an acceptable top-k for the exact logits within
those bounds (largest first), combine weights within the softmax's interval
for such logits (tests/topk_rule.py). The router inside the decode step is
checked stage by stage in test_gpu_stack_stages.py."""
import numpy as np
import pytest
import torch

from oracle import model as M, tolerance as T
from tests.gpu_util import device, bws
from topk_rule import acceptable_set, ordered, weight_interval
import synth

pytestmark = pytest.mark.gpu


def _router(E, d, seed):
    return synth.weight_fp32((E, d), seed=seed, index=7, device=device()).to(torch.bfloat16)


def _check(W, x, ids, w, z_gpu=None):
    """Returns the number of tokens whose set is the oracle's own top-k."""
    Wf = W.float().cpu().numpy().astype(np.float64)
    X = x.float().cpu().numpy().astype(np.float64)
    k = ids.shape[1]
    oid, ow, z, A = M.router_topk(Wf, X, k)
    ids, w = ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)
    if z_gpu is not None:
        ok, worst, at = T.check(z, z_gpu.cpu().numpy(), A)
        assert ok, (worst, at)
        b = T.bound(z, z_gpu.cpu().numpy(), A)
    else:
        b = T.bound(z, z, A)
    same = 0
    for n in range(z.shape[0]):
        assert acceptable_set(z[n], b[n], ids[n]), (n, ids[n], oid[n])
        assert ordered(z[n], b[n], ids[n]), (n, ids[n])
        lo, hi = weight_interval(z[n], b[n], ids[n])
        assert np.all(lo <= w[n]) and np.all(w[n] <= hi), (n, w[n], lo, hi)
        same += set(ids[n].tolist()) == set(oid[n].tolist())
    return same


@pytest.mark.parametrize("N", [1, 4, 8])
def test_router_ling_shape(N):
    # 512 experts over hidden 2560, top-8 ([LingMoE] section 3)
    m = bws()
    W = _router(512, 2560, seed=N)
    x = synth.activation_bf16(N, 2560, seed=80 + N, device=device())
    ids, w, z = m.moe_router_topk(W, x, 8, logits=True)
    torch.cuda.synchronize()
    same = _check(W, x, ids, w, z)
    # the GPU's FP32 sums sit far closer to the exact logits than the bound:
    # its set is the oracle's own unless two logits agree to about 1e-6
    assert same == N


@pytest.mark.parametrize("E,d,N,k", [(37, 256, 3, 5), (8, 64, 2, 8), (1, 8, 1, 1), (2048, 7168, 8, 8),
                                     (100, 2568, 5, 3)])
def test_router_shapes_and_edges(E, d, N, k):
    # a partial last CTA (37, 100 experts), every expert chosen (8 of 8), a
    # single expert, the largest sizes, a width that is not a multiple of 256
    m = bws()
    W = _router(E, d, seed=E + d)
    x = synth.activation_bf16(N, d, seed=E, device=device())
    ids, w, z = m.moe_router_topk(W, x, k, logits=True)
    ids2, w2 = m.moe_router_topk(W, x, k)   # logits kept in the workspace: same choice
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2) and torch.equal(w, w2)
    _check(W, x, ids, w, z)
    if k == E:
        assert torch.allclose(w.sum(dim=1), torch.ones(N, device=w.device), atol=1e-6)


def test_router_tie_picks_the_lower_id():
    # experts 3 and 7 have the same row, larger than every other: equal logits
    # to the bit, so expert 3 ranks first and, with both chosen, each weighs 1/2
    m = bws()
    E, d = 16, 512
    W = _router(E, d, seed=9)
    x = synth.activation_bf16(2, d, seed=9, device=device()).abs()
    W[3] = 0.125
    W[7] = 0.125
    ids1, w1 = m.moe_router_topk(W, x, 1)
    ids2, w2 = m.moe_router_topk(W, x, 2)
    torch.cuda.synchronize()
    assert ids1.cpu().tolist() == [[3], [3]] and w1.cpu().tolist() == [[1.0], [1.0]]
    assert ids2.cpu().tolist() == [[3, 7], [3, 7]] and w2.cpu().tolist() == [[0.5, 0.5], [0.5, 0.5]]


def test_router_near_ties_are_acceptable():
    # experts whose rows differ by one BF16 ulp in a single weight: their
    # logits lie within each other's bounds, so either may be chosen, and the
    # choice must still pass the acceptance rule with its weights in range
    m = bws()
    E, d, N = 64, 1024, 4
    W = _router(E, d, seed=21)
    x = synth.activation_bf16(N, d, seed=22, device=device()).abs()
    base = torch.full((d,), 0.0625, dtype=torch.bfloat16, device=device())
    for e in (5, 9, 40):
        W[e] = base
    W[9, 0] = torch.tensor(0.0625 + 2.0 ** -11, dtype=torch.bfloat16)   # one BF16 ulp above 2^-4
    ids, w, z = m.moe_router_topk(W, x, 2, logits=True)
    torch.cuda.synchronize()
    _check(W, x, ids, w, z)
    assert set(ids[:, 0].cpu().tolist()) <= {5, 9, 40}
