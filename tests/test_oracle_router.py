"""Pins of the oracle's MoE router (oracle.model.router_topk) and of the
top-k acceptance rule the GPU tests use (tests/topk_rule.py).

The router is this project's reading of [LingMoE] section 3 (each token goes
to 8 of 512 routed experts): logits z = W_r x, the k largest chosen (equal
logits: lower id first), weights the softmax of the chosen logits. The pins
below do not restate that code: they are hand-worked cases, closed forms of
special cases, a brute-force search over subsets and a library softmax."""
import itertools

import numpy as np
import pytest

from oracle import model as M
from topk_rule import acceptable_set, ordered, weight_interval


def _route(z_col, topk):
    """Route one token whose logits are z_col: W_r's first column holds them
    and x = [1, 0], so z = W_r x = z_col exactly."""
    E = len(z_col)
    W = np.zeros((E, 2))
    W[:, 0] = z_col
    W[:, 1] = np.arange(E) * 0.25   # multiplied by x[1] = 0
    return M.router_topk(W, np.array([[1.0, 0.0]]), topk)


def test_hand_worked_two_of_four_with_a_tie():
    # z = [0.5, 2, 2, -1]: the two largest are equal, so both weigh 1/2 and
    # expert 1 (the lower id) comes first
    ids, w, z, A = _route([0.5, 2.0, 2.0, -1.0], 2)
    assert ids.tolist() == [[1, 2]]
    assert w.tolist() == [[0.5, 0.5]]
    assert z.tolist() == [[0.5, 2.0, 2.0, -1.0]]
    assert A.tolist() == [[0.5, 2.0, 2.0, 1.0]]


def test_hand_worked_three_of_four():
    # chosen logits 2, 2, 0.5: weights 1 / (2 + e^-1.5) twice and
    # e^-1.5 / (2 + e^-1.5), with e^-1.5 = 0.22313016014842982
    ids, w, _, _ = _route([0.5, 2.0, 2.0, -1.0], 3)
    assert ids.tolist() == [[1, 2, 0]]
    np.testing.assert_allclose(w[0], [0.4498162176582741, 0.4498162176582741, 0.10036756468345168],
                               rtol=1e-15, atol=0)


def test_all_equal_logits_pick_the_lowest_ids_evenly():
    ids, w, _, _ = _route([1.25] * 7, 4)
    assert ids.tolist() == [[0, 1, 2, 3]]
    assert w.tolist() == [[0.25] * 4]


def test_choosing_every_expert_is_the_full_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    z = rng.standard_normal(9)
    ids, w, _, _ = _route(z, 9)
    assert sorted(ids[0].tolist()) == list(range(9))
    np.testing.assert_allclose(w[0], softmax(z)[ids[0]], rtol=1e-14)


@pytest.mark.parametrize("seed", range(20))
def test_brute_force_top_set_maximises_the_sum(seed):
    # the top-k set of distinct logits is the k-subset with the largest sum,
    # and its weights are the full softmax renormalised over it
    from scipy.special import softmax
    rng = np.random.default_rng(seed)
    E, k = 6, 3
    z = rng.standard_normal(E)
    ids, w, _, _ = _route(z, k)
    best = max(itertools.combinations(range(E), k), key=lambda s: sum(z[list(s)]))
    assert sorted(ids[0].tolist()) == sorted(best)
    assert np.all(np.diff(z[ids[0]]) <= 0), "largest first"
    p = softmax(z)[ids[0]]
    np.testing.assert_allclose(w[0], p / p.sum(), rtol=1e-14)


def test_several_tokens_and_a_real_product():
    # two tokens of d = 4 with BF16-exact operands; logits worked by hand:
    # token 0: x = [1, 0.5, 0, 0] -> z = [1.5, -0.5, 1.0]
    # token 1: x = [0, 0, 2, 1]   -> z = [0, 3.0, -1.0]
    W = np.array([[1.0, 1.0, 0.0, 0.0],
                  [0.0, -1.0, 1.0, 1.0],
                  [1.0, 0.0, -0.5, 0.0]])
    X = np.array([[1.0, 0.5, 0.0, 0.0], [0.0, 0.0, 2.0, 1.0]])
    ids, w, z, A = M.router_topk(W, X, 1)
    assert z.tolist() == [[1.5, -0.5, 1.0], [0.0, 3.0, -1.0]]
    assert A.tolist() == [[1.5, 0.5, 1.0], [0.0, 3.0, 1.0]]
    assert ids.tolist() == [[0], [1]]
    assert w.tolist() == [[1.0], [1.0]]


def test_rejects_topk_outside_the_experts():
    with pytest.raises(ValueError):
        _route([1.0, 2.0], 3)


def test_moe_layer_routes_with_the_router():
    # a router whose logits favour experts 2 and 0 sends the token there, so
    # the layer equals the MoE with those ids and the router's weights
    rng = np.random.default_rng(5)
    d, inter, E = 8, 4, 3
    experts = [tuple(rng.standard_normal(s) * 0.1 for s in ((inter, d), (inter, d), (d, inter))) for _ in range(E)]
    W_r = rng.standard_normal((E, d)) * 0.3
    r = rng.standard_normal((1, d))
    m = M.round_bf16(M.rmsnorm(r))
    ids, w, _, _ = M.router_topk(W_r, m, 2)
    got = M.moe_layer(r, {"moe": {"router": W_r, "topk": 2, "expert": lambda e: experts[e], "shared": None}})
    want = r + M.moe(m, ids, w, lambda e: experts[e], None)
    np.testing.assert_array_equal(got, want)


# ---- the acceptance rule -----------------------------------------------------

def test_rule_clear_margin_accepts_only_the_oracle_set():
    z = np.array([3.0, 2.0, 1.0, 0.0])
    b = np.full(4, 0.1)
    assert acceptable_set(z, b, [0, 1])
    assert acceptable_set(z, b, [1, 0])          # the set, not the order
    assert not acceptable_set(z, b, [0, 2])
    assert not acceptable_set(z, b, [0, 0])      # not distinct
    assert not acceptable_set(z, b, [0, 4])      # out of range


def test_rule_near_tie_accepts_either():
    # experts 1 and 2 within their bounds of each other: 2 - 0.6 <= 1 + 0.6
    z = np.array([3.0, 2.0, 1.0, 0.0])
    b = np.array([0.0, 0.6, 0.6, 0.0])
    assert acceptable_set(z, b, [0, 1]) and acceptable_set(z, b, [0, 2])
    assert not acceptable_set(z, b, [0, 3])
    assert ordered(z, b, [0, 2, 1]) and not ordered(z, b, [3, 0])


def test_rule_weight_interval():
    z = np.array([2.0, 2.0, 0.5, -1.0])
    lo, hi = weight_interval(z, np.zeros(4), [1, 2, 0])
    w = np.array([0.4498162176582741, 0.10036756468345168, 0.4498162176582741])
    assert np.all(lo <= w) and np.all(w <= hi)
    assert np.all(hi - lo <= 64 * 2.0 ** -24)
    # a logit bound of 0.01 moves a weight by about 1 % at most
    lo, hi = weight_interval(z, np.full(4, 0.01), [1, 2, 0])
    assert np.all(lo < w * 0.995) and np.all(hi > w * 1.005) and np.all(hi < w * 1.03)


@pytest.mark.parametrize("bad", ["ascending", "ties_high", "unnormalised"])
def test_router_planted_mistakes_are_caught(monkeypatch, bad):
    """Plausible slips in the routing rule must fail the hand-worked pins."""
    def broken(w_router, X, topk):
        from oracle.products import matvec
        z, A = matvec(w_router, X)
        N, E = z.shape
        ids = np.zeros((N, topk), dtype=np.int64)
        for n in range(N):
            if bad == "ascending":
                ids[n] = np.argsort(z[n], kind="stable")[:topk]
            elif bad == "ties_high":
                ids[n] = (E - 1 - np.argsort(-z[n][::-1], kind="stable"))[:topk]
            else:
                ids[n] = np.argsort(-z[n], kind="stable")[:topk]
        zc = np.take_along_axis(z, ids, axis=1)
        if bad == "unnormalised":   # the full softmax, not renormalised over the chosen
            e = np.exp(z - z.max(axis=1, keepdims=True))
            return ids, np.take_along_axis(e / e.sum(axis=1, keepdims=True), ids, axis=1), z, A
        e = np.exp(zc - zc[:, :1])
        return ids, e / e.sum(axis=1, keepdims=True), z, A

    monkeypatch.setattr(M, "router_topk", broken)
    failed = 0
    for pin in (test_hand_worked_two_of_four_with_a_tie, test_hand_worked_three_of_four,
                test_all_equal_logits_pick_the_lowest_ids_evenly):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, f"planted mistake {bad} passed every pin"
