"""Layer recipe around the weight stream: SwiGLU MLP, top-k MoE with a
shared expert, weightless RMSNorm, and the dense / MoE decode stacks.

Activations crossing a stage boundary are BF16 (``round_bf16``); the residual
stream is kept unrounded in FP64 here (FP32 on the GPU). Every matrix product
is the exact FP64 product of ``products``.

The pages give the order of the MLP (gate and up, SiLU, down: [Spark27B]
§ "Decode speed is bytes divided by bandwidth", flow figure) and state that
the token-mixing operation reads no weights. They give no normalisation,
mixer arithmetic, shared-expert width or combine weights; the readings used
for those (weightless RMSNorm, eps 1e-6; the mixer replaced by taking the
first d_in(W_o) entries of its input projection; combine weights normalised
to sum to 1; a shared expert of the routed experts' shape with weight 1; a
BF16 router whose k largest logits choose the experts, weighted by their
softmax) are this project's readings, not the pages'.
"""
import numpy as np

from .formats import round_bf16
from .products import matvec

RMS_EPS = 1e-6


def silu(g):
    """SiLU(g) = g / (1 + e^-g), FP64."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def rmsnorm(r, eps=RMS_EPS):
    """Weightless RMSNorm over the last axis: r / sqrt(mean(r^2) + eps)."""
    r = np.asarray(r, dtype=np.float64)
    ms = np.mean(r * r, axis=-1, keepdims=True)
    return r / np.sqrt(ms + eps)


def swiglu_hidden(w_gate, w_up, X):
    """h = BF16(SiLU(W_gate x) * (W_up x)) for each token row of X.
    Returns (h, g, u) with g, u the unrounded FP64 projections."""
    g, _ = matvec(w_gate, X)
    u, _ = matvec(w_up, X)
    return round_bf16(silu(g) * u), g, u


def mlp(w_gate, w_up, w_down, X):
    """Dense SwiGLU MLP: y = W_down BF16(SiLU(W_gate x) * W_up x)."""
    h, _, _ = swiglu_hidden(w_gate, w_up, X)
    y, _ = matvec(w_down, h)
    return y


def distinct_experts(ids):
    """Sorted distinct expert ids among all tokens' routed experts."""
    return np.unique(np.asarray(ids).reshape(-1))


def expected_distinct(n_experts, topk, n_tokens):
    """E[#distinct experts] when each of n_tokens independently routes to
    topk distinct experts chosen uniformly: E * (1 - (1 - k/E)^n)
    ([LingMoE] §八)."""
    return n_experts * (1.0 - (1.0 - topk / n_experts) ** n_tokens)


def router_topk(w_router, X, topk):
    """Routing of an MoE layer ([LingMoE] section 3: every token goes to 8 of
    the 512 routed experts, plus the shared one). The pages give no router
    arithmetic; the reading taken here:

    z[n, e]   = sum_j W_r[e, j] * x[n, j]   (exact, FP64; W_r and x BF16)
    ids[n]    = the topk experts with the largest z[n, .], largest first;
                of two equal logits the lower expert id ranks first
    route_w[n, i] = exp(z_i) / sum over the chosen j of exp(z_j)
                (the softmax over all experts, renormalised over the chosen)

    Returns (ids int64 [N, k], route_w [N, k], z [N, E], A [N, E]) with A the
    absolute sums the product bound uses."""
    z, A = matvec(w_router, X)
    N, E = z.shape
    if not 1 <= topk <= E:
        raise ValueError("topk must be in [1, n_experts]")
    ids = np.zeros((N, topk), dtype=np.int64)
    for n in range(N):
        # descending by logit; a stable sort keeps equal logits in id order
        ids[n] = np.argsort(-z[n], kind="stable")[:topk]
    zc = np.take_along_axis(z, ids, axis=1)
    e = np.exp(zc - zc[:, :1])
    return ids, e / e.sum(axis=1, keepdims=True), z, A


def moe(X, ids, route_w, expert, shared=None):
    """Top-k mixture of experts with an optional shared expert.

    X       [N, d] BF16 values (FP64)
    ids     [N, k] routed expert ids (distinct per token)
    route_w [N, k] combine weights
    expert(e) -> (w_gate, w_up, w_down) dequantized FP64 matrices of expert e
    shared       -> the same triple for the shared expert (weight 1), or None

    y_t = shared_mlp(x_t) + sum_k route_w[t, k] * mlp_{ids[t, k]}(x_t),
    each expert MLP evaluated on only the tokens routed to it ([LingMoE] §四
    and §八: only the activated experts' weights are read).
    """
    X = np.atleast_2d(np.asarray(X, dtype=np.float64))
    ids = np.asarray(ids)
    route_w = np.asarray(route_w, dtype=np.float64)
    N, d = X.shape
    Y = np.zeros((N, expert_out_dim(expert, ids, shared)), dtype=np.float64)
    if shared is not None:
        Y += mlp(*shared, X)
    for e in distinct_experts(ids):
        tok, slot = np.nonzero(ids == e)
        y_e = mlp(*expert(int(e)), X[tok])
        Y[tok] += route_w[tok, slot][:, None] * y_e
    return Y


def expert_out_dim(expert, ids, shared):
    if shared is not None:
        return shared[2].shape[0]
    return expert(int(np.asarray(ids).reshape(-1)[0]))[2].shape[0]


def dense_layer(r, layer):
    """One layer of the dense stack on the FP64 residual r [N, d].

    layer: dict with FP64 matrices
      'in'   list of input projections of the token mixer (concatenated)
      'out'  output projection of the token mixer, [d, d_v]
      'gate', 'up', 'down'  the MLP
    """
    a = round_bf16(rmsnorm(r))
    u = np.concatenate([matvec(w, a)[0] for w in layer["in"]], axis=1)
    u = round_bf16(u)
    d_v = layer["out"].shape[1]
    v = u[:, :d_v]                       # stand-in for the weight-free mixer
    r = r + matvec(layer["out"], v)[0]
    m = round_bf16(rmsnorm(r))
    r = r + mlp(layer["gate"], layer["up"], layer["down"], m)
    return r


def moe_layer(r, layer):
    """One layer of the MoE stack: r += FFN(BF16(RMSNorm(r))), the FFN being
    a dense SwiGLU MLP ('gate','up','down') or a MoE ('moe' dict with
    'expert', 'shared', and either 'ids' and 'route_w' given, or 'router'
    (W_r FP64 [E, d]) and 'topk', routed by router_topk on the layer's
    normalised input)."""
    m = round_bf16(rmsnorm(r))
    if "moe" in layer:
        L = layer["moe"]
        if "router" in L:
            ids, route_w, _, _ = router_topk(L["router"], m, L["topk"])
        else:
            ids, route_w = L["ids"], L["route_w"]
        return r + moe(m, ids, route_w, L["expert"], L["shared"])
    return r + mlp(layer["gate"], layer["up"], layer["down"], m)


def head_logits(r, w_head):
    """Output layer on the final residual: logits = W_head BF16(RMSNorm(r))."""
    x = round_bf16(rmsnorm(r))
    return matvec(w_head, x)


def decode_stack(x0, layers, w_head, layer_fn=dense_layer):
    """Whole decode step: residual r = x0, every layer in order, then the
    output layer. Returns (logits [N, V], abs-sum [N, V], final residual)."""
    r = np.atleast_2d(np.asarray(x0, dtype=np.float64)).copy()
    for L in layers:
        r = layer_fn(r, L)
    logits, A = head_logits(r, w_head)
    return logits, A, r
