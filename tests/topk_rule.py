"""When a GPU's top-k expert choice is right.

The GPU's router logits g_e meet |g_e - z_e| <= b_e around the oracle's
exact logits z_e (b_e: the product bound). A chosen set S of k experts is
then correct exactly when some logits within those bounds put S on top:
raise every chosen logit to z_e + b_e and lower every other to z_f - b_f;
S is acceptable when the lowest raised one is still >= the highest lowered
one. Where the oracle's k-th and (k+1)-th logits stand clear of each other
that leaves the oracle's own set as the only acceptable answer.

The combine weights are the softmax of the chosen logits. With each chosen
logit anywhere within its bound, weight i lies in
    [w_i e^{-b_i} / sum_j w_j e^{b_j},  w_i e^{b_i} / sum_j w_j e^{-b_j}]
(w the softmax of the exact logits over the same set), widened here by the
FP32 rounding of the GPU's exp, sum and division."""
import numpy as np


def acceptable_set(z, b, chosen):
    """Whether the expert ids `chosen` (1-D) are a correct top-k for exact
    logits z with bounds b (1-D over the experts)."""
    z = np.asarray(z, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    chosen = np.asarray(chosen)
    if len(set(chosen.tolist())) != chosen.size or chosen.min() < 0 or chosen.max() >= z.size:
        return False
    rest = np.setdiff1d(np.arange(z.size), chosen)
    if rest.size == 0:
        return True
    return bool((z[chosen] + b[chosen]).min() >= (z[rest] - b[rest]).max())


def ordered(z, b, chosen):
    """Whether `chosen` lists the experts largest logit first, up to the bounds."""
    z = np.asarray(z, dtype=np.float64)[np.asarray(chosen)]
    b = np.asarray(b, dtype=np.float64)[np.asarray(chosen)]
    return bool(np.all(z[:-1] + b[:-1] >= z[1:] - b[1:]))


def weight_interval(z, b, chosen, ulps=None):
    """(lo, hi) of each chosen expert's combine weight."""
    zc = np.asarray(z, dtype=np.float64)[np.asarray(chosen)]
    bc = np.asarray(b, dtype=np.float64)[np.asarray(chosen)]
    e = np.exp(zc - zc.max())
    w = e / e.sum()
    lo = w * np.exp(-bc) / np.sum(w * np.exp(bc))
    hi = w * np.exp(bc) / np.sum(w * np.exp(-bc))
    k = zc.size
    r = (4 * k + 16 if ulps is None else ulps) * 2.0 ** -24
    return lo * (1 - r), hi * (1 + r)
