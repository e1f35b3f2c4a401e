"""When a greedy choice over GPU logits is right.

The GPU's logits g_j meet |g_j - y_j| <= b_j around the oracle's exact logits
y_j (b_j: the product bound). Its choice t (the largest g, lowest index on
ties) is then correct exactly when some set of logits within those bounds
has t on top: y_t + b_t >= y_j - b_j for every other j. When the oracle's top
logit stands clear of the rest (its lower bound above every other upper
bound) that leaves the oracle's argmax as the only acceptable answer; when
the top two are within their bounds of each other, either is."""
import numpy as np


def acceptable(y, b, t):
    """Whether token t is a correct greedy choice for exact logits y with bounds b (1-D)."""
    y = np.asarray(y, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    lower = y - b
    others = np.delete(lower, t)
    return bool(others.size == 0 or y[t] + b[t] >= others.max())
