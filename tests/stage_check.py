"""Stage-by-stage checks of a decode step against the oracle.

A stack chains a few hundred products, and a BF16 activation the GPU rounds
one way where the FP64 oracle rounds the other is a legitimate difference
that the next stages amplify. So each stage is checked on its own, from the
GPU's own input to that stage as the verification tap recorded it
(bws_decode_step_tap), against the oracle's definition of that stage:

* a normalised input x = BF16(RMSNorm(r)): |x - RMSNorm(r)| <= 1e-4 |RMSNorm(r)|
  + 1/2 ulp (the product bound with the identity for W);
* a product y = W x: |y_gpu - W x| <= 1e-4 sum_j |w_ij x_j| + 1/2 ulp(y);
* a residual update r' = r + W x (FP32 on the GPU): the product bound on
  r' - r plus one FP32 ulp of r' for the addition;
* SwiGLU h = BF16(SiLU(W_g m) * W_u m): the product bounds of g and u carried
  through SiLU(g) * u, plus 1/2 ulp of h;
* an MoE layer: the slot table exactly; each slot's h and outputs as above;
  the combine r' = r + sum_s cw_s y_s from the GPU's slot outputs, within the
  FP32 rounding of that sum.

Weight rows come from a provider: `rows(idx)` returns the oracle's FP64
dequantized rows idx of a matrix, quantized by the oracle itself.
"""
import math

import numpy as np

from oracle import formats as F, model as M, products as P, quant as Q, tolerance as T

REL = T.REL
RMS_EPS = 1e-6


def f64(t):
    t = t.detach()
    if t.dtype.is_floating_point and t.element_size() == 2:
        t = t.float()
    # the MoE slot taps hold rows no token wrote (slots past the count, tokens
    # outside a slot); their bit patterns may be signalling NaNs, which only
    # the checks' masks ever see
    with np.errstate(invalid="ignore"):
        return t.cpu().numpy().astype(np.float64)


def f32_ulp(v):
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.where(a > 0, np.maximum(ex - 1, -126), -126)
    return np.ldexp(1.0, e - 23)


class Report:
    """Worst |err| / bound per stage kind; fails on any ratio above 1."""

    def __init__(self):
        self.worst = {}
        self.count = {}
        self.failures = []

    def add(self, kind, where, ok, worst, at):
        self.count[kind] = self.count.get(kind, 0) + 1
        if worst >= self.worst.get(kind, (0.0, None))[0]:
            self.worst[kind] = (worst, where)
        if not ok:
            self.failures.append((kind, where, worst, at))

    def assert_ok(self, expect=()):
        assert not self.failures, self.failures[:8]
        for kind in expect:
            assert self.count.get(kind, 0) > 0, f"no {kind} check ran"

    def summary(self):
        """kind -> (checks, worst |err| / bound)."""
        return {k: (self.count[k], round(self.worst[k][0], 4) if k in self.worst else None) for k in sorted(self.count)}


def check_norm(rep, where, x_gpu, r_gpu, eps=RMS_EPS):
    e = M.rmsnorm(r_gpu, eps)
    rep.add("rmsnorm", where, *T.check(e, x_gpu, np.abs(e)))


def check_product(rep, kind, where, W_rows, X, Y_gpu):
    """W_rows [R, d_in] FP64; X [N, d_in]; Y_gpu [N, R]."""
    y, A = P.matvec(W_rows, X)
    rep.add(kind, where, *T.check(y, Y_gpu, A))


def check_residual(rep, kind, where, W_rows, X, r_prev, r_next):
    """r_next = r_prev + W x over the rows of W_rows ([N, R] each)."""
    y, A = P.matvec(W_rows, X)
    err = np.abs(r_next - (r_prev + y))
    b = REL * A + 0.5 * F.bf16_ulp(np.abs(y)) + f32_ulp(r_next)
    ratio = err / np.where(b > 0, b, 1.0)
    i = int(np.argmax(ratio)) if ratio.size else 0
    worst = float(ratio.reshape(-1)[i]) if ratio.size else 0.0
    rep.add(kind, where, worst <= 1.0, worst, np.unravel_index(i, ratio.shape) if ratio.size else None)


def check_swiglu(rep, where, Wg_rows, Wu_rows, X, H_gpu):
    """H_gpu [N, R] = BF16(SiLU(Wg x) * Wu x) over the rows of Wg_rows / Wu_rows."""
    g, Ag = P.matvec(Wg_rows, X)
    u, Au = P.matvec(Wu_rows, X)
    h = M.silu(g) * u
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = np.abs(sig * (1.0 + g * (1.0 - sig)))
    tg, tu = REL * Ag, REL * Au
    extra = dsilu * np.abs(u) * tg + np.abs(M.silu(g)) * tu + 1.1 * tg * tu + 1e-6 * np.abs(h)
    rep.add("swiglu", where, *T.check(h, H_gpu, np.zeros_like(h), extra=extra))


def check_combine(rep, where, r_prev, r_next, cw, ys, live):
    """r_next[t] = r_prev[t] + sum over live slots s (in order) of cw[s, t] ys[s, t]
    (FP32 on the GPU: one rounding per fused multiply-add and one for the sum)."""
    acc = np.zeros_like(r_prev)
    mag = np.zeros_like(r_prev)
    for s in range(live):
        acc += cw[s][:, None] * ys[s]
        mag += np.abs(cw[s][:, None] * ys[s])
    err = np.abs(r_next - (r_prev + acc))
    b = (live + 2) * 2.0 ** -24 * mag + f32_ulp(r_next) + f32_ulp(acc)
    ratio = err / np.where(b > 0, b, 1.0)
    i = int(np.argmax(ratio))
    rep.add("combine", where, float(ratio.reshape(-1)[i]) <= 1.0, float(ratio.reshape(-1)[i]),
            np.unravel_index(i, ratio.shape))


def check_slot_table(rep, where, ids, route_w, has_shared, n_slots, slot_expert, cw):
    """The slot table the routing must build: the shared expert first, then the
    distinct routed experts in ascending id order; cw[s, t] the token's
    weight for the slot's expert (1 for the shared one, 0 if unused)."""
    ids = np.asarray(ids)
    want = ([-1] if has_shared else []) + sorted(set(ids.reshape(-1).tolist()))
    ok = n_slots == len(want) and list(slot_expert[:n_slots]) == want
    N = ids.shape[0]
    for s, e in enumerate(want[:n_slots] if ok else []):
        for t in range(N):
            w = 1.0 if e == -1 else float(np.sum(np.where(ids[t] == e, route_w[t], 0.0)))
            ok = ok and np.float32(cw[s, t]) == np.float32(w)
    rep.add("slot_table", where, ok, 0.0 if ok else math.inf, None)


def check_router(rep, where, W_r, X, z_gpu, ids_gpu, rw_gpu):
    """The router stage: logits z = W_r x at the product bound over every
    expert; each token's chosen experts an acceptable top-k for the exact
    logits within those bounds, listed largest first; their weights within
    the softmax's interval for logits anywhere in their bounds
    (tests/topk_rule.py). Also counts the tokens whose set is the oracle's
    own top-k exactly."""
    from topk_rule import acceptable_set, ordered, weight_interval
    z, A = P.matvec(W_r, X)
    rep.add("router", where, *T.check(z, z_gpu, A))
    b = T.bound(z, z_gpu, A)
    k = ids_gpu.shape[1]
    ok, worst = True, 0.0
    for n in range(z.shape[0]):
        ids = np.asarray(ids_gpu[n], dtype=np.int64)
        if not (acceptable_set(z[n], b[n], ids) and ordered(z[n], b[n], ids)):
            ok, worst = False, math.inf
            continue
        lo, hi = weight_interval(z[n], b[n], ids)
        mid, half = (lo + hi) / 2, (hi - lo) / 2
        r = float(np.max(np.abs(rw_gpu[n] - mid) / half))
        worst = max(worst, r)
        ok = ok and r <= 1.0
        own = set(np.argsort(-z[n], kind="stable")[:k].tolist())
        rep.count["router_oracle_set"] = rep.count.get("router_oracle_set", 0) + (own == set(ids.tolist()))
    rep.add("router_topk", where, ok, worst, None)


def sample_rows(n, k, seed):
    """Rows to check of an n-row output: the first and last two and k others."""
    if n <= k + 4:
        return np.arange(n)
    rng = np.random.default_rng(seed)
    pick = set([0, 1, n - 2, n - 1]) | set(rng.choice(n, size=k, replace=False).tolist())
    return np.array(sorted(pick))


def check_dense_stack(rep, stack, recs, logits, x0, rows_of, k_rows=None, seed=0):
    """All stages of a dense stack's step from its tap records.

    rows_of(layer, name) -> provider (idx -> FP64 rows) of a matrix, name in
    mixer_in (the concatenated input projections), mixer_out, gate, up, down,
    head (layer None). k_rows: rows sampled per product (None: every row)."""
    it = iter(recs)

    def nxt(kind):
        k, t = next(it)
        assert k == kind, (k, kind)
        return t

    def pick(n, salt):
        return np.arange(n) if k_rows is None else sample_rows(n, k_rows, seed * 100003 + salt)

    r_prev = None
    for li, L in enumerate(stack.layers_py):
        assert L["kind"] in ("mixer_mlp", "mlp")
        if L["kind"] == "mixer_mlp":
            a, r_a, v = f64(nxt("a")), f64(nxt("r")), f64(nxt("v"))
            if r_prev is None:
                assert np.array_equal(r_a, F.round_bf16(f64(x0))), "r must start as x0"
            else:
                _check_down(rep, li - 1, stack, rows_of, r_prev, h_prev, r_a, pick)
            check_norm(rep, (li, "a"), a, r_a)
            dv = v.shape[1]
            rows = pick(dv, 10 * li + 1)
            check_product(rep, "mixer_in", (li,), rows_of(li, "mixer_in")(rows), a, v[:, rows])
            r_in = r_a
            m, r_m, h = f64(nxt("m")), f64(nxt("r")), f64(nxt("h"))
            rows = pick(stack.hidden, 10 * li + 2)
            check_residual(rep, "mixer_out", (li,), rows_of(li, "mixer_out")(rows), v, r_in[:, rows], r_m[:, rows])
        else:
            m, r_m, h = f64(nxt("m")), f64(nxt("r")), f64(nxt("h"))
            if r_prev is not None:
                _check_down(rep, li - 1, stack, rows_of, r_prev, h_prev, r_m, pick)
        check_norm(rep, (li, "m"), m, r_m)
        rows = pick(h.shape[1], 10 * li + 3)
        check_swiglu(rep, (li,), rows_of(li, "gate")(rows), rows_of(li, "up")(rows), m, h[:, rows])
        r_prev, h_prev = r_m, h
    xh, r_f = f64(nxt("x_head")), f64(nxt("r"))
    if r_prev is not None:
        _check_down(rep, len(stack.layers_py) - 1, stack, rows_of, r_prev, h_prev, r_f, pick)
    check_norm(rep, ("head", "x"), xh, r_f)
    V = logits.shape[1]
    rows = pick(V, 7)
    check_product(rep, "head", ("head",), rows_of(None, "head")(rows), xh, f64(logits)[:, rows])


def _check_down(rep, li, stack, rows_of, r_m, h, r_next, pick):
    rows = pick(stack.hidden, 10 * li + 4)
    check_residual(rep, "down", (li,), rows_of(li, "down")(rows), h, r_m[:, rows], r_next[:, rows])


def check_moe_stack(rep, stack, recs, logits, x0, rows_of, expert_rows, k_rows=None, seed=0):
    """All stages of an MoE stack (dense MLP layers, then MoE layers).

    expert_rows(layer, e, name) -> provider of expert e's (-1: shared) gate,
    up or down rows. A layer with a router is checked at the router stage
    (check_router), then from the ids and weights the GPU chose."""
    it = iter(recs)

    def nxt(kind):
        k, t = next(it)
        assert k == kind, (k, kind)
        return t

    def pick(n, salt):
        return np.arange(n) if k_rows is None else sample_rows(n, k_rows, seed * 100003 + salt)

    pend = None   # the previous layer's update, checked against the r the next prep normalised
    for li, L in enumerate(stack.layers_py):
        m, r_m = f64(nxt("m")), f64(nxt("r"))
        if pend is None:
            assert np.array_equal(r_m, F.round_bf16(f64(x0))), "r must start as x0"
        else:
            pend(r_m)
        check_norm(rep, (li, "m"), m, r_m)
        if L["kind"] == "mlp":
            h = f64(nxt("h"))
            rows = pick(h.shape[1], 10 * li + 3)
            check_swiglu(rep, (li,), rows_of(li, "gate")(rows), rows_of(li, "up")(rows), m, h[:, rows])

            def pend(r_next, li=li, r_m=r_m, h=h):
                rows = pick(stack.hidden, 10 * li + 4)
                check_residual(rep, "down", (li,), rows_of(li, "down")(rows), h, r_m[:, rows], r_next[:, rows])
            continue
        if L.get("router") is not None:
            z_g = f64(nxt("z"))
            ids, rw = nxt("ids").cpu().numpy(), nxt("route_w").cpu().numpy()
            check_router(rep, (li,), f64(L["router"]), m, z_g, ids, rw.astype(np.float64))
        else:
            ids, rw = L["ids_host"].numpy(), L["route_w_host"].numpy()
        n_slots = int(nxt("n_slots").item())
        slot_expert = nxt("slot_expert").cpu().numpy()
        cw = nxt("cw").cpu().numpy().astype(np.float64)
        hs, ys = f64(nxt("h_slots")), f64(nxt("y_slots"))
        w = L["moe"]
        check_slot_table(rep, (li,), ids, rw, w.shared is not None, n_slots, slot_expert, cw)
        for s in range(n_slots):
            e = int(slot_expert[s])
            toks = np.nonzero(cw[s] != 0)[0]
            if toks.size == 0:
                continue
            rows = pick(w.inter, 1000 * li + s)
            check_swiglu(rep, (li, "slot", s), expert_rows(li, e, "gate")(rows), expert_rows(li, e, "up")(rows),
                         m[toks], hs[s][toks][:, rows])
            rows = pick(stack.hidden, 1000 * li + 500 + s)
            check_product(rep, "expert_down", (li, "slot", s), expert_rows(li, e, "down")(rows), hs[s][toks],
                          ys[s][toks][:, rows])

        def pend(r_next, li=li, r_m=r_m, cw=cw, ys=ys, n_slots=n_slots):
            check_combine(rep, (li,), r_m, r_next, cw, ys, n_slots)
    xh, r_f = f64(nxt("x_head")), f64(nxt("r"))
    if pend is not None:
        pend(r_f)
    check_norm(rep, ("head", "x"), xh, r_f)
    rows = pick(logits.shape[1], 7)
    check_product(rep, "head", ("head",), rows_of(None, "head")(rows), xh, f64(logits)[:, rows])


# ---- weight-row providers -----------------------------------------------------

def dequant_rows(qm, rows):
    """Oracle dequantization of rows of a device QMatrix (its codes taken as
    they are: for stacks whose codes the oracle itself wrote)."""
    c = qm.codes[rows].cpu().numpy()
    if qm.fmt == 1:
        return P.nvfp4_dequantize(c, qm.scales[rows].cpu().numpy(), np.float32(qm.scale32.item()))
    if qm.fmt == 2:
        return P.mxfp4_dequantize(c, qm.scales[rows].cpu().numpy())
    return P.fp8_dequantize(c, qm.scale32[rows].cpu().numpy())


def concat_provider(providers, d_outs):
    """Rows of the concatenation of several matrices (the mixer inputs)."""
    offs = np.cumsum([0] + list(d_outs))

    def rows(idx):
        idx = np.asarray(idx)
        which = np.searchsorted(offs, idx, side="right") - 1
        out = None
        for k in np.unique(which):
            sel = np.nonzero(which == k)[0]
            r = providers[int(k)](idx[sel] - offs[k])
            if out is None:
                out = np.zeros((len(idx), r.shape[1]))
            out[sel] = r
        return out
    return rows
