"""Pins for the oracle's quantizers (CPU only)."""
import numpy as np
import pytest

from oracle import formats as F
from oracle import quant as Q
from oracle import products as P
from tests.conftest import load_golden, golden_float
import synth


def _golden_W(name, key="W"):
    g = load_golden(name)
    W = np.array([[golden_float(v) for v in row] for row in g[key]], dtype=np.float32)
    return g, W


def test_nvfp4_hand_example():
    g, W = _golden_W("nvfp4_hand.json")
    codes, scales, s_t = Q.nvfp4_quantize(W)
    assert s_t == np.float32(g["s_t"])
    assert codes.tolist() == g["codes"]
    assert scales.tolist() == g["scales"]
    w_hat = P.nvfp4_dequantize(codes, scales, s_t)
    assert list(w_hat[1]) == g["w_hat_row1"]


def _bits_f32(h):
    return np.array([int(h, 16)], dtype=np.uint32).view(np.float32)[0]


def test_nvfp4_hand_example_non_power_of_two_tensor_scale():
    """A tensor scale of 29/28 in FP32: the example's scale codes and element
    codes depend on the order of the FP32 scale arithmetic (worked by hand in
    nvfp4_hand_st.json), so a reordered division fails here."""
    g = load_golden("nvfp4_hand_st.json")
    W = np.zeros(g["shape"], dtype=np.float32)
    for e in g["nonzero"]:
        v = _bits_f32(e["bits"])
        assert v == np.float32(float(e["w"]))
        W[e["at"][0], e["at"][1]] = v
    codes, scales, s_t = Q.nvfp4_quantize(W)
    assert np.float32(s_t).view(np.uint32) == int(g["s_t_bits"], 16)
    assert scales.tolist() == g["scales"]
    q = np.zeros(g["shape"], dtype=np.uint8)
    for e in g["codes_nonzero"]:
        q[e["at"][0], e["at"][1]] = e["code"]
    assert codes.tolist() == Q.pack_nibbles(q).tolist()


def test_mxfp4_hand_example():
    g, W = _golden_W("mxfp4_hand.json")
    codes, scales = Q.mxfp4_quantize(W)
    assert scales.tolist() == g["scales"]
    assert codes.tolist() == g["codes"]


def test_mxfp8_hand_example():
    # five rows worked by hand: ordinary values, ties to the even mantissa, a
    # subnormal, signed zero, saturation at 448, an all-zero block, a large
    # exponent and the scale's clamp at 2^-127
    g, X = _golden_W("mxfp8_hand.json", "X")
    codes, scales = Q.mxfp8_quantize(X)
    assert scales.tolist() == g["scales"]
    assert codes.tolist() == g["codes"]


def test_mxfp8_invariants():
    X = synth.weight_fp32((16, 512), seed=3, index=1, std=1.0).numpy()
    X[2, :32] = 0.0
    X[4, 32:64] *= 1e-30
    codes, scales = Q.mxfp8_quantize(X)
    x_hat = P.mxfp8_dequantize(codes, scales)
    blk = np.abs(X.astype(np.float64)).reshape(16, 16, 32)
    amax = blk.max(axis=2)
    X_scale = F.e8m0_decode(scales)
    nz = amax > 0
    # the block's largest value lands in [256, 448] after scaling (448 when it saturates)
    top = np.abs(x_hat).reshape(16, 16, 32).max(axis=2)
    assert np.all(top[nz] / X_scale[nz] >= 256) and np.all(top[nz] / X_scale[nz] <= 448)
    assert np.all(scales[~nz] == 0) and np.all(x_hat.reshape(16, 16, 32)[~nz] == 0)
    # every value within half an E4M3 step of its block: 2^-4 relative for
    # normals, half the subnormal step 2^-10 X below them; saturated ones
    # lose at most (512 - 448) / 512 of the block maximum
    err = np.abs(x_hat - X.astype(np.float64)).reshape(16, 16, 32)
    bound = np.maximum(2.0 ** -4 * blk, 2.0 ** -10 * X_scale[..., None]) + (blk * X_scale[..., None] ** -1 > 448) * blk
    assert np.all(err <= bound)
    # quantizing the dequantized values again changes nothing
    c2, s2 = Q.mxfp8_quantize(x_hat.astype(np.float32))
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)


def test_mxfp8_exact_round_trip():
    # values that are E4M3 numbers times the block's power of two come back exactly
    rng = np.random.default_rng(0)
    vals = F.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    vals = vals[vals >= 2.0 ** -6]
    x = rng.choice(vals, size=(3, 64)) * rng.choice([-1.0, 1.0], size=(3, 64))
    x[:, 0] = 448.0   # fixes the block exponent at 0 (floor(log2 448) - 8 = 0)
    x[:, 32] = -448.0
    codes, scales = Q.mxfp8_quantize(x.astype(np.float32))
    assert np.all(scales == 127)
    assert np.array_equal(P.mxfp8_dequantize(codes, scales), x)


def test_fp8_hand_example():
    g, W = _golden_W("fp8_hand.json")
    codes, s_r = Q.fp8_rowwise_quantize(W)
    assert s_r.tolist() == g["row_scale"]
    assert codes.tolist() == g["codes"]


@pytest.fixture(scope="module")
def W_rand():
    W = synth.weight_fp32((96, 512), seed=7, index=0).numpy()
    W[3, :16] = 0.0                            # an all-zero block
    W[5, 16:32] *= 1e-6                        # a block far below the others
    W[7, 40] = 0.5                             # an outlier
    return W


def test_nvfp4_invariants(W_rand):
    codes, scales, s_t = Q.nvfp4_quantize(W_rand)
    assert codes.shape == (96, 256) and scales.shape == (96, 32)
    q = F.e2m1_decode(Q.unpack_nibbles(codes)).reshape(96, 32, 16)
    sb = F.e4m3_decode(scales)
    amax_b = np.abs(W_rand.reshape(96, 32, 16)).max(axis=2)
    normal = (scales & 0x78) != 0
    # the largest weight of every block with a normal scale maps to |q| = 6
    assert np.all(np.abs(q).max(axis=2)[normal & (amax_b > 0)] == 6.0)
    assert np.nanmax(sb) <= 448.0
    # the block holding the tensor amax gets the top of E4M3's range
    r, c = np.unravel_index(np.argmax(np.abs(W_rand)), W_rand.shape)
    assert sb[r, c // 16] >= 416.0
    # zero block -> zero scale code and zero codes
    assert scales[3, 0] == 0 and np.all(q[3, 0] == 0)
    # |w - w_hat| <= d_b for blocks with a normal scale
    w_hat = P.nvfp4_dequantize(codes, scales, s_t).reshape(96, 32, 16)
    d_b = (sb.astype(np.float32) * s_t).astype(np.float64)
    err = np.abs(W_rand.reshape(96, 32, 16) - w_hat)
    assert np.all(err[normal] <= d_b[normal][:, None])
    # byte count: 4 + 8/16 bits per weight
    assert codes.nbytes + scales.nbytes == 96 * 512 * 4.5 / 8


def test_nvfp4_requantize_is_identity(W_rand):
    codes, scales, s_t = Q.nvfp4_quantize(W_rand)
    w_hat = P.nvfp4_dequantize(codes, scales, s_t).astype(np.float32)
    # re-encode w_hat under the same scales: w_hat / d_b is the grid value
    d_b = (F.e4m3_decode(scales).astype(np.float32) * s_t).astype(np.float32)
    live = d_b > 0                                   # zero blocks: scale 0, codes 0
    ratio = (w_hat.reshape(96, 32, 16) / np.where(live, d_b, 1)[..., None]).astype(np.float32)
    q2 = np.where(live[..., None], F.e2m1_encode(ratio), 0)
    q1 = Q.unpack_nibbles(codes).reshape(96, 32, 16)
    same = (q1 & 7) == (q2 & 7)
    assert np.all(same)


def test_nvfp4_outlier_only_coarsens_its_block():
    W = synth.weight_fp32((1, 64), seed=3).numpy()
    c0, s0, t0 = Q.nvfp4_quantize(W, s_t=np.float32(1.0 / 2688))
    W2 = W.copy()
    W2[0, 5] = 50 * np.abs(W).max()
    c1, s1, t1 = Q.nvfp4_quantize(W2, s_t=np.float32(1.0 / 2688))
    assert np.array_equal(s0[0, 1:], s1[0, 1:])
    assert np.array_equal(c0[0, 8:], c1[0, 8:])


def test_nvfp4_zero_tensor():
    codes, scales, s_t = Q.nvfp4_quantize(np.zeros((4, 32), np.float32))
    assert s_t == 1.0 and not codes.any() and not scales.any()


def test_mxfp4_grid_roundtrip():
    rng = np.random.default_rng(5)
    grid = F.e2m1_decode(np.arange(16))
    for k in (-20, -3, 0, 7, 100):
        vals = rng.choice(grid, size=(4, 64)).astype(np.float64)
        vals[:, ::32] = 6.0                    # pin amax = 6*2^k
        W = np.ldexp(vals, k).astype(np.float32)
        codes, scales = Q.mxfp4_quantize(W)
        assert np.all(scales == 127 + k)
        assert np.array_equal(P.mxfp4_dequantize(codes, scales), W.astype(np.float64))


def test_mxfp4_scale_rule(W_rand):
    codes, scales = Q.mxfp4_quantize(W_rand)
    amax = np.abs(W_rand.reshape(96, 16, 32)).max(axis=2)
    e = scales.astype(np.int64) - 127
    nz = amax > 0
    # 2^(e+2) <= amax < 2^(e+3): the block amax lands in [4, 8) before clipping
    assert np.all(np.ldexp(1.0, e[nz] + 2) <= amax[nz])
    assert np.all(amax[nz] < np.ldexp(1.0, e[nz] + 3))
    w_hat = P.mxfp4_dequantize(codes, scales)
    assert np.all(np.abs(w_hat) <= np.ldexp(6.0, e).repeat(32, axis=1) + 0)


def test_fp8_row_max_encodes_near_448(W_rand):
    codes, s_r = Q.fp8_rowwise_quantize(W_rand)
    W = W_rand
    for i in range(W.shape[0]):
        j = np.argmax(np.abs(W[i]))
        c = codes[i, j] & 0x7F
        # 0x7E unless fl32 rounding of s_r pushes amax/s_r just above 448
        assert c == 0x7E
    w_hat = P.fp8_dequantize(codes, s_r)
    rel = np.abs(W - w_hat) / np.maximum(np.abs(W), 1e-30)
    normal = np.abs(W) >= (2.0 ** -6) * s_r[:, None]
    assert np.all(rel[normal] <= 2.0 ** -4 + 1e-7)


def _nvfp4_reordered(scale_order, elem_order):
    """The oracle's NVFP4 quantizer with one step of its FP32 sequence done
    in another order (a planted mistake)."""
    from oracle.formats import e2m1_encode, e4m3_encode, e4m3_decode
    f32 = np.float32

    def quant(W, s_t=None):
        W = np.asarray(W, dtype=f32)
        d_out, d_in = W.shape
        s_t = Q.nvfp4_tensor_scale(W) if s_t is None else f32(s_t)
        blk = W.reshape(d_out, d_in // 16, 16)
        amax_b = np.max(np.abs(blk), axis=2).astype(f32)
        if scale_order:
            sb = (amax_b / f32(f32(6.0) * s_t)).astype(f32)
        else:
            sb = ((amax_b / f32(6.0)).astype(f32) / s_t).astype(f32)
        sc = e4m3_encode(sb)
        dec = e4m3_decode(sc).astype(f32)
        with np.errstate(divide="ignore", invalid="ignore"):
            if elem_order:
                ratio = ((blk / s_t).astype(f32) / dec[..., None]).astype(f32)
            else:
                ratio = (blk / (dec * s_t).astype(f32)[..., None]).astype(f32)
        q = np.where((dec > 0)[..., None], e2m1_encode(ratio), 0).astype(np.uint8)
        return Q.pack_nibbles(q.reshape(d_out, d_in)), sc, s_t
    return quant


@pytest.mark.parametrize("scale_order,elem_order", [(True, False), (False, True)])
def test_reordered_scale_arithmetic_fails_the_hand_example(monkeypatch, scale_order, elem_order):
    monkeypatch.setattr(Q, "nvfp4_quantize", _nvfp4_reordered(scale_order, elem_order))
    with pytest.raises(AssertionError):
        test_nvfp4_hand_example_non_power_of_two_tensor_scale()


def test_reorder_helper_matches_the_oracle_when_not_reordered():
    W = synth.weight_fp32((8, 64), seed=3, index=0).numpy()
    a = Q.nvfp4_quantize(W)
    b = _nvfp4_reordered(False, False)(W)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]


@pytest.mark.parametrize("bad", ["emax7", "no_clamp", "ceil_log2", "no_saturation"])
def test_mxfp8_planted_mistakes_fail_the_hand_rows(monkeypatch, bad):
    """Plausible slips in the MXFP8 rule must fail the hand-worked rows."""
    def broken(X):
        X = np.atleast_2d(np.asarray(X, dtype=np.float32))
        n, d = X.shape
        blk = X.reshape(n, d // 32, 32).astype(np.float64)
        amax = np.max(np.abs(blk), axis=2)
        nz = amax > 0
        fl = Q.floor_log2(np.where(nz, amax, 1.0))
        if bad == "ceil_log2":
            fl = np.ceil(np.log2(np.where(nz, amax, 1.0))).astype(np.int64)
        e = np.where(nz, fl - (7 if bad == "emax7" else 8), -127)
        if bad != "no_clamp":
            e = np.clip(e, -127, 127)
        scaled = np.ldexp(blk, -e[..., None]).astype(np.float32)
        q = F.e4m3_encode(scaled)
        if bad == "no_saturation":   # wraps past 448 into the NaN pattern
            q = np.where(np.abs(scaled) > 448, (q & 0x80) | 0x7F, q)
        q = np.where(nz[..., None], q, 0).astype(np.uint8)
        return q.reshape(n, d), (e + 127).astype(np.uint8)

    monkeypatch.setattr(Q, "mxfp8_quantize", broken)
    with pytest.raises(AssertionError):
        test_mxfp8_hand_example()
