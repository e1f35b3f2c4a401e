"""Quantizers: NVFP4, MXFP4, row-wise FP8, and MXFP8 activations.

Every rounding decision is taken in FP32 (numpy float32 arithmetic is IEEE
round-to-nearest-even), in the order written below, so that codes can be
compared bit for bit with a kernel that performs the same FP32 operations.
"""
import numpy as np

from .formats import e2m1_encode, e4m3_encode, e4m3_decode

NVFP4_BLOCK = 16
MXFP4_BLOCK = 32
_F32 = np.float32


def pack_nibbles(q):
    """[..., 2k] 4-bit codes -> [..., k] bytes; element 2k in the low nibble."""
    q = np.asarray(q, dtype=np.uint8)
    return (q[..., 0::2] & 0xF) | ((q[..., 1::2] & 0xF) << 4)


def unpack_nibbles(b):
    """[..., k] bytes -> [..., 2k] 4-bit codes (inverse of pack_nibbles)."""
    b = np.asarray(b, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


def nvfp4_tensor_scale(W):
    """Per-tensor FP32 scale s_t = amax/(6*448), so that every block scale
    amax_b/6/s_t lands in E4M3's range ([Spark27B] § "Fewer bytes per
    weight: NVFP4": one 32-bit scale per tensor brings the block scales into
    the range E4M3 can represent). An all-zero tensor, or one whose s_t
    underflows to 0, uses s_t = 1."""
    W = np.asarray(W, dtype=_F32)
    amax = _F32(np.max(np.abs(W))) if W.size else _F32(0.0)
    s_t = _F32(amax / _F32(6.0 * 448.0))
    if not s_t > 0:
        s_t = _F32(1.0)
    return s_t


def nvfp4_quantize(W, s_t=None):
    """NVFP4: E2M1 codes, one E4M3 scale per 16 consecutive weights along
    d_in, one FP32 tensor scale ([Spark27B] § "Fewer bytes per weight:
    NVFP4"; the block scale makes the block's largest magnitude map to 6).

    FP32 sequence per block b (this project's reading; the pages give only
    the two scale levels and that amax maps to 6):
      sb   = fl32(fl32(amax_b / 6) / s_t)
      code = E4M3_rne_satfinite(sb)
      d_b  = fl32(dec(code) * s_t)
      q_j  = E2M1_rne_satfinite(fl32(w_j / d_b))   if d_b > 0, else code 0
    Returns (codes uint8 [d_out, d_in/2], scales uint8 [d_out, d_in/16],
    s_t float32).
    """
    W = np.asarray(W, dtype=_F32)
    d_out, d_in = W.shape
    assert d_in % NVFP4_BLOCK == 0
    if s_t is None:
        s_t = nvfp4_tensor_scale(W)
    s_t = _F32(s_t)
    blk = W.reshape(d_out, d_in // NVFP4_BLOCK, NVFP4_BLOCK)
    amax_b = np.max(np.abs(blk), axis=2).astype(_F32)
    sb = ((amax_b / _F32(6.0)).astype(_F32) / s_t).astype(_F32)
    scale_codes = e4m3_encode(sb)
    d_b = (e4m3_decode(scale_codes).astype(_F32) * s_t).astype(_F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (blk / d_b[..., None]).astype(_F32)
    q = e2m1_encode(ratio)
    q = np.where((d_b > 0)[..., None], q, 0).astype(np.uint8)
    return pack_nibbles(q.reshape(d_out, d_in)), scale_codes, s_t


def floor_log2(a):
    """floor(log2 a) for a > 0, exact for every FP32 value (subnormals
    included), from the binary exponent rather than a logarithm."""
    _, ex = np.frexp(np.asarray(a, dtype=np.float64))
    return ex - 1


def mxfp4_quantize(W):
    """MXFP4: E2M1 codes with one E8M0 (power-of-two) scale per 32 weights
    along d_in. [LingMoE] §十七 only says small blocks share a scale; the
    block size, the scale rule and clipping are read from the OCP MX
    specification:
      e    = clamp(floor(log2 amax_b) - 2, -127, 127)   (2 = E2M1's emax)
      code = e + 127
      q_j  = E2M1_rne_satfinite(w_j * 2^-e)             (exact scaling)
    A block with amax_b = 0 gets scale code 0 and all-zero codes.
    Returns (codes uint8 [rows, d_in/2], scales uint8 [rows, d_in/32])."""
    W = np.asarray(W, dtype=_F32)
    rows, d_in = W.shape
    assert d_in % MXFP4_BLOCK == 0
    blk = W.reshape(rows, d_in // MXFP4_BLOCK, MXFP4_BLOCK).astype(np.float64)
    amax_b = np.max(np.abs(blk), axis=2)
    nz = amax_b > 0
    e = np.where(nz, floor_log2(np.where(nz, amax_b, 1.0)) - 2, -127)
    e = np.clip(e, -127, 127)
    scaled = np.ldexp(blk, -e[..., None])
    q = e2m1_encode(scaled)
    q = np.where(nz[..., None], q, 0).astype(np.uint8)
    return pack_nibbles(q.reshape(rows, d_in)), (e + 127).astype(np.uint8)


MXFP8_BLOCK = 32


def mxfp8_quantize(X):
    """MXFP8 activations for the W4A8 product: E4M3 elements with one E8M0
    (power-of-two) scale per 32 consecutive values along the row. [LingMoE]
    §三 runs the MoE baseline as W4A8 (MXFP4 weights, 8-bit activations) and
    does not give the activation quantizer; it is read, as for MXFP4, from
    the OCP MX specification, with E4M3's largest exponent 8:
      e    = clamp(floor(log2 amax_b) - 8, -127, 127)
      code = e + 127
      q_j  = E4M3_rne_satfinite(x_j * 2^-e)             (exact scaling)
    A block with amax_b = 0 gets scale code 0 and all-zero codes.
    X: [N, d] values (BF16 activations held in any float type).
    Returns (codes uint8 [N, d] E4M3, scales uint8 [N, d/32] E8M0)."""
    X = np.atleast_2d(np.asarray(X, dtype=_F32))
    n, d = X.shape
    assert d % MXFP8_BLOCK == 0
    blk = X.reshape(n, d // MXFP8_BLOCK, MXFP8_BLOCK).astype(np.float64)
    amax_b = np.max(np.abs(blk), axis=2)
    nz = amax_b > 0
    e = np.where(nz, floor_log2(np.where(nz, amax_b, 1.0)) - 8, -127)
    e = np.clip(e, -127, 127)
    scaled = np.ldexp(blk, -e[..., None])
    q = e4m3_encode(scaled.astype(_F32))
    q = np.where(nz[..., None], q, 0).astype(np.uint8)
    return q.reshape(n, d), (e + 127).astype(np.uint8)


def fp8_rowwise_quantize(W):
    """Row-wise FP8 E4M3 with an FP32 scale per row, as used for the output
    layer ([LingMoE] §七: the BF16 head is quantized to FP8 online at load
    time; [Spark27B] § "Decode speed is bytes divided by bandwidth": the
    248,320 x 5,120 output layer read in full every step). Reading:
      s_r  = fl32(amax_r / 448)
      code = E4M3_rne_satfinite(fl32(w / s_r))
    A row whose s_r is 0 gets s_r = 0 and all-zero codes.
    Returns (codes uint8 [rows, cols], row_scale float32 [rows])."""
    W = np.asarray(W, dtype=_F32)
    amax_r = np.max(np.abs(W), axis=1).astype(_F32)
    s_r = (amax_r / _F32(448.0)).astype(_F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (W / s_r[:, None]).astype(_F32)
    codes = e4m3_encode(ratio)
    codes = np.where((s_r > 0)[:, None], codes, 0).astype(np.uint8)
    return codes, s_r
