"""Number formats of the weight stream.

[Spark27B] § "Fewer bytes per weight: NVFP4": an E2M1 element (1 sign,
2 exponent, 1 mantissa bit) holds only 0, ±0.5, ±1, ±1.5, ±2, ±3, ±4, ±6;
block scales are 8-bit E4M3. The exact bit layouts are not printed on the
pages; the readings used here are the OCP FP8 / MX
definitions: E2M1 bias 1 with the e=0 code meaning 0.5*m, E4M3 bias 7 with
no infinities (S.1111.111 is NaN, max 448), E8M0 = 2^(e-127) with 0xFF NaN.

Encoders round to nearest, ties to the even code (mantissa LSB 0), and
saturate to the largest finite value; a negative input that rounds to zero
keeps its sign bit.
"""
import numpy as np

E2M1_MAX = 6.0
E4M3_MAX = 448.0


def e2m1_decode(codes):
    """4-bit codes (low nibble used) -> float64 values."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return np.where(s == 1, -mag, mag)


def e4m3_decode(codes):
    """8-bit E4M3 codes -> float64 values (NaN for S.1111.111)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m.astype(np.float64), -9),
                   np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e8m0_decode(codes):
    """8-bit E8M0 scale codes -> float64 2^(code-127) (NaN for 0xFF)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    v = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, v)


def _positive_grid(decode, n_codes):
    codes = np.arange(n_codes, dtype=np.int64)
    vals = decode(codes)
    return codes, vals


_E2M1_CODES, _E2M1_VALS = _positive_grid(e2m1_decode, 8)       # codes 0..7
_E4M3_CODES, _E4M3_VALS = _positive_grid(e4m3_decode, 127)     # codes 0..126


def _rne_encode(v, grid_codes, grid_vals, sign_bit):
    """Nearest grid point to |v| (ties to even code), saturating, sign kept.

    All comparisons are exact: |v| (an FP32 value held in FP64) is compared
    with the midpoint of its two neighbouring grid values, which is exactly
    representable in FP64.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    top = grid_vals[-1]
    hi_idx = np.searchsorted(grid_vals, a, side="left")      # first >= a
    hi_idx = np.clip(hi_idx, 1, len(grid_vals) - 1)
    lo_idx = hi_idx - 1
    lo = grid_vals[lo_idx]
    hi = grid_vals[hi_idx]
    mid = (lo + hi) / 2.0
    lo_c = grid_codes[lo_idx]
    hi_c = grid_codes[hi_idx]
    even_c = np.where((lo_c & 1) == 0, lo_c, hi_c)
    code = np.where(a < mid, lo_c, np.where(a > mid, hi_c, even_c))
    code = np.where(a >= top, grid_codes[-1], code)           # satfinite
    code = np.where(a <= grid_vals[0], grid_codes[0], code)   # exact zero
    neg = np.signbit(v)
    return (code | np.where(neg, sign_bit, 0)).astype(np.uint8)


def e2m1_encode(v):
    """FP32 values -> 4-bit E2M1 codes (uint8, low nibble), RNE, satfinite."""
    return _rne_encode(v, _E2M1_CODES, _E2M1_VALS, 0x8)


def e4m3_encode(v):
    """FP32 values -> E4M3 codes (uint8), RNE, satfinite (never NaN)."""
    return _rne_encode(v, _E4M3_CODES, _E4M3_VALS, 0x80)


def round_bf16(v):
    """Round float64 values to the nearest BF16 value (ties to even).

    BF16 keeps 8 significant bits; below 2^-126 the spacing stays 2^-133
    (subnormals). Magnitudes that round past the largest finite BF16 become
    infinite. Returned as float64.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex - 1, -126)
    ulp = np.ldexp(1.0, e - 7)
    r = np.round(v / ulp) * ulp
    r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, v), r)
    return np.where(np.isfinite(v), r, v)


def bf16_ulp(v):
    """Spacing of BF16 values at |v| (the ulp used by the tolerance)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.where(a > 0, np.maximum(ex - 1, -126), -126)
    return np.ldexp(1.0, e - 7)


def bf16_bits_to_float(bits):
    """uint16 BF16 bit patterns -> float64 values."""
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def float_to_bf16_bits(v):
    """float64 values that are exactly BF16-representable -> uint16 bits."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)
