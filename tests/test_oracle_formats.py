"""Pins for the oracle's codecs and rounding (CPU only)."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from tests.conftest import load_golden, golden_float


def test_e2m1_decode_is_the_pages_grid():
    grid = load_golden("page_figures.json")["e2m1_values"]["value"]
    vals = F.e2m1_decode(np.arange(16))
    assert list(vals[:8]) == grid
    assert list(-vals[8:]) == grid               # sign bit 3
    assert np.signbit(vals[8])                  # code 0x8 is -0


def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.e4m3_decode(np.arange(256))
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.array_equal(both_nan, np.isnan(ref))
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert F.e4m3_decode(0x7E) == 448.0 and F.e4m3_decode(0x01) == 2.0 ** -9
    assert F.e4m3_decode(0x08) == 2.0 ** -6


def test_e8m0_decode():
    assert F.e8m0_decode(127) == 1.0
    assert F.e8m0_decode(0) == 2.0 ** -127
    assert F.e8m0_decode(254) == 2.0 ** 127
    assert np.isnan(F.e8m0_decode(255))


def test_e2m1_ties_worked_by_hand():
    for v, want in load_golden("e2m1_ties.json")["cases"]:
        code = F.e2m1_encode(np.float32(v))
        got = F.e2m1_decode(code)
        w = golden_float(want)
        assert got == w and np.signbit(got) == np.signbit(w), (v, got, w)


def _rne_e2m1_by_rounding(v):
    """Independent E2M1 rounding: within each binade of the grid the points
    are equally spaced, so nearest-even is np.round (half to even) of v over
    the spacing; the grid's mantissa parity equals the integer parity."""
    a = np.abs(v.astype(np.float64))
    spacing = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.round(a / spacing) * spacing
    r = np.minimum(r, 6.0)
    return np.where(np.signbit(v), -r, r)


def test_e2m1_rounding_against_independent_rule():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 0x41000000, size=2_000_000, dtype=np.uint32)
    v = bits.view(np.float32)
    v = np.concatenate([v, -v, np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])])
    # every grid midpoint and its FP32 neighbours
    mids = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])
    near = np.concatenate([np.nextafter(mids, np.float32(0)), mids,
                           np.nextafter(mids, np.float32(10))])
    v = np.concatenate([v, near, -near]).astype(np.float32)
    got = F.e2m1_decode(F.e2m1_encode(v))
    want = _rne_e2m1_by_rounding(v)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_e4m3_rounding_matches_torch_below_overflow():
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 0x43E80000, size=2_000_000, dtype=np.uint32)  # < 464
    v = bits.view(np.float32)
    grid = F.e4m3_decode(np.arange(127))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    near = np.concatenate([np.nextafter(mids, np.float32(0)), mids,
                           np.nextafter(mids, np.float32(1000))])
    v = np.concatenate([v, near]).astype(np.float32)
    v = np.concatenate([v, -v])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(v), ref)


def test_e4m3_saturates():
    v = np.float32([464.0, 480.0, 1e30, -1e30, 448.0, 455.0])
    assert list(F.e4m3_encode(v)) == [0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0x7E]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) < 3.3e38)]
    halfway = ((rng.integers(0, 2 ** 16, 1000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    v = np.concatenate([v, halfway[np.isfinite(halfway)]])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = F.round_bf16(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_ulp():
    assert F.bf16_ulp(1.0) == 2.0 ** -7
    assert F.bf16_ulp(1.5) == 2.0 ** -7
    assert F.bf16_ulp(2.0) == 2.0 ** -6
    assert F.bf16_ulp(0.0) == 2.0 ** -133
    assert F.bf16_ulp(-3.0) == 2.0 ** -6


@pytest.mark.parametrize("bad", ["drop_sign", "ties_up"])
def test_planted_mistakes_are_caught(monkeypatch, bad):
    """A plausible slip in the encoder must fail the independent pins."""
    orig = F._rne_encode

    def broken(v, codes, vals, sign_bit):
        c = orig(v, codes, vals, sign_bit)
        if bad == "drop_sign":
            return c & ~np.uint8(sign_bit)
        a = np.abs(np.asarray(v, np.float64))
        hi = np.searchsorted(vals, a)
        hi = np.clip(hi, 1, len(vals) - 1)
        tie = a == (vals[hi - 1] + vals[hi]) / 2
        return np.where(tie, (codes[hi] | (c & sign_bit)).astype(np.uint8), c)

    monkeypatch.setattr(F, "_rne_encode", broken)
    with pytest.raises(AssertionError):
        test_e2m1_ties_worked_by_hand()
