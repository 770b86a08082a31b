"""Pins for the oracle's E4M3 codec (CPU only).

What pins it, independently of its own code:
  * the format facts the pages print (max 448, smallest step 2^-9) from
    tests/golden/e4m3_format.txt;
  * torch's float8_e4m3fn conversions (a library routine) on every code and on
    millions of in-range fp32 values, including every rounding tie;
  * ml_dtypes' float8_e4m3fn where it is installed (a second library);
  * hand-derived boundary cases of the saturating, ties-to-even encoder.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_format.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        name, value, _cite = line.split()
        vals[name] = float(value)
    return vals


def _torch_decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_encode(y: np.ndarray) -> np.ndarray:
    return torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


ALL = np.arange(256, dtype=np.uint8)
NAN_CODES = {0x7F, 0xFF}


def test_decode_all_codes_match_torch():
    mine = oracle.e4m3_value(ALL)
    ref = _torch_decode(ALL)
    for c in range(256):
        if c in NAN_CODES:
            assert np.isnan(mine[c]) and np.isnan(ref[c])
        else:
            assert mine[c] == ref[c], hex(c)
            assert np.signbit(mine[c]) == np.signbit(ref[c]), hex(c)


def test_decode_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    ref = ALL.view(ml.float8_e4m3fn).astype(np.float64)
    mine = oracle.e4m3_value(ALL)
    ok = np.isnan(ref) & np.isnan(mine) | (ref == mine)
    assert ok.all()


def test_format_facts_from_pages():
    g = _golden()
    vals = oracle.e4m3_value(ALL)
    finite = vals[np.isfinite(vals)]
    assert finite.max() == g["max_finite"]
    assert finite.min() == -g["max_finite"]
    assert finite[finite > 0].min() == g["min_nonzero"]
    # 2^(exponent bits) binades x 2^(mantissa bits) steps = 128 magnitudes, minus one NaN
    assert len(set(np.abs(finite))) == 2 ** int(g["exponent_bits"]) * 2 ** int(g["mantissa_bits"]) - 1


def test_round_trip_every_representable_value():
    vals = oracle.e4m3_value(ALL).astype(np.float32)
    codes = oracle.e4m3_encode(vals)
    for c in range(256):
        if c in NAN_CODES:
            assert codes[c] == 0x7F
        else:
            assert codes[c] == c, (hex(c), hex(codes[c]))


@pytest.mark.parametrize("y,code", [
    (448.0, 0x7E), (449.0, 0x7E), (463.99, 0x7E), (464.0, 0x7E), (1e30, 0x7E),
    (float("inf"), 0x7E), (-448.0, 0xFE), (-1e30, 0xFE), (float("-inf"), 0xFE),
    (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (1.5 * 2.0 ** -10, 0x01), (-(2.0 ** -10), 0x80),
    (2.5 * 2.0 ** -9, 0x02), (3.5 * 2.0 ** -9, 0x04), (7.5 * 2.0 ** -9, 0x08),
    (0.0, 0x00), (-0.0, 0x80), (1.0, 0x38), (-1.0, 0xB8),
    (1.0625, 0x38), (1.0625 + 2 ** -20, 0x39), (1.1875, 0x3A), (15.5, 0x58), (14.5, 0x56), (13.5, 0x56),
    (240.0, 0x77), (248.0, 0x78), (432.0, 0x7E), (416.0, 0x7D), (1e-45, 0x00),
])
def test_boundaries(y, code):
    assert int(oracle.e4m3_encode(np.array([y], np.float32))[0]) == code


def test_nan_encodes_to_nan_code():
    y = np.array([np.nan, -np.nan], np.float32)
    assert list(oracle.e4m3_encode(y)) == [0x7F, 0x7F]


def test_every_tie_is_even():
    """Midpoints between neighbouring magnitudes go to the even mantissa."""
    mags = np.sort(np.unique(np.abs(oracle.e4m3_value(ALL[:0x7F]))))
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (mags[:-1] + mags[1:]) / 2)   # exact in fp32
    for sgn in (1.0, -1.0):
        y = (sgn * mids).astype(np.float32)
        mine = oracle.e4m3_encode(y)
        assert np.array_equal(mine, _torch_encode(y))
        assert np.all((mine & 1) == 0)                     # even mantissa


def test_random_in_range_match_torch():
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    y = bits.view(np.float32)
    y = y[np.isfinite(y) & (np.abs(y) <= 448.0)]
    assert y.size > 1_000_000
    assert np.array_equal(oracle.e4m3_encode(y, threads=4), _torch_encode(y))


def test_dense_sweep_small_magnitudes_match_torch():
    """Every 7th fp32 pattern between 2^-12 and 2^-4 (subnormal/normal seam)."""
    lo = np.float32(2.0 ** -12).view(np.uint32)
    hi = np.float32(2.0 ** -4).view(np.uint32)
    bits = np.arange(lo, hi, 7, dtype=np.uint32)
    y = np.concatenate([bits.view(np.float32), -bits.view(np.float32)])
    assert np.array_equal(oracle.e4m3_encode(y, threads=4), _torch_encode(y))


def test_dense_sweep_top_binades_match_torch():
    """Every fp32 pattern in [128, 448] (ties at the top of the range)."""
    lo = np.float32(128.0).view(np.uint32)
    hi = np.float32(448.0).view(np.uint32)
    y = np.arange(lo, hi + 1, dtype=np.uint32).view(np.float32)
    assert np.array_equal(oracle.e4m3_encode(y, threads=4), _torch_encode(y))


def test_random_in_range_match_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(99)
    y = (rng.standard_normal(1 << 20) * rng.choice([1e-3, 1.0, 50.0], 1 << 20)).astype(np.float32)
    y = np.clip(y, -448, 448)
    ref = y.astype(ml.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(y), ref)


def test_saturation_where_torch_gives_nan():
    """torch's cast does not saturate (it returns NaN past 464); the oracle
    saturates every finite or infinite value beyond 448 to +-448."""
    y = np.array([464.0, 500.0, 1e6, 3e38, -470.0], np.float32)
    assert list(oracle.e4m3_encode(y)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
