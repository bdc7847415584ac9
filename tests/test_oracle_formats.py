"""Pins of the oracle's number formats and rounding (CPU only).

Each check compares the oracle with something other than itself: the formats'
published value tables (golden files), PyTorch's own float8/bfloat16
conversions, and exact rational brute force by enumeration."""
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import brute, formats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_e2m1_table_matches_published_grid():
    for code, val in _read_golden("e2m1_grid.txt"):
        got = formats.E2M1_TABLE[int(code)]
        assert got == float(val)
        assert np.signbit(got) == np.signbit(float(val))


def test_e4m3_published_points():
    for hx, val in _read_golden("e4m3_points.txt"):
        got = formats.E4M3_TABLE[int(hx, 16)]
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val) and np.signbit(got) == np.signbit(float(val))


def test_e4m3_all_bytes_match_torch_float8():
    raw = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = formats.E4M3_TABLE
    nan = np.isnan(raw)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(raw[~nan], ours[~nan])
    assert nan.sum() == 2  # 0x7F, 0xFF


def test_rne_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    # dense sweep of float32 values over the whole e4m3 range, plus exact
    # midpoints and their float32 neighbours
    mags = formats.E4M3_TABLE[:0x7F]
    mids = (mags[:-1] + mags[1:]) / 2
    x = np.concatenate([
        rng.uniform(0, 448, 200000),
        np.exp2(rng.uniform(-12, np.log2(448), 200000)),
        mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
        np.nextafter(mids.astype(np.float32), np.float32(0)), mags,
    ]).astype(np.float32)
    x = x[x <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = formats.rne_e4m3(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_rne_e4m3_saturates_and_ties_to_even():
    assert formats.rne_e4m3(np.array([448.0, 464.0, 1e30]))[2] == 0x7E
    assert np.all(formats.rne_e4m3(np.array([448.0, 464.0, 500.0, 1e30])) == 0x7E)
    # tie between 1.0 (0x38, even) and 1.125 (0x39): goes to 1.0
    assert formats.rne_e4m3(np.array([1.0625]))[0] == 0x38
    # tie between 1.125 (0x39) and 1.25 (0x3A): goes to 1.25
    assert formats.rne_e4m3(np.array([1.1875]))[0] == 0x3A
    # half of the smallest subnormal ties to zero; just above it rounds up
    assert formats.rne_e4m3(np.array([2.0 ** -10]))[0] == 0x00
    assert formats.rne_e4m3(np.array([np.nextafter(2.0 ** -10, 1)]))[0] == 0x01


def _brute_pairs(values, kind):
    for v in values:
        fv = Fraction(float(v))
        if kind == "e2m1":
            yield brute.rne_e2m1(fv, np.signbit(v))
        else:
            yield brute.rne_e4m3(fv)


def test_rne_e2m1_against_exact_enumeration():
    grid = formats.E2M1_TABLE[:8]
    mids = (grid[:-1] + grid[1:]) / 2
    pts = np.concatenate([grid, mids, np.nextafter(mids, 0), np.nextafter(mids, 10),
                          [6.0, 6.5, 7.0, 100.0, 1e-30, 0.0]])
    rng = np.random.default_rng(1)
    pts = np.concatenate([pts, rng.uniform(0, 8, 3000)])
    vals = np.concatenate([pts, -pts, [-0.0]])
    got = formats.rne_e2m1(vals)
    want = np.array(list(_brute_pairs(vals, "e2m1")), dtype=np.uint8)
    assert np.array_equal(got, want)


def test_rne_e2m1_worked_ties():
    # ties go to the even code: 0.25->0, 0.75->1, 1.25->1, 1.75->2,
    # 2.5->2, 3.5->4, 5->4; above 6 saturates
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5])
    assert list(formats.e2m1_decode(formats.rne_e2m1(x))) == [0, 1, 1, 2, 2, 4, 4, 6]
    # negative values that round to zero keep the sign bit (code 0x8)
    assert formats.rne_e2m1(np.array([-0.1, -0.0, 0.1])).tolist() == [8, 8, 0]


def test_rne_e4m3_against_exact_enumeration():
    mags = formats.E4M3_TABLE[:0x7F]
    mids = (mags[:-1] + mags[1:]) / 2
    rng = np.random.default_rng(2)
    vals = np.concatenate([mags, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e3),
                           rng.uniform(0, 500, 1500), np.exp2(rng.uniform(-14, 9, 1500))])
    got = formats.rne_e4m3(vals)
    want = np.array(list(_brute_pairs(vals, "e4m3")), dtype=np.uint8)
    assert np.array_equal(got, want)


def test_scale_quotient_float_division_equals_exact_rounding():
    """amax/6 -> e4m3 through one float64 division equals the exact rounding
    of the real quotient, on every float32 value within 64 ulp of each
    6 * (e4m3 midpoint) and on a random sample of float32 values."""
    mags = formats.E4M3_TABLE[:0x7F]
    mids6 = ((mags[:-1] + mags[1:]) / 2 * 6).astype(np.float32)
    bits = mids6.view(np.int32)[:, None] + np.arange(-64, 65, dtype=np.int32)[None, :]
    a = bits.reshape(-1).view(np.float32)
    rng = np.random.default_rng(3)
    a = np.concatenate([a, np.exp2(rng.uniform(-16, 12, 200000)).astype(np.float32)])
    a = a[(a > 0) & np.isfinite(a)].astype(np.float64)
    got = formats.rne_e4m3(a / 6.0)
    # exact: compare a against 6 * midpoints (exact in float64) instead of dividing
    lt = np.searchsorted(mids6.astype(np.float64), a, side="left")
    le = np.searchsorted(mids6.astype(np.float64), a, side="right")
    assert np.array_equal(mids6.astype(np.float64), (mags[:-1] + mags[1:]) / 2 * 6)
    want = np.where(le != lt, np.where(lt % 2 == 0, lt, lt + 1), lt)
    assert np.array_equal(got, want)


def test_round_to_bf16_matches_torch_on_float32():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.uniform(-30, 30, 100000),
                        [0.0, -0.0, 1e-40, 3.4e38]]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = formats.round_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_round_to_bf16_from_float64_by_enumeration():
    """float64 -> bf16 directly: compare with the nearest of the two bf16
    neighbours found by enumeration (exact Fractions, ties to even bits)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(3000) * 10.0 ** rng.uniform(-5, 5, 3000)
    # exact bf16 midpoints and tiny offsets around them (float32 cannot hold these)
    base = (np.float32(1.0) + np.arange(0, 128, dtype=np.float32) / 128).astype(np.float64)
    x = np.concatenate([x, base + 2.0 ** -8, base + 2.0 ** -8 + 2.0 ** -40,
                        base + 2.0 ** -8 - 2.0 ** -40])
    got = formats.round_to_bf16(x)
    for v, g in zip(x, got):
        b32 = struct.unpack("<I", struct.pack("<f", v))[0]
        cands = set()
        for hi in ((b32 >> 16) - 1, b32 >> 16, (b32 >> 16) + 1):
            hi &= 0xFFFF
            c = struct.unpack("<f", struct.pack("<I", hi << 16))[0]
            if np.isfinite(c):
                cands.add((hi, c))
        fv = Fraction(float(v))
        best = min(cands, key=lambda hc: (abs(Fraction(hc[1]) - fv), hc[0] & 1))
        assert g == best[1], (v, g, best)


def test_e2m1_roundtrip_all_codes():
    codes = np.arange(16, dtype=np.uint8)
    vals = formats.e2m1_decode(codes)
    back = formats.rne_e2m1(vals)
    assert np.array_equal(back, codes)


def test_e4m3_roundtrip_all_finite_positive():
    b = np.arange(0x7F, dtype=np.uint8)
    assert np.array_equal(formats.rne_e4m3(formats.e4m3_decode(b)), b)
