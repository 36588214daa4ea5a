"""Pins of the oracle's E4M3 and bfloat16 conversions (CPU only).

Pinned against: hand-worked values of the format (tests/golden), PyTorch's
float8_e4m3fn and bfloat16 conversions (library special cases), and an
independent exhaustive nearest-value search over binary32 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden


def _f32(s):
    return np.float32(float(s))


def test_encode_golden_boundaries():
    rows = read_golden("e4m3_encode_boundaries.txt")
    assert len(rows) >= 20
    xs = np.array([_f32(r[0]) for r in rows], np.float32)
    want = np.array([int(r[1], 16) for r in rows], np.uint8)
    got = oracle.e4m3_encode(xs)
    bad = [(rows[i][0], hex(got[i]), rows[i][1]) for i in np.nonzero(got != want)[0]]
    assert not bad, bad


def test_decode_golden_values():
    rows = read_golden("e4m3_decode_values.txt")
    codes = np.array([int(r[0], 16) for r in rows], np.uint8)
    want = np.array([float(r[1]) for r in rows])
    got = oracle.e4m3_decode(codes)
    nan = np.isnan(want)
    assert (np.isnan(got) == nan).all()
    np.testing.assert_array_equal(got[~nan], want[~nan])
    np.testing.assert_array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and (np.isnan(got) == nan).all()
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    np.testing.assert_array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _torch_encode(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(1)
    # wide log-uniform magnitudes, both signs, within the range torch rounds
    # (torch's conversion does not saturate beyond 464)
    mag = np.exp2(rng.uniform(-14, np.log2(463.0), 2_000_000)).astype(np.float32)
    x = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    # every representable value, every midpoint, and their binary32 neighbours
    vals = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids]).astype(np.float32)
    nb = np.concatenate([pts, np.nextafter(pts, np.float32(0)), np.nextafter(pts, np.float32(1e9))])
    x = np.concatenate([x, nb, -nb]).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(x), _torch_encode(x))


@pytest.mark.slow
def test_encode_exhaustive_vs_nearest_value_search():
    """Every positive binary32 in [2^-11, 2^9) and a stride of the rest.

    Independent definition: the code is the index of the nearest of the 127
    non-negative finite E4M3 values (they are increasing in the code), ties to
    the even code, saturating at 448.
    """
    vals = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()
    assert np.all(np.diff(vals) > 0)

    def nearest(x64):
        idx = np.clip(np.searchsorted(vals, x64), 1, len(vals) - 1)
        lo, hi = idx - 1, idx
        dlo, dhi = x64 - vals[lo], vals[hi] - x64
        pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
        pick = np.where(x64 >= vals[-1], len(vals) - 1, pick)
        return pick.astype(np.uint8)

    lo_bits = np.float32(2.0 ** -11).view(np.uint32)
    hi_bits = np.float32(2.0 ** 9).view(np.uint32)
    chunk = 1 << 24
    for start in range(int(lo_bits), int(hi_bits), chunk):
        bits = np.arange(start, min(start + chunk, int(hi_bits)), dtype=np.uint32)
        x = bits.view(np.float32)
        got = oracle.e4m3_encode(x)
        want = nearest(x.astype(np.float64))
        if not np.array_equal(got, want):
            i = np.nonzero(got != want)[0][0]
            pytest.fail("x=%r got %#x want %#x" % (x[i], got[i], want[i]))
        if start % (8 * chunk) == 0:  # sign symmetry on a subset
            np.testing.assert_array_equal(oracle.e4m3_encode(-x[::97]), got[::97] | 0x80)
    # everything below 2^-11 encodes to zero, everything at/after 448 saturates
    tiny = np.arange(1, int(lo_bits), 4099, dtype=np.uint32).view(np.float32)
    assert (oracle.e4m3_encode(tiny) == 0).all()
    big = np.arange(int(np.float32(448).view(np.uint32)), 0x7F800001, 4099,
                    dtype=np.uint32).view(np.float32)
    assert (oracle.e4m3_encode(big) == 0x7E).all()


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(1_000_000) * np.exp2(rng.integers(-30, 30, 1_000_000))).astype(
        np.float32)
    # exact ties: low 16 bits == 0x8000, kept halves of both parities
    hi = rng.integers(0, 1 << 16, 8192, dtype=np.uint32)
    hi = hi[((hi >> 7) & 0xFF) < 0xFE]
    ties = ((hi << 16) | 0x8000).astype(np.uint32).view(np.float32)
    assert (hi & 1).min() == 0 and (hi & 1).max() == 1
    x = np.concatenate([x, ties, -ties]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_round_f32_is_nearest():
    rng = np.random.default_rng(3)
    c = rng.standard_normal(100_000) * 1e3
    np.testing.assert_array_equal(oracle.round_f32(c), c.astype(np.float32))
