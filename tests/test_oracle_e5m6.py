"""Pins of the oracle's E5M6 format and its 1x128 quantiser (CPU only).

The report (section 3.3.1) names a customised E5M6 format (5-bit exponent,
6-bit mantissa) for one class of activations; the oracle reads it as an
IEEE-style format (bias 15, exponent field 31 for infinity/NaN, subnormals,
largest finite 65024) with round-to-nearest-even and saturation, and applies
the same 1x128 fine-grained grouping as the E4M3 activations with the scale
amax / 65024.  Pinned against: hand-worked boundary values
(tests/golden/e5m6_encode_boundaries.txt), the IEEE binary16 values (a library
type with the same exponent field: every E5M6 value is a binary16 whose four
low mantissa bits are zero), an exhaustive nearest-value search over binary32
inputs, the quantiser's invariants, and the bit-level definition of the packed
storage layout.
"""
import numpy as np
import pytest

import oracle
from conftest import read_golden

MAX = 65024.0


def _f32(s):
    return np.float32(float(s))


def test_encode_golden_boundaries():
    rows = read_golden("e5m6_encode_boundaries.txt")
    assert len(rows) >= 25
    xs = np.array([_f32(r[0]) for r in rows], np.float32)
    want = np.array([int(r[1], 16) for r in rows], np.uint16)
    got = oracle.e5m6_encode(xs)
    bad = [(rows[i][0], hex(got[i]), rows[i][1]) for i in np.nonzero(got != want)[0]]
    assert not bad, bad


def test_decode_all_codes_are_binary16_with_four_zero_low_bits():
    codes = np.arange(4096, dtype=np.uint16)
    ref = (codes.astype(np.uint16) << 4).view(np.float16).astype(np.float64)
    got = oracle.e5m6_decode(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2 * 63  # exponent field 31 with a nonzero mantissa, both signs
    assert (np.isnan(got) == nan).all()
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    np.testing.assert_array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    assert got[0x7BF] == MAX and got[0x040] == 2.0 ** -14 and got[0x001] == 2.0 ** -20
    assert np.isinf(got[0x7C0]) and got[0xFC0] == -np.inf


def _finite_table():
    """Non-negative finite E5M6 values in code order (increasing), codes 0..0x7BF."""
    codes = np.arange(0x7C0, dtype=np.uint16)
    v = oracle.e5m6_decode(codes)
    assert np.all(np.diff(v) > 0)
    return codes, v


def _nearest_even(x, codes, v):
    """Code of the nearest table value to each x >= 0 (binary64 distances),
    ties to the even code (= even mantissa), saturating at the top."""
    i = np.searchsorted(v, x, side="left")
    i = np.clip(i, 1, len(v) - 1)
    lo, hi = v[i - 1], v[i]
    dlo, dhi = x - lo, hi - x
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[i] % 2 == 0))
    out = np.where(pick_hi, codes[i], codes[i - 1])
    out = np.where(x >= v[-1], codes[-1], out)
    return out.astype(np.uint16)


@pytest.mark.slow
def test_encode_is_nearest_value_for_every_binary32_in_range():
    """Every binary32 in [2^-22, 2^16], one binade at a time, plus both signs of a
    sample: the encoder returns the nearest E5M6 value, ties to even."""
    codes, v = _finite_table()
    for e in range(-22, 16):
        bits = (np.arange(1 << 23, dtype=np.uint32) | np.uint32((e + 127) << 23))
        x = bits.view(np.float32)
        got = oracle.e5m6_encode(x)
        want = _nearest_even(x.astype(np.float64), codes, v)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, "2^%d binade: x=%r got %#x want %#x" % (
            e, float(x[bad[0]]), got[bad[0]], want[bad[0]])
    rng = np.random.default_rng(3)
    x = np.exp2(rng.uniform(-30, 20, 200_000)).astype(np.float32)
    np.testing.assert_array_equal(oracle.e5m6_encode(-x), oracle.e5m6_encode(x) | 0x800)


def test_saturation_and_specials():
    x = np.array([MAX, 70000.0, np.inf, -np.inf, 3.0e38, np.nan, -np.nan, 0.0, -0.0],
                 np.float32)
    got = oracle.e5m6_encode(x)
    assert [hex(c) for c in got[:5]] == ["0x7bf", "0x7bf", "0x7bf", "0xfbf", "0x7bf"]
    assert got[5] & 0x7FF == 0x7FF and got[6] & 0x7FF == 0x7FF
    assert got[7] == 0x000 and got[8] == 0x800


def _groups(rng, M, K, spread=20):
    """bfloat16 bits of rows whose 1x128 groups span many binades and signs."""
    mag = np.exp2(rng.uniform(-spread, spread, (M, K))).astype(np.float32)
    x = (mag * rng.choice([-1.0, 1.0], (M, K))).astype(np.float32)
    u = x.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)  # RNE to bfloat16


def _bf16_f64(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_quantiser_scale_invariants_and_error_bound():
    rng = np.random.default_rng(5)
    xb = _groups(rng, 64, 512)
    q, sx = oracle.quant_act_1x128_e5m6(xb)
    x = _bf16_f64(xb)
    dec = oracle.e5m6_decode(q)
    for kb in range(512 // 128):
        g = x[:, kb * 128:(kb + 1) * 128]
        s = sx[kb].astype(np.float64)
        amax = np.abs(g).max(axis=1)
        # s = fl32(amax / 65024)
        np.testing.assert_array_equal(sx[kb], (amax.astype(np.float32) / np.float32(MAX)))
        qs = dec[:, kb * 128:(kb + 1) * 128]
        assert np.all(np.abs(qs) <= MAX)
        # the amax element always encodes to +-65024: |amax / s| is within a
        # few binary32 ulps of 65024, far inside half an E5M6 ulp (256)
        i = np.abs(g).argmax(axis=1)
        assert np.all(np.abs(qs[np.arange(64), i]) == MAX)
        # dequantisation error: half an E5M6 ulp of x/s, plus the binary32
        # rounding of the quotient that comes before the E5M6 rounding
        r = g / s[:, None]
        a = np.abs(r)
        ulp = np.where(a < 2.0 ** -14, 2.0 ** -20,
                       np.exp2(np.floor(np.log2(np.maximum(a, 2.0 ** -14)))) / 64.0)
        assert np.all(np.abs(qs - r) <= 0.5 * ulp + a * 2.0 ** -24)
        np.testing.assert_array_equal(np.signbit(qs), np.signbit(g))


def test_quantiser_power_of_two_equivariance_and_zero_group():
    rng = np.random.default_rng(6)
    xb = _groups(rng, 8, 256, spread=8)
    q, sx = oracle.quant_act_1x128_e5m6(xb)
    for j in (-7, 3, 11):
        # multiply every element by 2^j: adds j to each bfloat16 exponent field
        e = ((xb >> 7) & 0xFF).astype(np.int32)
        assert np.all((e + j > 0) & (e + j < 255))
        xj = ((xb & 0x807F) | ((e + j).astype(np.uint16) << 7)).astype(np.uint16)
        qj, sj = oracle.quant_act_1x128_e5m6(xj)
        np.testing.assert_array_equal(qj, q)
        np.testing.assert_array_equal(sj, sx * np.float32(2.0 ** j))
    z = np.zeros((2, 128), np.uint16)
    z[1] = 0x8000  # -0.0
    qz, sz = oracle.quant_act_1x128_e5m6(z)
    assert np.all(sz == 1.0) and np.all(qz[0] == 0) and np.all(qz[1] == 0x800)


def test_packing_bit_layout():
    # hand-worked: codes 0x123, 0xABC -> bytes 0x23, 0xC1, 0xAB
    p = oracle.pack_e5m6(np.array([[0x123, 0xABC]], np.uint16))
    assert p.tolist() == [[0x23, 0xC1, 0xAB]]
    # definition: element i is bits 12 i .. 12 i + 11 of the row read as one
    # little-endian integer
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 4096, (3, 256)).astype(np.uint16)
    packed = oracle.pack_e5m6(codes)
    assert packed.shape == (3, 384)
    for r in range(3):
        big = int.from_bytes(packed[r].tobytes(), "little")
        assert [(big >> (12 * i)) & 0xFFF for i in range(256)] == codes[r].tolist()
    np.testing.assert_array_equal(oracle.unpack_e5m6(packed), codes)
