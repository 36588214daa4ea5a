"""Pins of the oracle's power-of-two-scale quantisers (CPU only): the variant
whose scales a block-scaled (MXFP8) tensor-core MMA can apply exactly.

Pinned against: the defining properties of the exponent over every positive
bfloat16 amax (feasible: amax / 2^e <= 448; minimal: 2^(e-1) would not do;
clamped to the UE8M0 range), the pinned E4M3 encoder applied to the exactly
scaled values, the reduction to the amax/448 quantiser when amax / 448 is a
power of two, and a brute-force exact product for the GEMM with these
scales (binary64 is exact there: every scale is a power of two).
"""
import math
from fractions import Fraction

import numpy as np

import oracle


def _bf16_values(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def test_exponent_is_minimal_and_feasible_for_every_bf16_amax():
    bits = np.arange(1, 0x7F80, dtype=np.uint32)       # every positive finite bfloat16
    amax = _bf16_values(bits).astype(np.float64)
    e = np.array([oracle.pow2_exponent(a) for a in amax], np.int64)
    assert e.min() == -127 and e.max() <= 127
    feasible = amax <= 448.0 * np.ldexp(1.0, e)
    minimal = (e == -127) | (amax > 448.0 * np.ldexp(1.0, e - 1))
    bad = np.nonzero(~(feasible & minimal))[0]
    assert bad.size == 0, "amax %r -> e %d" % (amax[bad[0]], e[bad[0]])
    # clamped only where amax is below 448 * 2^-128
    assert np.all((e > -127) | (amax <= 448.0 * 2.0 ** -127))
    assert oracle.pow2_exponent(0.0) == 0


def _groups(rng, M, K, spread=30):
    mag = np.exp2(rng.uniform(-spread, spread, (M, K)))
    x = (mag * rng.choice([-1.0, 1.0], (M, K))).astype(np.float32)
    u = x.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def test_act_codes_are_e4m3_of_exactly_scaled_values():
    rng = np.random.default_rng(11)
    xb = _groups(rng, 32, 512)
    xq, se8 = oracle.quant_act_1x128_pow2(xb)
    x = _bf16_values(xb).astype(np.float64)
    for kb in range(4):
        g = x[:, kb * 128:(kb + 1) * 128]
        e = se8[kb].astype(np.int64) - 127
        amax = np.abs(g).max(axis=1)
        np.testing.assert_array_equal(e, [oracle.pow2_exponent(a) for a in amax])
        scaled = g * np.ldexp(1.0, -e)[:, None]          # exact in binary64
        want = oracle.e4m3_encode(scaled.astype(np.float32))
        np.testing.assert_array_equal(xq[:, kb * 128:(kb + 1) * 128], want)
        r = np.abs(amax * np.ldexp(1.0, -e))
        assert np.all((r > 224.0) & (r <= 448.0))


def test_reduces_to_the_amax_over_448_quantiser_when_that_is_a_power_of_two():
    rng = np.random.default_rng(12)
    xb = _groups(rng, 16, 256, spread=4)
    # force each group's amax to 448 * 2^j (bfloat16 448 = 0x43E0), j in [-20, 20]
    x = _bf16_values(xb).copy()
    for m in range(16):
        for kb in range(2):
            j = int(rng.integers(-20, 21))
            g = x[m, kb * 128:(kb + 1) * 128]
            g *= np.float32(2.0 ** j) / np.float32(np.abs(g).max()) * np.float32(0.9)
            g[int(rng.integers(0, 128))] = np.float32(448.0 * 2.0 ** j)
    xb2 = (x.view(np.uint32) >> 16).astype(np.uint16)  # exact: values chosen bf16-representable
    assert np.array_equal((xb2.astype(np.uint32) << 16).view(np.float32).max(), x.max())
    q_pow2, se8 = oracle.quant_act_1x128_pow2(xb2)
    q_ref, s_ref = oracle.quant_act_1x128(xb2)
    np.testing.assert_array_equal(oracle.e8_scales(se8), s_ref)
    np.testing.assert_array_equal(q_pow2, q_ref)


def test_weight_block_exponent_repeated_per_row():
    rng = np.random.default_rng(13)
    wb = _groups(rng, 256, 384, spread=10)             # w [K=256, N=384]
    wq, se8 = oracle.quant_weight_128x128_pow2(wb)
    w = _bf16_values(wb).astype(np.float64)
    assert wq.shape == (384, 256) and se8.shape == (2, 384)
    for kb in range(2):
        for nb in range(3):
            blk = w[kb * 128:(kb + 1) * 128, nb * 128:(nb + 1) * 128]
            e = oracle.pow2_exponent(np.abs(blk).max())
            assert np.all(se8[kb, nb * 128:(nb + 1) * 128] == e + 127)
            want = oracle.e4m3_encode((blk * 2.0 ** -e).astype(np.float32)).T
            np.testing.assert_array_equal(wq[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128],
                                          want)


def test_gemm_with_pow2_scales_is_exact():
    """M=2, N=128, K=256: the oracle's binary64 block-scaled product equals the
    exact rational sum (all scales powers of two, all codes exact)."""
    rng = np.random.default_rng(14)
    xb = _groups(rng, 2, 256, spread=6)
    wb = _groups(rng, 256, 128, spread=6)
    aq, sa8 = oracle.quant_act_1x128_pow2(xb)
    bq, sb8 = oracle.quant_weight_128x128_pow2(wb)
    got = oracle.gemm_blockscaled(aq, oracle.e8_scales(sa8), bq, oracle.e8_scales(sb8),
                                  oracle.BSCALE_ROW1x128)
    dec = [None if math.isnan(v) else Fraction(float(v))
           for v in oracle.e4m3_decode(np.arange(256, dtype=np.uint8))]
    for m in range(2):
        for n in range(0, 128, 17):
            acc = Fraction(0)
            for k in range(256):
                kb = k // 128
                acc += (dec[aq[m, k]] * dec[bq[n, k]] * Fraction(2) ** (int(sa8[kb, m]) - 127)
                        * Fraction(2) ** (int(sb8[kb, n]) - 127))
            assert Fraction(float(got[m, n])) == acc, (m, n)
