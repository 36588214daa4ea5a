"""Pins of the limited-precision accumulation model (CPU).

The model (oracle/accumulation.py) follows the DeepSeek-V3 Technical Report,
section 3.3.2 and Figure 7 (b): a tensor-core sum that keeps about 14 bits,
with or without promotion to full precision every N_C = 128 elements.

Pinned against integer arithmetic (truncation, and the exact sums at full
width), hand-worked closed forms in which promotion recovers terms that the
narrow accumulator drops, and the error bound that truncation implies.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import accumulation as acc
from fp8_fine_grained_22_b300 import inputs

DEC = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(
    torch.float64).numpy()
ONE = 0x38      # E4M3 1.0: exponent field 7 (bias 7), mantissa 0
TINY = 0x01     # E4M3 smallest subnormal, 2^-9


def test_truncate_against_integer_shifts():
    rng = np.random.default_rng(0)
    vals = [int(v) for v in rng.integers(1, 2 ** 40, size=2000)] + [1, 2, 3, 2 ** 14 - 1,
                                                                     2 ** 14, 2 ** 14 + 1]
    for bits in (1, 5, 14, 24, 40):
        x = np.array(vals, dtype=np.float64)
        got = acc.truncate_significand(x, bits)
        for v, gv in zip(vals, got):
            s = max(0, v.bit_length() - bits)
            assert gv == float((v >> s) << s)
        assert np.array_equal(acc.truncate_significand(-x, bits), -got)  # toward zero
    assert acc.truncate_significand(np.array([0.0, -0.0]), 14).tolist() == [0.0, 0.0]
    y = rng.standard_normal(1000)
    assert np.array_equal(acc.truncate_significand(y, 53), y)
    # 1 + 2^-13 + 2^-14 needs 15 bits; at 14 the last one goes
    assert acc.truncate_significand(np.array([1 + 2.0 ** -13 + 2.0 ** -14]), 14)[0] == 1 + 2.0 ** -13


def _codes(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = inputs.bf16_bits(inputs.act(M, K, g))
    w = inputs.bf16_bits(inputs.weight(K, N, g))
    aq, sa = oracle.quant_act_1x128(x)
    wq, _, sw = oracle.quant_weight_128x128(w)
    return aq, sa, wq, sw


def _int_sum(aq, bq):
    """Exact code-product sums in int64 (each decoded value x 2^9 is an integer)."""
    ai = np.round(DEC[aq] * 512).astype(np.int64)
    bi = np.round(DEC[bq] * 512).astype(np.int64)
    return (ai @ bi.T).astype(np.float64) / 2.0 ** 18


def test_full_width_is_exact():
    aq, sa, wq, sw = _codes(64, 128, 512, 1)
    raw = acc.limited_accumulation_gemm(aq, wq, bits=53, chunk=32, interval=0)
    assert np.array_equal(raw, _int_sum(aq, wq))
    promoted = acc.limited_accumulation_gemm(aq, wq, bits=53, chunk=32, interval=128, sa=sa, sb=sw)
    ref = oracle.gemm_blockscaled(aq, sa, wq, sw)
    assert np.allclose(promoted, ref, rtol=1e-14, atol=0)


def _one_big_then_tiny(K):
    """Row 0: product 1 at k = 0, then 2^-18 at every other k; all 128 columns equal."""
    aq = np.full((1, K), TINY, np.uint8)
    bq = np.full((128, K), TINY, np.uint8)
    aq[0, 0] = ONE
    bq[:, 0] = ONE
    sa = np.ones((K // 128, 1), np.float32)
    sb = np.ones((1, K // 128), np.float32)
    return aq, bq, sa, sb


def test_hand_worked_narrow_accumulator():
    K = 256
    aq, bq, sa, sb = _one_big_then_tiny(K)
    exact = 1 + 255 * 2.0 ** -18
    assert _int_sum(aq, bq)[0, 0] == exact
    # 12 bits: the ulp at 1 is 2^-11.  Every 32-product step adds at most
    # 2^-13 to a sum near 1, so without promotion nothing small survives.
    c = acc.limited_accumulation_gemm(aq, bq, bits=12, chunk=32, interval=0)
    assert np.all(c == 1.0)
    # with promotion the second block restarts from zero: its four steps of
    # 32 * 2^-18 = 2^-13 sum exactly to 2^-11, and the first block gives 1
    c = acc.limited_accumulation_gemm(aq, bq, bits=12, chunk=32, interval=128, sa=sa, sb=sb)
    assert np.all(c == 1 + 2.0 ** -11)
    # 14 bits, one step per product: 1 + 2^-18 always cuts back to 1
    c = acc.limited_accumulation_gemm(aq, bq, bits=14, chunk=1, interval=0)
    assert np.all(c == 1.0)
    # 14 bits, 32-product steps: step 1 is 1 + 31 * 2^-18 -> 1 (31 * 2^-18 < 2^-13);
    # each later step adds 2^-13, kept exactly: 1 + 7 * 2^-13
    c = acc.limited_accumulation_gemm(aq, bq, bits=14, chunk=32, interval=0)
    assert np.all(c == 1 + 7 * 2.0 ** -13)
    # wide enough for every term: exact
    c = acc.limited_accumulation_gemm(aq, bq, bits=24, chunk=32, interval=0)
    assert np.all(c == exact)


def _abs_sums(aq, bq, K, blk):
    a = np.abs(DEC[aq])
    b = np.abs(DEC[bq])
    return np.stack([a[:, k:k + blk] @ b[:, k:k + blk].T for k in range(0, K, blk)])


@pytest.mark.parametrize("bits", [10, 14])
def test_truncation_error_bounds(bits):
    """Each cut loses less than 2^(1 - bits) of a running sum whose magnitude
    never exceeds the sum of |products| seen so far, so
      no promotion: |C - exact| <= (K / chunk) 2^(1 - bits) S_K
      promotion:    |C - exact| <= sum_kb |sa sb| (128 / chunk) 2^(1 - bits) S_kb."""
    M, N, K, chunk = 32, 128, 1024, 32
    aq, sa, wq, sw = _codes(M, N, K, 2)
    u = 2.0 ** (1 - bits)
    s_blocks = _abs_sums(aq, wq, K, 128)                  # [K/128, M, N]
    raw = acc.limited_accumulation_gemm(aq, wq, bits, chunk, 0)
    err = np.abs(raw - _int_sum(aq, wq))
    assert np.all(err <= (K // chunk) * u * s_blocks.sum(0))
    pro = acc.limited_accumulation_gemm(aq, wq, bits, chunk, 128, sa=sa, sb=sw)
    ref = oracle.gemm_blockscaled(aq, sa, wq, sw)
    scale = sa.astype(np.float64)[:, :, None] * sw.astype(np.float64).T[:, None, :].repeat(128, 2)
    bound = ((128 // chunk) * u * scale * s_blocks).sum(0)
    assert np.all(np.abs(pro - ref) <= bound + 1e-12 * np.abs(ref))


def test_promotion_keeps_the_error_flat_in_k():
    """The effect the report describes: a ~14-bit accumulator over the whole
    of K loses accuracy in proportion to K; promoting every 128 elements
    keeps it at the level of one block."""
    fro_raw, fro_pro = [], []
    for K in (512, 2048, 4096):
        aq, sa, wq, sw = _codes(64, 128, K, 3)
        raw = acc.limited_accumulation_gemm(aq, wq, 14, 32, 0)
        pro = acc.limited_accumulation_gemm(aq, wq, 14, 32, 128, sa=sa, sb=sw)
        fro_raw.append(acc.relative_errors(raw, _int_sum(aq, wq))[0])
        fro_pro.append(acc.relative_errors(pro, oracle.gemm_blockscaled(aq, sa, wq, sw))[0])
    assert fro_raw[0] < fro_raw[1] < fro_raw[2]
    assert fro_raw[2] > 4 * fro_raw[0]
    assert max(fro_pro) < 2 * min(fro_pro)
    assert fro_raw[2] > 10 * fro_pro[2]


def error_table(Ks=(128, 512, 2048, 4096, 7168), M=128, N=128, seed=0):
    """Rows (K, bits, relative Frobenius error without promotion, with
    promotion) on the Fprop input recipe; printed when run as a script."""
    rows = []
    for K in Ks:
        aq, sa, wq, sw = _codes(M, N, K, seed)
        exact_raw = _int_sum(aq, wq)
        exact = oracle.gemm_blockscaled(aq, sa, wq, sw)
        for bits in (14, 24):
            raw = acc.limited_accumulation_gemm(aq, wq, bits, 32, 0)
            pro = acc.limited_accumulation_gemm(aq, wq, bits, 32, 128, sa=sa, sb=sw)
            rows.append((K, bits, acc.relative_errors(raw, exact_raw)[0],
                         acc.relative_errors(pro, exact)[0]))
    return rows


if __name__ == "__main__":
    print("| K | bits kept | rel. Frobenius error, no promotion | with promotion every 128 |")
    print("|---|---|---|---|")
    for K, bits, e_raw, e_pro in error_table():
        print(f"| {K} | {bits} | {e_raw:.2e} | {e_pro:.2e} |")
