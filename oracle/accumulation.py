"""Emulated limited-precision tensor-core accumulation (a diagnostic model).

TEST INFRASTRUCTURE ONLY, like the rest of this package: the product path
never imports it.  Plain numpy, binary64.

DeepSeek-V3 Technical Report, section 3.3.2 (increasing accumulation
precision) and Figure 7 (b): the FP8 MMA of the H800 keeps only about 14
bits of its running sum, far fewer than FP32; the method therefore copies the
tensor core's partial sums to FP32 registers on the CUDA cores every
N_C = 128 elements of the inner dimension, multiplies them by the group
scaling factors there and finishes the accumulation in full precision.

This module models such an accumulator so that the effect can be shown on
the host, with and without that promotion:

* the products of decoded E4M3 codes inside one MMA step of ``chunk``
  elements of K are summed exactly (the tensor core's adder tree);
* the step's sum is added to the running tensor-core sum, and the result is
  cut to ``bits`` significant bits, rounding toward zero;
* with promotion every ``interval`` elements, the running tensor-core sum is
  multiplied by its group's scales (1x128 on A, 128x128 on B), added to a
  binary64 accumulator, and the tensor-core sum restarts at zero;
* without promotion (``interval`` 0) the whole of K is summed on the tensor
  core and no scales are applied (a per-tensor scale would multiply the
  result afterwards and change no relative error).

Readings (the report gives only "about 14 bits"): the bit count includes the
leading one; the cut rounds toward zero; one MMA step is summed exactly
(K = 32 for FP8 MMA steps); the promoted sum is kept in binary64 so that the
model measures the tensor core's loss alone.
"""
from __future__ import annotations

import numpy as np

from . import e4m3_decode


def truncate_significand(x, bits: int) -> np.ndarray:
    """Each value of ``x`` cut to ``bits`` significant bits, toward zero.

    Zero stays zero.  Exact in binary64 for 1 <= bits <= 53.
    """
    assert 1 <= bits <= 53
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                 # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.trunc(np.ldexp(m, bits)), e - bits)


def limited_accumulation_gemm(aq, bq, bits: int, chunk: int = 32, interval: int = 128,
                              sa=None, sb=None) -> np.ndarray:
    """C [M, N] as the modelled accumulator forms it.

    aq: uint8 [M, K] E4M3 codes; bq: uint8 [N, K] codes (the weight, K-major).
    With ``interval`` > 0 (a multiple of ``chunk`` that divides 128), sa f32
    [K/128, M] and sb f32 [N/128, K/128] are the 1x128 and 128x128 scales and
    the result is the promoted, scaled product.  With ``interval`` 0 the
    result is the unscaled sum of code products over all of K.
    """
    aq = np.asarray(aq, dtype=np.uint8)
    bq = np.asarray(bq, dtype=np.uint8)
    M, K = aq.shape
    N, K2 = bq.shape
    assert K == K2 and K % chunk == 0
    a = e4m3_decode(aq)
    b = e4m3_decode(bq)
    if interval:
        assert interval % chunk == 0 and 128 % interval == 0 and K % 128 == 0 and N % 128 == 0
        sa = np.asarray(sa, dtype=np.float64)
        sb = np.asarray(sb, dtype=np.float64)
        assert sa.shape == (K // 128, M) and sb.shape == (N // 128, K // 128)
        nb_of_col = np.arange(N) // 128
    acc = np.zeros((M, N), np.float64)
    tc = np.zeros((M, N), np.float64)
    for k0 in range(0, K, chunk):
        k1 = k0 + chunk
        # one MMA step: at most 32 products, each exact in binary64, whose
        # partial sums stay below 2^23 on a grid of 2^-18, hence exact
        step = a[:, k0:k1] @ b[:, k0:k1].T
        tc = truncate_significand(tc + step, bits)
        if interval and k1 % interval == 0:
            kb = k0 // 128
            acc += tc * sa[kb][:, None] * sb[nb_of_col, kb][None, :]
            tc = np.zeros((M, N), np.float64)
    return acc if interval else tc


def relative_errors(approx, exact):
    """(relative Frobenius error, largest elementwise relative error over
    elements with |exact| >= 1e-3 * max|exact|)."""
    approx = np.asarray(approx, np.float64)
    exact = np.asarray(exact, np.float64)
    fro = float(np.linalg.norm(approx - exact) / np.linalg.norm(exact))
    big = np.abs(exact) >= 1e-3 * np.abs(exact).max()
    elt = float(np.max(np.abs(approx - exact)[big] / np.abs(exact)[big]))
    return fro, elt
