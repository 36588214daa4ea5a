"""The MXFP8 variant on the GPU vs the CPU oracle: the power-of-two-scale
quantisers bit-exact (codes and UE8M0 bytes), and the block-scaled tensor-core
GEMM (fp8_gemm_mxfp8) against the oracle's binary64 product with the same
power-of-two scales: FP32 output within relative Frobenius error 1e-5 and the
FP32 accumulation bound elementwise, BF16 output within 1 ulp."""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import U32, bits, check_bf16, check_f32, magnitude, np_u8, sample_rows
from test_quant_parity import _edge_matrix

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("M,K", [(1, 128), (63, 256), (130, 1024), (1000, 640)])
def test_act_quantiser(M, K):
    x = inputs.act(M, K, torch.Generator().manual_seed(M + K + 1))
    xq, se8 = fp8fg.fp8_quant_act_1x128_pow2(x.to(DEV))
    torch.cuda.synchronize()
    oq, os8 = oracle.quant_act_1x128_pow2(bits(x))
    np.testing.assert_array_equal(np_u8(xq), oq)
    np.testing.assert_array_equal(np_u8(se8), os8)


def test_act_quantiser_edge_groups():
    x = _edge_matrix()
    xq, se8 = fp8fg.fp8_quant_act_1x128_pow2(x.to(DEV))
    torch.cuda.synchronize()
    oq, os8 = oracle.quant_act_1x128_pow2(bits(x))
    np.testing.assert_array_equal(np_u8(xq), oq)
    np.testing.assert_array_equal(np_u8(se8), os8)
    assert np_u8(se8)[0, 0] == 127  # all-zero group: e = 0


def test_act_quantiser_every_bf16_amax():
    """One group per positive bfloat16 amax value (its exponent decides the codes)."""
    amax = torch.arange(1, 0x7F80, dtype=torch.int32)
    g = torch.Generator().manual_seed(3)
    fill = (torch.rand(amax.numel(), 127, generator=g) * 2 - 1)
    a = (amax.to(torch.int32) << 16).view(torch.float32)[:, None]
    x = torch.cat([a, fill * a], 1).to(torch.bfloat16)   # |fill * a| <= a
    xq, se8 = fp8fg.fp8_quant_act_1x128_pow2(x.to(DEV))
    torch.cuda.synchronize()
    oq, os8 = oracle.quant_act_1x128_pow2(bits(x))
    np.testing.assert_array_equal(np_u8(se8), os8)
    np.testing.assert_array_equal(np_u8(xq), oq)


@pytest.mark.parametrize("K,N", [(128, 128), (256, 384), (7168, 4096)])
def test_weight_quantiser(K, N):
    w = inputs.weight(K, N, torch.Generator().manual_seed(K + N))
    wq, se8 = fp8fg.fp8_quant_weight_128x128_pow2(w.to(DEV))
    torch.cuda.synchronize()
    oq, os8 = oracle.quant_weight_128x128_pow2(bits(w))
    np.testing.assert_array_equal(np_u8(wq), oq)
    np.testing.assert_array_equal(np_u8(se8), os8)


def _operands(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    aq, sa8 = oracle.quant_act_1x128_pow2(bits(inputs.act(M, K, g)))
    bq, sb8 = oracle.quant_weight_128x128_pow2(bits(inputs.weight(K, N, g)))
    return aq, sa8, bq, sb8


def _compare(out, aq, sa8, bq, sb8, rows=None):
    """The GPU result against the oracle's binary64 product with the same scales.
    The tensor core accumulates the whole K range in FP32, one rounding per
    32-element MMA step, so the elementwise bound is u (K/32 + 32) S."""
    M, K = aq.shape
    rows = np.arange(M) if rows is None else rows
    sa, sb = oracle.e8_scales(sa8), oracle.e8_scales(sb8)
    ref = oracle.gemm_blockscaled(aq, sa, bq, sb, oracle.BSCALE_ROW1x128, rows=rows)
    sbm = sb.T.astype(np.float64)                     # [N, K/128]
    S = lambda idx: magnitude(aq, sa, bq, sbm, rows[idx])
    o = out.cpu()
    if o.dtype == torch.float32:
        got = o.numpy()[rows].astype(np.float64)
        check_f32(got, ref)
        d = np.abs(got - ref)
        gamma = U32 * (K // 32 + 32)
        loose = np.nonzero((d > gamma * np.abs(ref)).any(axis=1))[0]
        if loose.size:
            assert np.all(d[loose] <= gamma * S(loose) + 1e-300)
        return 0
    return check_bf16(o.view(torch.int16).numpy().view(np.uint16)[rows], ref, S=S, K=4 * K)


def test_smallest_tile():
    aq, sa8, bq, sb8 = _operands(128, 256, 128, seed=1)
    out = fp8fg.fp8_gemm_mxfp8(_t(aq), _t(sa8), _t(bq), _t(sb8), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    _compare(out, aq, sa8, bq, sb8)


SHAPES = [(1, 128, 128), (37, 384, 256), (130, 256, 1024), (257, 512, 384), (300, 640, 128)]


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_shapes(M, N, K, out_dtype):
    aq, sa8, bq, sb8 = _operands(M, N, K, seed=M + N + K)
    out = fp8fg.fp8_gemm_mxfp8(_t(aq), _t(sa8), _t(bq), _t(sb8), out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    _compare(out, aq, sa8, bq, sb8)


def test_dense_fprop_size_end_to_end():
    """X[8192, 2048] . W[2048, 7168] -> BF16: the GPU quantisers feed the GPU GEMM;
    the oracle quantises the same inputs and forms the product; 1024 rows that
    include every 128-row tile's first and last row."""
    wl = inputs.fprop_dense()
    xq, sx8 = fp8fg.fp8_quant_act_1x128_pow2(wl.x.to(DEV))
    wq, sw8 = fp8fg.fp8_quant_weight_128x128_pow2(wl.w.to(DEV))
    y = fp8fg.fp8_gemm_mxfp8(xq, sx8, wq, sw8, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    aq, sa8 = oracle.quant_act_1x128_pow2(bits(wl.x))
    bq, sb8 = oracle.quant_weight_128x128_pow2(bits(wl.w))
    np.testing.assert_array_equal(np_u8(xq), aq)
    np.testing.assert_array_equal(np_u8(wq), bq)
    _compare(y, aq, sa8, bq, sb8, rows=sample_rows(wl.M, 1024, seed=5))


def test_trio_fprop_size_fp32():
    """X[8192, 7168] . W[7168, 4096] -> FP32 (long K: 224 MMA steps accumulate in TMEM)."""
    wl = inputs.training_trio()
    aq, sa8 = oracle.quant_act_1x128_pow2(bits(wl.x))
    bq, sb8 = oracle.quant_weight_128x128_pow2(bits(wl.w))
    out = fp8fg.fp8_gemm_mxfp8(_t(aq), _t(sa8), _t(bq), _t(sb8), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    _compare(out, aq, sa8, bq, sb8, rows=sample_rows(wl.M, 1024, seed=6))
