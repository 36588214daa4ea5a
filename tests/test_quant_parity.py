"""GPU quantisers vs the CPU oracle: codes and scales must be bit-exact.

Sizes span several CTAs with ragged tails, the full workload sizes, strided
inputs/outputs and the degenerate groups (all-zero, signed zeros, values that
round to zero, bf16 subnormals whose scale is an FP32 subnormal).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import bits, np_u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _act(M, K, seed):
    return inputs.act(M, K, torch.Generator().manual_seed(seed))


def _assert_1x128(x):
    xq, sx = fp8fg.fp8_quant_act_1x128(x.to(DEV))
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_act_1x128(bits(x))
    np.testing.assert_array_equal(np_u8(xq), oq)
    np.testing.assert_array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("M,K", [(1, 128), (63, 256), (65, 384), (130, 1024), (1000, 640)])
def test_1x128_small(M, K):
    _assert_1x128(_act(M, K, M + K))


@pytest.mark.parametrize("M,K", [(8192, 2048), (8192, 7168)])
def test_1x128_full_size(M, K):
    _assert_1x128(_act(M, K, 7))


def test_1x128_strided_input_and_output():
    x_full = _act(100, 512 + 24, 3)
    x = x_full.to(DEV)[:, 8:8 + 512]  # row stride 536, 16-byte aligned start
    xq_buf = torch.full((100, 512 + 32), 0xAB, dtype=torch.uint8, device=DEV)
    xq, sx = fp8fg.fp8_quant_act_1x128(x, xq=xq_buf[:, 16:16 + 512])
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_act_1x128(bits(x_full[:, 8:8 + 512].contiguous()))
    np.testing.assert_array_equal(np_u8(xq_buf[:, 16:16 + 512]), oq)
    np.testing.assert_array_equal(sx.cpu().numpy(), os_)
    # bytes outside the output view are untouched
    assert (np_u8(xq_buf[:, :16]) == 0xAB).all() and (np_u8(xq_buf[:, 16 + 512:]) == 0xAB).all()


def _edge_matrix():
    x = torch.zeros(8, 256, dtype=torch.float32)
    x[1, 0] = -0.0
    x[2, 7] = -3.0
    x[2, 8] = -1e-6          # rounds to -0 after scaling
    x[3] = torch.linspace(-2.0, 2.0, 256)
    x[4, :] = 1e-39          # bf16 subnormals: FP32-subnormal scale
    x[4, 3] = -9.2e-41
    x[5, :128] = 3.0e38      # near the bf16 maximum
    x[5, 128:] = -2.5e-38
    x[6, ::2] = 448.0
    x[6, 1::2] = 464.0
    x[7] = torch.randn(256) * 1e-30
    return x.to(torch.bfloat16)


def test_1x128_edge_groups():
    x = _edge_matrix()
    _assert_1x128(x)
    # sign of zero codes follows the input
    xq, _ = fp8fg.fp8_quant_act_1x128(x.to(DEV))
    q = np_u8(xq)
    assert q[1, 0] == 0x80 and q[0, 0] == 0x00 and q[2, 8] == 0x80


def _assert_128x1(x):
    xqT, sxT = fp8fg.fp8_quant_act_128x1(x.to(DEV))
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_act_128x1(bits(x))
    np.testing.assert_array_equal(np_u8(xqT), oq)
    np.testing.assert_array_equal(sxT.cpu().numpy().view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("M,K", [(128, 64), (256, 192), (384, 1024)])
def test_128x1_small(M, K):
    _assert_128x1(_act(M, K, M * 3 + K))


@pytest.mark.parametrize("which", ["x", "dy"])
def test_128x1_full_size(which):
    g = torch.Generator().manual_seed(9)
    x = inputs.act(8192, 7168, g) if which == "x" else inputs.grad(8192, 4096, g)
    _assert_128x1(x)


def test_128x1_strided_input():
    """A column window of a wider matrix (row stride 512 elements), with a
    64-column last tile: the loader's row stride and its zero-filled tail."""
    big = _act(256, 512, 17)
    x = big[:, 64:64 + 192]
    xqT, sxT = fp8fg.fp8_quant_act_128x1(big.to(DEV)[:, 64:64 + 192])
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_act_128x1(bits(x.contiguous()))
    np.testing.assert_array_equal(xqT.cpu().numpy(), oq)
    np.testing.assert_array_equal(sxT.cpu().numpy().view(np.uint32), os_.view(np.uint32))


def test_128x1_edge_groups():
    x = _edge_matrix().T.contiguous()  # [256, 8]: pad to 64 columns
    xp = torch.zeros(256, 64, dtype=torch.bfloat16)
    xp[:, :8] = x
    _assert_128x1(xp)


def _assert_128x128(w, want_wq=True, want_wqT=True):
    wq, wqT, sw = fp8fg.fp8_quant_weight_128x128(w.to(DEV), want_wq=want_wq, want_wqT=want_wqT)
    torch.cuda.synchronize()
    oq, oqT, os_ = oracle.quant_weight_128x128(bits(w))
    if want_wq:
        np.testing.assert_array_equal(np_u8(wq), oq)
    if want_wqT:
        np.testing.assert_array_equal(np_u8(wqT), oqT)
    np.testing.assert_array_equal(sw.cpu().numpy().view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("K,N", [(128, 128), (256, 384), (640, 256)])
def test_128x128_small(K, N):
    _assert_128x128(inputs.weight(K, N, torch.Generator().manual_seed(K + N)))


@pytest.mark.parametrize("K,N", [(2048, 7168), (7168, 4096)])
def test_128x128_full_size(K, N):
    _assert_128x128(inputs.weight(K, N, torch.Generator().manual_seed(5)))


def test_128x128_single_output_and_edges():
    w = torch.zeros(256, 256, dtype=torch.bfloat16)
    w[:128, :128] = _edge_matrix()[:, :128].repeat(16, 1)
    w[128:, 128:] = 1e-39
    _assert_128x128(w, want_wq=True, want_wqT=False)
    _assert_128x128(w, want_wq=False, want_wqT=True)


def test_zero_rows_is_noop():
    x = torch.empty(0, 256, dtype=torch.bfloat16, device=DEV)
    xq, sx = fp8fg.fp8_quant_act_1x128(x)
    assert xq.shape == (0, 256) and sx.shape == (2, 0)
