"""fp8_quant_act_dual: the 1x128 and 128x1 quantisations of one activation in
one launch, against the CPU oracle bit for bit (codes and scale bits), and
against the two separate entry points.

Sizes span several 128x128 tiles and both full trio activations; the input
may be a column window of a wider matrix, the 1x128 output a window of a
wider buffer (bytes outside it untouched); the degenerate groups of
test_quant_parity (signed zeros, values that round to zero, bf16 subnormals
with FP32-subnormal scales, groups below the fast-division threshold) appear
in both orientations.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import bits, np_u8
from test_quant_parity import _edge_matrix

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _assert_dual(x, x_dev=None):
    xd = x.to(DEV) if x_dev is None else x_dev
    xq, sx, xqT, sxT = fp8fg.fp8_quant_act_dual(xd)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    xb = bits(x.contiguous())
    oq, os_ = oracle.quant_act_1x128(xb)
    oqT, osT = oracle.quant_act_128x1(xb)
    np.testing.assert_array_equal(np_u8(xq), oq)
    np.testing.assert_array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    np.testing.assert_array_equal(np_u8(xqT), oqT)
    np.testing.assert_array_equal(sxT.cpu().numpy().view(np.uint32), osT.view(np.uint32))
    return xq, sx, xqT, sxT


@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (384, 1024), (1280, 640)])
def test_dual_small(M, K):
    _assert_dual(inputs.act(M, K, torch.Generator().manual_seed(M + 7 * K)))


@pytest.mark.parametrize("which", ["x", "dy"])
def test_dual_full_size_matches_separate_calls(which):
    g = torch.Generator().manual_seed(11)
    x = inputs.act(8192, 7168, g) if which == "x" else inputs.grad(8192, 4096, g)
    xd = x.to(DEV)
    xq, sx, xqT, sxT = _assert_dual(x, xd)
    q1, s1 = fp8fg.fp8_quant_act_1x128(xd)
    qT, sT = fp8fg.fp8_quant_act_128x1(xd)
    torch.cuda.synchronize()
    assert torch.equal(xq, q1) and torch.equal(xqT, qT)
    assert torch.equal(sx.view(torch.int32), s1.view(torch.int32))
    assert torch.equal(sxT.view(torch.int32), sT.view(torch.int32))


def test_dual_strided_input_and_output():
    big = inputs.act(256, 640, torch.Generator().manual_seed(5))
    x = big[:, 128:128 + 384]            # row stride 640 elements
    xq_buf = torch.full((256, 384 + 32), 0xCD, dtype=torch.uint8, device=DEV)
    xq = xq_buf[:, 16:16 + 384]
    _, sx, xqT, sxT = fp8fg.fp8_quant_act_dual(big.to(DEV)[:, 128:128 + 384], xq=xq)
    torch.cuda.synchronize()
    xb = bits(x.contiguous())
    oq, os_ = oracle.quant_act_1x128(xb)
    oqT, osT = oracle.quant_act_128x1(xb)
    np.testing.assert_array_equal(np_u8(xq_buf[:, 16:16 + 384]), oq)
    np.testing.assert_array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    np.testing.assert_array_equal(np_u8(xqT), oqT)
    np.testing.assert_array_equal(sxT.cpu().numpy().view(np.uint32), osT.view(np.uint32))
    assert (np_u8(xq_buf[:, :16]) == 0xCD).all() and (np_u8(xq_buf[:, 16 + 384:]) == 0xCD).all()


def test_dual_edge_groups_both_orientations():
    e = _edge_matrix()                    # [8, 256]: degenerate 1x128 groups in rows
    x = torch.zeros(256, 256, dtype=torch.bfloat16)
    x[:8, :] = e                          # ... as rows of the first token group
    x[128:, :8] = e.T[:128]               # ... and as columns of the second (128x1 groups)
    x[128:, 8:16] = e.T[128:]
    _assert_dual(x)


def test_dual_shape_errors():
    x = torch.zeros(256, 192, dtype=torch.bfloat16, device=DEV)   # K % 128 != 0
    with pytest.raises(fp8fg.Fp8Error) as ex:
        fp8fg.fp8_quant_act_dual(x)
    assert ex.value.status == 2  # FP8_ERR_SHAPE
    x = torch.zeros(200, 256, dtype=torch.bfloat16, device=DEV)   # M % 128 != 0
    with pytest.raises(fp8fg.Fp8Error) as ex:
        fp8fg.fp8_quant_act_dual(x, sxT=torch.empty(1, 256, device=DEV))
    assert ex.value.status == 2
