"""fp8_quant_fprop_operands (activation 1x128 + weight 128x128 in one launch)
vs the CPU oracle: codes and scales bit-exact, as for the single-operand
quantisers.

Sizes mix few and many items of each kind (the grid walks the weight blocks
first, then the activation tiles), with ragged activation rows, strided
inputs and outputs, either weight orientation alone, the degenerate groups,
and the full Fprop workload sizes.
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


def _check(x, w, want_wq=True, want_wqT=False):
    xq, sx, wq, wqT, sw = fp8fg.fp8_quant_fprop_operands(x.to(DEV), w.to(DEV), want_wq=want_wq,
                                                         want_wqT=want_wqT)
    torch.cuda.synchronize()
    if x.shape[0]:
        oq, os_ = oracle.quant_act_1x128(bits(x))
        np.testing.assert_array_equal(np_u8(xq), oq)
        np.testing.assert_array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    if w.shape[1]:
        wq_o, wqT_o, sw_o = oracle.quant_weight_128x128(bits(w))
        if want_wq:
            np.testing.assert_array_equal(np_u8(wq), wq_o)
        if want_wqT:
            np.testing.assert_array_equal(np_u8(wqT), wqT_o)
        np.testing.assert_array_equal(sw.cpu().numpy().view(np.uint32), sw_o.view(np.uint32))


@pytest.mark.parametrize("M,K,N", [
    (1, 128, 128), (63, 256, 384), (65, 384, 128), (1000, 640, 256), (3000, 256, 1280),
    (130, 1024, 2048)])
def test_small(M, K, N):
    g = torch.Generator().manual_seed(M + K + N)
    _check(inputs.act(M, K, g), inputs.weight(K, N, g))


def test_both_weight_orientations_and_each_alone():
    g = torch.Generator().manual_seed(4)
    x, w = inputs.act(300, 512, g), inputs.weight(512, 640, g)
    _check(x, w, want_wq=True, want_wqT=True)
    _check(x, w, want_wq=False, want_wqT=True)


def test_edge_groups():
    x = _edge_matrix()                       # [8, 256]
    w = torch.zeros(256, 256, dtype=torch.bfloat16)
    w[:128, :128] = _edge_matrix()[:, :128].repeat(16, 1)
    w[128:, 128:] = 1e-39
    _check(x, w, want_wq=True, want_wqT=True)


def test_one_operand_empty():
    g = torch.Generator().manual_seed(6)
    _check(torch.zeros(0, 256, dtype=torch.bfloat16), inputs.weight(256, 384, g))
    _check(inputs.act(77, 256, g), torch.zeros(256, 0, dtype=torch.bfloat16))


def test_strided_input_and_output():
    g = torch.Generator().manual_seed(8)
    x_full = inputs.act(100, 512 + 24, g)
    w_full = inputs.weight(512, 256 + 8, g)
    x = x_full.to(DEV)[:, 8:8 + 512]
    w = w_full.to(DEV)[:, :256]             # row stride 264
    xq_buf = torch.full((100, 512 + 32), 0xAB, dtype=torch.uint8, device=DEV)
    xq, sx, wq, _, sw = fp8fg.fp8_quant_fprop_operands(x, w, xq=xq_buf[:, 16:16 + 512])
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_act_1x128(bits(x_full[:, 8:8 + 512].contiguous()))
    np.testing.assert_array_equal(np_u8(xq_buf[:, 16:16 + 512]), oq)
    np.testing.assert_array_equal(sx.cpu().numpy(), os_)
    assert (np_u8(xq_buf[:, :16]) == 0xAB).all() and (np_u8(xq_buf[:, 16 + 512:]) == 0xAB).all()
    wq_o, _, sw_o = oracle.quant_weight_128x128(bits(w_full[:, :256].contiguous()))
    np.testing.assert_array_equal(np_u8(wq), wq_o)
    np.testing.assert_array_equal(sw.cpu().numpy(), sw_o)


def test_fprop_workload_sizes():
    """8192 x 2048 activations with the 2048 x 7168 weight, as the Fprop step runs it."""
    wl = inputs.fprop_dense(seed=0)
    _check(wl.x, wl.w)


def test_same_bits_as_the_single_operand_calls():
    g = torch.Generator().manual_seed(10)
    x, w = inputs.act(4096, 1024, g).to(DEV), inputs.weight(1024, 3072, g).to(DEV)
    xq, sx, wq, wqT, sw = fp8fg.fp8_quant_fprop_operands(x, w, want_wqT=True)
    xq1, sx1 = fp8fg.fp8_quant_act_1x128(x)
    wq1, wqT1, sw1 = fp8fg.fp8_quant_weight_128x128(w, want_wqT=True)
    torch.cuda.synchronize()
    assert torch.equal(xq, xq1) and torch.equal(wq, wq1) and torch.equal(wqT, wqT1)
    assert torch.equal(sx.view(torch.int32), sx1.view(torch.int32))
    assert torch.equal(sw.view(torch.int32), sw1.view(torch.int32))
