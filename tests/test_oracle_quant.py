"""Pins of the oracle's fine-grained quantisers (CPU only).

Each quantiser is checked against an independent PyTorch restatement
(torch's IEEE float32 division and its float8_e4m3fn cast are library
routines), against invariants the method fixes (scale bound, the amax element
hits the top of the E4M3 range, half-ulp dequantisation error, power-of-two
scale equivariance, the all-zero group), and against layout identities
between the three quantisers.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import inputs


def _bits(t):
    return inputs.bf16_bits(t)


def _torch_group_quant(xf, dim):
    """xf: float32 tensor whose ``dim`` axes form the groups."""
    amax = xf.abs().amax(dim=dim, keepdim=True)
    s = torch.where(amax == 0, torch.ones_like(amax), amax / torch.tensor(448.0))
    q = (xf / s).to(torch.float8_e4m3fn).view(torch.uint8)
    return q, s


@pytest.fixture(scope="module")
def acts():
    g = torch.Generator().manual_seed(11)
    return inputs.act(256, 640, g)


def test_1x128_matches_torch_restatement(acts):
    x = acts
    M, K = x.shape
    xq, sx = oracle.quant_act_1x128(_bits(x))
    xf = x.float().view(M, K // 128, 128)
    q, s = _torch_group_quant(xf, dim=2)
    np.testing.assert_array_equal(xq, q.reshape(M, K).numpy())
    np.testing.assert_array_equal(sx, s.reshape(M, K // 128).T.numpy())


def test_128x1_matches_torch_restatement(acts):
    x = acts
    M, K = x.shape
    xqT, sxT = oracle.quant_act_128x1(_bits(x))
    xf = x.float().view(M // 128, 128, K)
    q, s = _torch_group_quant(xf, dim=1)
    np.testing.assert_array_equal(xqT, q.reshape(M, K).T.numpy())
    np.testing.assert_array_equal(sxT, s.reshape(M // 128, K).numpy())


def test_128x128_matches_torch_restatement():
    g = torch.Generator().manual_seed(12)
    w = inputs.weight(384, 256, g)
    K, N = w.shape
    wq, wqT, sw = oracle.quant_weight_128x128(_bits(w))
    wf = w.float().view(K // 128, 128, N // 128, 128)
    q, s = _torch_group_quant(wf, dim=(1, 3))
    q = q.reshape(K, N).numpy()
    np.testing.assert_array_equal(wqT, q)
    np.testing.assert_array_equal(wq, q.T)
    np.testing.assert_array_equal(sw, s.reshape(K // 128, N // 128).T.numpy())


def _dequant_bound(x64, q, s64):
    """Half an E4M3 ulp of the quotient (plus its binary32 rounding), times s."""
    r = np.abs(x64 / s64)
    e = np.floor(np.log2(np.maximum(r, 2.0 ** -6)))
    ulp = np.exp2(e - 3)  # 3 mantissa bits; subnormal grid 2^-9 below 2^-6
    return (0.5 * ulp + r * 2.0 ** -24) * s64


def test_1x128_invariants(acts):
    x = acts
    M, K = x.shape
    xb = _bits(x)
    xq, sx = oracle.quant_act_1x128(xb)
    x64 = x.double().numpy()
    s64 = np.repeat(sx.T.astype(np.float64), 128, axis=1)
    dq = oracle.e4m3_decode(xq) * s64
    # |x / s| <= 448 after saturation, and dequantisation error within half an ulp
    assert np.all(np.abs(oracle.e4m3_decode(xq)) <= 448)
    assert np.all(np.abs(dq - x64) <= _dequant_bound(x64, xq, s64))
    # scale is fl32(amax / 448) of each group
    amax = np.abs(x64.reshape(M, K // 128, 128)).max(axis=2).astype(np.float32)
    np.testing.assert_array_equal(sx.T, amax / np.float32(448))
    # the element holding the amax encodes to the largest finite magnitude
    grp = np.abs(x64.reshape(M, K // 128, 128))
    arg = grp.argmax(axis=2)
    codes = xq.reshape(M, K // 128, 128)
    top = np.take_along_axis(codes, arg[..., None], axis=2)[..., 0]
    assert np.all((top & 0x7F) == 0x7E)
    # sign symmetry
    xq_neg, sx_neg = oracle.quant_act_1x128(_bits(-x))
    np.testing.assert_array_equal(sx_neg, sx)
    np.testing.assert_array_equal(xq_neg, xq ^ 0x80)


def test_power_of_two_equivariance(acts):
    x = acts[:64]
    xq, sx = oracle.quant_act_1x128(_bits(x))
    for j in (-20, -3, 5, 30):
        y = (x.float() * 2.0 ** j).to(torch.bfloat16)  # exact scaling
        assert torch.equal(y.float(), x.float() * 2.0 ** j)
        yq, sy = oracle.quant_act_1x128(_bits(y))
        np.testing.assert_array_equal(yq, xq)
        np.testing.assert_array_equal(sy, sx * np.float32(2.0 ** j))


def test_zero_and_single_element_groups():
    x = torch.zeros(3, 256, dtype=torch.bfloat16)
    x[1, 5] = -3.0
    x[2, 200] = 1e-30
    xq, sx = oracle.quant_act_1x128(_bits(x))
    assert sx[0, 0] == 1.0 and sx[1, 0] == 1.0 and sx[0, 2] == 1.0  # all-zero groups
    assert np.all(xq[0] == 0)
    assert sx[0, 1] == np.float32(3.0) / np.float32(448.0)
    assert xq[1, 5] == 0xFE and np.count_nonzero(xq[1]) == 1
    assert xq[2, 200] == 0x7E


def test_negative_zero_keeps_sign():
    x = torch.zeros(1, 128, dtype=torch.bfloat16)
    x[0, 0] = 100.0
    x[0, 1] = -0.0
    x[0, 2] = -1e-5  # rounds to zero after scaling
    xq, _ = oracle.quant_act_1x128(_bits(x))
    assert xq[0, 1] == 0x80 and xq[0, 2] == 0x80 and xq[0, 3] == 0x00


def test_layout_identities(acts):
    x = acts
    xb = _bits(x)
    # 128x1 of X is the transpose of 1x128 of X^T
    xqT, sxT = oracle.quant_act_128x1(xb)
    tq, ts = oracle.quant_act_1x128(np.ascontiguousarray(xb.T))
    np.testing.assert_array_equal(xqT, tq)
    np.testing.assert_array_equal(sxT, ts)
    # 1x128 is row-local: quantising a gathered set of rows gathers the result
    perm = np.random.default_rng(5).permutation(x.shape[0])[:97]
    xq, sx = oracle.quant_act_1x128(xb)
    gq, gs = oracle.quant_act_1x128(xb[perm])
    np.testing.assert_array_equal(gq, xq[perm])
    np.testing.assert_array_equal(gs, sx[:, perm])
    # 128x128 of W^T is the transpose of 128x128 of W
    g = torch.Generator().manual_seed(13)
    w = _bits(inputs.weight(256, 384, g))
    wq, wqT, sw = oracle.quant_weight_128x128(w)
    vq, vqT, sv = oracle.quant_weight_128x128(np.ascontiguousarray(w.T))
    np.testing.assert_array_equal(vq, wqT)
    np.testing.assert_array_equal(vqT, wq)
    np.testing.assert_array_equal(sv, sw.T)
