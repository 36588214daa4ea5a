"""GPU E5M6 quantiser (fp8_quant_act_1x128_e5m6) vs the CPU oracle: packed
codes and scales bit-exact, at small ragged sizes, the training trio's
activation size, strided input and output, and the degenerate groups; and an
exhaustive check of the arithmetic over every bfloat16 (x, amax) pair against
IEEE division followed by an E5M6 rounding written with PyTorch operations."""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import bits, np_u8
from test_quant_parity import _edge_matrix

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _assert(x):
    xq, sx = fp8fg.fp8_quant_act_1x128_e5m6(x.to(DEV))
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_act_1x128_e5m6(bits(x))
    np.testing.assert_array_equal(np_u8(xq), oracle.pack_e5m6(oq))
    np.testing.assert_array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    return xq


@pytest.mark.parametrize("M,K", [(1, 128), (63, 256), (65, 384), (130, 1024), (1000, 640)])
def test_small(M, K):
    _assert(inputs.act(M, K, torch.Generator().manual_seed(M + 3 * K)))


def test_trio_activation_size():
    _assert(inputs.act(8192, 7168, torch.Generator().manual_seed(17)))


def test_edge_groups():
    x = _edge_matrix()
    xq = _assert(x)
    codes = oracle.unpack_e5m6(np_u8(xq))
    assert codes[1, 0] == 0x800 and codes[0, 0] == 0x000
    assert codes[2, 7] == 0xFBF  # the group's amax element encodes to -65024
    # -1e-6 against an amax of 3: |x / s| ~ 0.02, a normal E5M6 value (E4M3 gives -0)
    assert codes[2, 8] & 0x800 and codes[2, 8] != 0x800


def test_strided_input_and_output():
    x_full = inputs.act(100, 512 + 24, torch.Generator().manual_seed(4))
    x = x_full.to(DEV)[:, 8:8 + 512]
    buf = torch.full((100, 768 + 64), 0xAB, dtype=torch.uint8, device=DEV)
    xq, sx = fp8fg.fp8_quant_act_1x128_e5m6(x, xq=buf[:, 32:32 + 768])
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_act_1x128_e5m6(bits(x_full[:, 8:8 + 512].contiguous()))
    np.testing.assert_array_equal(np_u8(buf[:, 32:32 + 768]), oracle.pack_e5m6(oq))
    np.testing.assert_array_equal(sx.cpu().numpy(), os_)
    assert (np_u8(buf[:, :32]) == 0xAB).all() and (np_u8(buf[:, 800:]) == 0xAB).all()


def _torch_e5m6(q):
    """E5M6 codes of binary32 values with PyTorch operations (frexp/round),
    independent of the library's integer rounding."""
    a = q.abs()
    neg = torch.signbit(q).to(torch.int32) << 11
    m_sub = torch.round(a * 2.0 ** 20).to(torch.int32)          # ties to even
    fr, ex = torch.frexp(a)                                      # a = fr 2^ex, fr in [0.5, 1)
    m = torch.round((2.0 * fr - 1.0) * 64.0).to(torch.int32)
    e = ex.to(torch.int32) - 1
    carry = m == 64
    m = torch.where(carry, torch.zeros_like(m), m)
    e = e + carry.to(torch.int32)
    m_norm = ((e + 15) << 6) | m
    mag = torch.where(a < 2.0 ** -14, m_sub, m_norm)
    mag = torch.where(a >= 65024.0, torch.full_like(mag, 0x7BF), mag)
    return neg | mag


def _groups(amax_pat):
    """int16 [G, 128] groups: column 0 the amax pattern, then every |x| <= amax."""
    p = amax_pat.to(torch.int64)
    n = p + 1
    ng = (2 * n + 126) // 127
    G = int(ng.sum())
    grp_amax = torch.repeat_interleave(p, ng)
    start = torch.cumsum(ng, 0) - ng
    gi = torch.arange(G, device=DEV) - torch.repeat_interleave(start, ng)
    nn = torch.repeat_interleave(n, ng)[:, None]
    j = (gi[:, None] * 127 + torch.arange(127, device=DEV)[None, :]) % (2 * nn)
    x = (j % nn) | ((j // nn) << 15)
    return torch.cat([grp_amax[:, None], x], 1).to(torch.int32).to(torch.int16)


def _unpack(xq):
    """uint8 [G, 192] -> int32 codes [G, 128] on the device."""
    b = xq.to(torch.int32).view(xq.shape[0], 64, 3)
    c0 = b[:, :, 0] | ((b[:, :, 1] & 0xF) << 8)
    c1 = (b[:, :, 1] >> 4) | (b[:, :, 2] << 4)
    return torch.stack([c0, c1], 2).view(xq.shape[0], 128)


def test_all_bf16_pairs_match_ieee_division():
    amax_all = torch.arange(1, 0x7F80, device=DEV, dtype=torch.int32)
    n_pairs = 0
    for chunk in amax_all.split(192):
        g = _groups(chunk)
        xb = g.view(torch.bfloat16)
        xq, sx = fp8fg.fp8_quant_act_1x128_e5m6(xb)
        xf = xb.float()
        s = xf[:, :1].abs() / torch.tensor(65024.0, device=DEV)
        assert torch.equal(sx[0].view(torch.int32), s[:, 0].view(torch.int32)), "scale mismatch"
        ref = _torch_e5m6(xf / s)
        got = _unpack(xq)
        bad = (got != ref).nonzero()
        if bad.numel():
            i, k = bad[0].tolist()
            pytest.fail("group amax %#06x x %#06x: got %#x want %#x" % (
                g[i, 0].item() & 0xFFFF, g[i, k].item() & 0xFFFF, got[i, k].item(),
                ref[i, k].item()))
        n_pairs += g.shape[0] * 127
    assert n_pairs > 1.0e9
