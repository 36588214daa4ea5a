"""Exhaustive check of the quantiser's arithmetic on the GPU.

A 1x128 group's codes depend only on each element x and the group's amax.
For EVERY positive finite bf16 amax and EVERY bf16 x with |x| <= amax (both
signs, including zeros and subnormals) this builds groups [amax, x, x, ...],
quantises them with the library, and compares scales and codes with IEEE
single-precision division followed by PyTorch's float8_e4m3fn conversion
(library routines, independent of this library's kernels).  About 1.07e9
(x, amax) pairs.  A random sample of the groups is also checked against the
CPU oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _groups(amax_pat):
    """int16 [G, 128] groups: column 0 the amax pattern, then every |x| <= amax."""
    p = amax_pat.to(torch.int64)
    n = p + 1                      # magnitudes 0..p
    cnt = 2 * n                    # both signs
    ng = (cnt + 126) // 127
    G = int(ng.sum())
    grp_amax = torch.repeat_interleave(p, ng)
    start = torch.cumsum(ng, 0) - ng
    gi = torch.arange(G, device=DEV) - torch.repeat_interleave(start, ng)
    nn = torch.repeat_interleave(n, ng)[:, None]
    j = (gi[:, None] * 127 + torch.arange(127, device=DEV)[None, :]) % (2 * nn)
    mag = j % nn
    sign = j // nn
    x = mag | (sign << 15)
    out = torch.cat([grp_amax[:, None], x], 1)
    return out.to(torch.int32).to(torch.int16)  # wraps 0x8000.. to negative int16


def test_all_bf16_pairs_match_ieee_division():
    amax_all = torch.arange(1, 0x7F80, device=DEV, dtype=torch.int32)
    rng = np.random.default_rng(0)
    sample = []
    n_pairs = 0
    for chunk in amax_all.split(192):
        g = _groups(chunk)
        xb = g.view(torch.bfloat16)
        xq, sx = fp8fg.fp8_quant_act_1x128(xb)
        xf = xb.float()
        s = xf[:, :1].abs() / torch.tensor(448.0, device=DEV)
        ref = (xf / s).to(torch.float8_e4m3fn).view(torch.uint8)
        assert torch.equal(sx[0].view(torch.int32), s[:, 0].view(torch.int32)), "scale mismatch"
        bad = (xq != ref).nonzero()
        if bad.numel():
            i, k = bad[0].tolist()
            pytest.fail("group amax %#06x x %#06x: got %#x want %#x" % (
                g[i, 0].item() & 0xFFFF, g[i, k].item() & 0xFFFF, xq[i, k].item(), ref[i, k].item()))
        n_pairs += g.shape[0] * 127
        pick = torch.from_numpy(rng.choice(g.shape[0], 8, replace=False)).to(DEV)
        sample.append((g[pick].cpu(), xq[pick].cpu(), sx[0][pick].cpu()))
    assert n_pairs > 1.0e9
    # the same groups through the CPU oracle
    gs = torch.cat([s[0] for s in sample]).numpy().view(np.uint16)
    oq, os_ = oracle.quant_act_1x128(gs)
    np.testing.assert_array_equal(torch.cat([s[1] for s in sample]).numpy(), oq)
    np.testing.assert_array_equal(torch.cat([s[2] for s in sample]).numpy(), os_[0])
