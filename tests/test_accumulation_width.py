"""How many bits does the tensor core keep while it sums one 128-wide K block?

The DeepSeek-V3 Technical Report (section 3.3.2) observes that the FP8 MMA of
the H800 keeps only about 14 bits of the running sum, which is why partial
sums are promoted to FP32 every N_C = 128 elements.  This diagnostic measures
the same property of the B300 tcgen05 FP8 MMA through the library's GEMM
(scales 1, one K block): one large product 2^e followed by 127 products of
2^-7 each.  The exact block sum 2^e + 127/128 needs e + 7 significant bits;
an accumulator that keeps b bits loses the small terms once e + 7 > b.
The test records the widest e for which the sum is exact, and requires it to
be at least the 24 bits of IEEE binary32 (FP32 accumulation; the promotion
every 128 elements then only guards the cross-block sum).
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_22_b300 import fp8fg

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _e4m3(v):
    return torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).item()


def test_block_sum_keeps_binary32_precision():
    K, N = 128, 128
    # E4M3 pairs whose product is 2^e for e = 0..16 (448 x 448 caps e at 17)
    big = []
    for e in range(0, 17):
        a = 2.0 ** (e // 2)
        b = 2.0 ** (e - e // 2)
        big.append((e, _e4m3(a), _e4m3(b)))
    M = len(big)
    aq = np.zeros((M, K), np.uint8)
    bq = np.zeros((N, K), np.uint8)
    for i, (e, ca, _) in enumerate(big):
        aq[i, 0] = ca
        aq[i, 1:] = _e4m3(0.125)  # 2^-3
    bq[:, 1:] = _e4m3(0.0625)     # 2^-4: each small product is 2^-7
    for n in range(N):
        bq[n, 0] = big[n % M][2]
    sa = np.ones((1, M), np.float32)
    sb = np.ones((1, 1), np.float32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    c = fp8fg.fp8_gemm_blockscaled(t(aq), t(sa), t(bq), t(sb), out_dtype=torch.float32)
    torch.cuda.synchronize()
    got = c.cpu().numpy().astype(np.float64)
    exact_bits = []
    for i, (e, _, _) in enumerate(big):
        n = i  # column whose big B entry pairs with row i's big A entry
        want = 2.0 ** e + 127.0 / 128.0
        exact_bits.append((e + 7, got[i, n] == want))
    widest = max([bits for bits, ok in exact_bits if ok], default=0)
    print("block sums exact up to %d significant bits: %s" % (widest, exact_bits))
    assert all(ok for bits, ok in exact_bits if bits <= 24), exact_bits
