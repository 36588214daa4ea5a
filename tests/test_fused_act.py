"""GEMMs with the 1x128 activation quantisation fused in (A read as bfloat16
and quantised inside the kernel): bitwise equal to the two-step path
fp8_quant_act_1x128 -> fp8_gemm_blockscaled / fp8_grouped_gemm_moe, which is
itself checked against the oracle; the decode workload is also compared with
the oracle directly, every row."""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import bits, group_rows
from test_grouped_parity import _compare, _quant_experts

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _weights(K, N, g, bmode):
    w = inputs.weight(K, N, g).to(DEV)
    if bmode == fp8fg.FP8_BSCALE_BLOCK128:
        wq, _, sw = fp8fg.fp8_quant_weight_128x128(w)
        return wq, sw
    # Dgrad layout: B = wqT [K_w][N_w] codes with the weight scales read transposed
    _, wqT, sw = fp8fg.fp8_quant_weight_128x128(w, want_wq=False, want_wqT=True)
    return wqT, sw


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (37, 256, 384), (130, 512, 1024),
                                   (300, 768, 256), (1024, 1024, 2048)])
def test_dense_equals_two_step(M, N, K, out_dtype):
    g = torch.Generator().manual_seed(M + N + K)
    x = inputs.act(M, K, g).to(DEV)
    wq, sw = _weights(K, N, g, fp8fg.FP8_BSCALE_BLOCK128)
    y = fp8fg.fp8_gemm_blockscaled_bf16a(x, wq, sw, out_dtype=out_dtype)
    xq, sx = fp8fg.fp8_quant_act_1x128(x)
    ref = fp8fg.fp8_gemm_blockscaled(xq, sx, wq, sw, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    assert torch.equal(y.view(torch.int16) if out_dtype == torch.bfloat16 else y.view(torch.int32),
                       ref.view(torch.int16) if out_dtype == torch.bfloat16 else ref.view(torch.int32))


def test_dense_dgrad_layout_and_strided_input():
    g = torch.Generator().manual_seed(9)
    M, K_w, N_w = 200, 512, 768          # Dgrad: dY [M, N_w] . W^T -> [M, K_w]
    w = inputs.weight(K_w, N_w, g).to(DEV)
    _, wqT, sw = fp8fg.fp8_quant_weight_128x128(w, want_wq=False, want_wqT=True)
    dy_full = inputs.grad(M, N_w + 64, g).to(DEV)
    dy = dy_full[:, 32:32 + N_w]         # row stride N_w + 64
    y = fp8fg.fp8_gemm_blockscaled_bf16a(dy, wqT, sw, bmode=fp8fg.FP8_BSCALE_BLOCK128_T)
    dq, sd = fp8fg.fp8_quant_act_1x128(dy)
    ref = fp8fg.fp8_gemm_blockscaled(dq, sd, wqT, sw, bmode=fp8fg.FP8_BSCALE_BLOCK128_T)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("counts", [[3, 0, 130, 1], [128, 256, 127], [0, 0, 1], [300, 0]])
def test_grouped_equals_two_step(counts):
    g = torch.Generator().manual_seed(sum(counts) + 5)
    E, K, N = len(counts), 384, 512
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offsets[-1])
    x = inputs.act(max(T, 1), K, g)[:T].to(DEV)
    w = torch.stack([inputs.weight(K, N, g) for _ in range(E)]).to(DEV)
    wq = torch.empty((E, N, K), dtype=torch.uint8, device=DEV)
    sw = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=DEV)
    for e in range(E):
        fp8fg.fp8_quant_weight_128x128(w[e], wq=wq[e], sw=sw[e])
    off = torch.from_numpy(offsets).to(DEV)
    y = torch.full((T, N), 7.0, dtype=torch.bfloat16, device=DEV)
    fp8fg.fp8_grouped_gemm_moe_bf16a(x, wq, sw, off, c=y)
    xq, sx = fp8fg.fp8_quant_act_1x128(x)
    ref = torch.full((T, N), 7.0, dtype=torch.bfloat16, device=DEV)
    fp8fg.fp8_grouped_gemm_moe(xq, sx, wq, sw, off, c=ref)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def test_decode_workload_against_the_oracle():
    """32 experts with 1-256 rows: bitwise the two-step path, and every row within
    the BF16 tolerance of the oracle."""
    wl = inputs.moe_decode()
    x = wl.x.to(DEV)
    bq, sb = _quant_experts(wl.w)                       # the oracle's weight codes
    bq_d, sb_d = torch.from_numpy(bq).to(DEV), torch.from_numpy(sb).to(DEV)
    off = torch.from_numpy(np.asarray(wl.offsets, np.int32)).to(DEV)
    y = fp8fg.fp8_grouped_gemm_moe_bf16a(x, bq_d, sb_d, off)
    xq, sx = fp8fg.fp8_quant_act_1x128(x)
    ref = fp8fg.fp8_grouped_gemm_moe(xq, sx, bq_d, sb_d, off)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    aq, sa = oracle.quant_act_1x128(bits(wl.x))
    _compare(y, aq, sa, bq, sb, wl.offsets, np.arange(int(wl.offsets[-1])))
