"""GPU MoE Wgrad path vs the CPU oracle: per-expert 128x1 quantisation
(fp8_quant_act_128x1_grouped, bit-exact codes, scales and padded offsets) and
the grouped-K Wgrad GEMM (fp8_grouped_gemm_moe_wgrad, FP32 within relative
Frobenius 1e-5 and the elementwise FP32 accumulation bound)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import b_scale_matrix, bits, check_f32, check_f32_elementwise, magnitude, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _quant(x, offsets, E):
    off = torch.from_numpy(np.asarray(offsets, np.int32)).to(DEV)
    T = x.shape[0]
    Tp = fp8fg.padded_tokens(T, E)
    xqT = torch.full((x.shape[1], Tp), 0xEE, dtype=torch.uint8, device=DEV)
    sxT = torch.full((Tp // 128, x.shape[1]), -5.0, dtype=torch.float32, device=DEV)
    xqT, sxT, pofs = fp8fg.fp8_quant_act_128x1_grouped(x.to(DEV), off, E, Tp=Tp, xqT=xqT, sxT=sxT)
    torch.cuda.synchronize()
    return xqT, sxT, pofs


def _check_quant(x, offsets, E):
    xqT, sxT, pofs = _quant(x, offsets, E)
    rq, rs, rpofs = oracle.quant_act_128x1_grouped(bits(x), offsets)
    P = int(rpofs[-1])
    assert pofs.cpu().numpy().tolist() == rpofs.tolist()
    got_q = xqT.cpu().numpy()
    assert np.array_equal(got_q[:, :P], rq)
    assert np.all(got_q[:, P:] == 0xEE)  # past the last expert: untouched
    got_s = sxT.cpu().numpy()
    assert np.array_equal(got_s[:P // 128].view(np.uint32), rs.view(np.uint32))
    return xqT, sxT, pofs, rq, rs, rpofs


def _compare_wgrad(dw, rq, rs, rdq, rds, pofs, rows):
    ref = oracle.grouped_wgrad(rq, rs, rdq, rds, pofs, rows=rows)
    got = dw.cpu().numpy()[:, rows]
    E = ref.shape[0]
    for e in range(E):
        lo, hi = int(pofs[e]), int(pofs[e + 1])
        if hi == lo:
            assert np.all(got[e] == 0)
            continue
        check_f32(got[e], ref[e])
        a, sa = rq[:, lo:hi], rs[lo // 128:hi // 128]
        b, sb = rdq[:, lo:hi], rds[lo // 128:hi // 128]
        sbm = b_scale_matrix(sb, oracle.BSCALE_ROW1x128, b.shape[0], hi - lo)
        S = lambda idx, a=a, sa=sa, b=b, sbm=sbm: magnitude(a, sa, b, sbm, rows[idx])
        check_f32_elementwise(got[e], ref[e], hi - lo, S)


@pytest.mark.parametrize("counts", [[3, 0, 130, 1], [128, 256], [0, 0, 1], [257, 5, 0, 300]])
def test_grouped_128x1_quantiser(counts):
    g = torch.Generator().manual_seed(sum(counts) + 3)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    T = int(offsets[-1])
    x = inputs.act(max(T, 1), 384, g)[:T]
    _check_quant(x, offsets, len(counts))


@pytest.mark.parametrize("counts", [[3, 0, 130, 1], [257, 5, 0, 300], [0, 0]])
def test_grouped_wgrad_small(counts):
    g = torch.Generator().manual_seed(7 * sum(counts) + 1)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    T, M, N, E = int(offsets[-1]), 256, 384, len(counts)
    x = inputs.act(max(T, 1), M, g)[:T]
    dy = inputs.grad(max(T, 1), N, g)[:T]
    xqT, sxT, pofs, rq, rs, rpofs = _check_quant(x, offsets, E)
    dqT, sdT, _, rdq, rds, _ = _check_quant(dy, offsets, E)
    dw = torch.full((E, M, N), 9.0, dtype=torch.float32, device=DEV)
    fp8fg.fp8_grouped_gemm_moe_wgrad(xqT, sxT, dqT, sdT, pofs, c=dw)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    _compare_wgrad(dw, rq, rs, rdq, rds, rpofs, np.arange(M))


def test_bad_padded_offsets_reported_on_device():
    M, N, Tp, E = 128, 128, 256, 2
    aq = torch.zeros((M, Tp), dtype=torch.uint8, device=DEV)
    bq = torch.zeros((N, Tp), dtype=torch.uint8, device=DEV)
    sa = torch.ones((Tp // 128, M), device=DEV)
    sb = torch.ones((Tp // 128, N), device=DEV)
    pofs = torch.tensor([0, 100, 256], dtype=torch.int32, device=DEV)  # not a multiple of 128
    dw = torch.full((E, M, N), 9.0, dtype=torch.float32, device=DEV)
    fp8fg.fp8_grouped_gemm_moe_wgrad(aq, sa, bq, sb, pofs, c=dw)
    assert fp8fg.device_error() == 7  # FP8_ERR_DEVICE_SHAPE
    assert bool((dw == 9.0).all())


def test_moe_prefill_wgrad_workload():
    """The prefill routing's Wgrad: X [7893, 7168], dY [7893, 4096] -> dW [32, 7168, 4096]."""
    wl = inputs.moe_prefill()
    T = int(wl.offsets[-1])
    dy = inputs.grad(T, wl.N, torch.Generator().manual_seed(10))
    xqT, sxT, pofs, rq, rs, rpofs = _check_quant(wl.x, wl.offsets, wl.E)
    dqT, sdT, _, rdq, rds, _ = _check_quant(dy, wl.offsets, wl.E)
    dw = fp8fg.fp8_grouped_gemm_moe_wgrad(xqT, sxT, dqT, sdT, pofs)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    # 1024 rows of every expert's dW, including the first and last row of every 128-row M tile
    _compare_wgrad(dw, rq, rs, rdq, rds, rpofs, sample_rows(wl.K, 1024, seed=12))


def test_full_width_two_experts():
    """dW [2, 7168, 4096] from 700 + 300 tokens (ragged groups in both experts)."""
    g = torch.Generator().manual_seed(11)
    counts = [700, 300]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    T, M, N, E = int(offsets[-1]), 7168, 4096, 2
    x = inputs.act(T, M, g)
    dy = inputs.grad(T, N, g)
    xqT, sxT, pofs, rq, rs, rpofs = _check_quant(x, offsets, E)
    dqT, sdT, _, rdq, rds, _ = _check_quant(dy, offsets, E)
    dw = fp8fg.fp8_grouped_gemm_moe_wgrad(xqT, sxT, dqT, sdT, pofs)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    _compare_wgrad(dw, rq, rs, rdq, rds, rpofs, sample_rows(M, 1024, seed=13))
