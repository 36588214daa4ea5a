"""GPU block-scaled FP8 GEMM vs the CPU oracle.

Bars: FP32 output within relative Frobenius error 1e-5 of the oracle's
binary64 result; BF16 output within 1 bfloat16 ulp of RNE_bf16(fl32(C)) per
element (see parity.check_bf16 for the cancellation reading).  Operand codes
and scales are produced by the oracle and uploaded, so the GEMM is tested in
isolation; the end-to-end test quantises on the GPU instead.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import (b_scale_matrix, bits, check_bf16, check_f32, check_f32_elementwise,
                    magnitude, np_u8, sample_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _operands(M, N, K, bmode, seed):
    """Oracle-quantised A [M,K] (1x128) and B [N,K] per bmode."""
    g = _gen(seed)
    x = inputs.act(M, K, g)
    aq, sa = oracle.quant_act_1x128(bits(x))
    if bmode == oracle.BSCALE_ROW1x128:
        b = inputs.grad(N, K, g)
        bq, sb = oracle.quant_act_1x128(bits(b))
    else:
        w = inputs.weight(K, N, g)
        bq, _, sw = oracle.quant_weight_128x128(bits(w))
        sb = sw if bmode == oracle.BSCALE_BLOCK128 else np.ascontiguousarray(sw.T)
    return aq, sa, bq, sb


def _run(aq, sa, bq, sb, bmode, out_dtype, c=None):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    out = fp8fg.fp8_gemm_blockscaled(t(aq), t(sa), t(bq), t(sb), bmode=bmode,
                                     out_dtype=out_dtype, c=c)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    return out


def _compare(out, aq, sa, bq, sb, bmode, rows=None):
    """Every requested row (default: all), elementwise against the oracle."""
    M, K = aq.shape
    N = bq.shape[0]
    rows = np.arange(M) if rows is None else rows
    ref = oracle.gemm_blockscaled(aq, sa, bq, sb, bmode, rows=rows)
    o = out.cpu()
    sbm = b_scale_matrix(sb, bmode, N, K)
    S = lambda idx: magnitude(aq, sa, bq, sbm, rows[idx])  # formed only where needed
    if o.dtype == torch.float32:
        got = o.numpy()[rows]
        check_f32(got, ref)
        check_f32_elementwise(got, ref, K, S)
        return 0
    return check_bf16(o.view(torch.int16).numpy().view(np.uint16)[rows], ref, S=S, K=K)


def test_small_fp32_workload():
    """M=128, N=256, K=512 with outlier-channel activations; FP32 output."""
    wl = inputs.small_dense()
    aq, sa = oracle.quant_act_1x128(bits(wl.x))
    bq, _, sw = oracle.quant_weight_128x128(bits(wl.w))
    out = _run(aq, sa, bq, sw, 0, torch.float32)
    _compare(out, aq, sa, bq, sw, 0)


# N % 256 == 0 runs the dense kernel on CTA pairs when there is more than one
# 128-row block: (257, 512, 384) gives a pair whose second CTA has no valid
# row, (640, 768, 256) an odd number of 128-row blocks; (1, 256, 128), a
# single row block, runs one CTA per 128 x 128 tile.
SHAPES = [(1, 128, 128), (37, 384, 256), (130, 256, 1024), (257, 512, 384), (300, 640, 128),
          (1, 256, 128), (640, 768, 256)]


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("bmode", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_shapes(M, N, K, bmode, out_dtype):
    aq, sa, bq, sb = _operands(M, N, K, bmode, seed=M + N + K + bmode)
    out = _run(aq, sa, bq, sb, bmode, out_dtype)
    _compare(out, aq, sa, bq, sb, bmode)


@pytest.mark.parametrize("bmode", [0, 1, 2])
def test_clusters_walk_many_tiles(bmode):
    """More cluster tiles than clusters fit on the GPU (each cluster walks
    several), a ragged last row block: rows sampled from every row block."""
    M, N, K = 4096 + 128 + 5, 1024, 256
    aq, sa, bq, sb = _operands(M, N, K, bmode, seed=90 + bmode)
    out = _run(aq, sa, bq, sb, bmode, torch.float32)
    _compare(out, aq, sa, bq, sb, bmode, rows=sample_rows(M, 256, seed=bmode))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_output_stride_and_canaries(out_dtype):
    M, N, K = 70, 256, 256
    aq, sa, bq, sb = _operands(M, N, K, 0, seed=77)
    buf = torch.full((M + 5, N + 64), -7.0, dtype=out_dtype, device=DEV)
    c = buf[:M, 32:32 + N]
    _run(aq, sa, bq, sb, 0, out_dtype, c=c)
    _compare(c, aq, sa, bq, sb, 0)
    b = buf.cpu().float()
    assert (b[:, :32] == -7).all() and (b[:, 32 + N:] == -7).all() and (b[M:] == -7).all()


def test_repeated_calls_identical():
    aq, sa, bq, sb = _operands(256, 512, 512, 0, seed=5)
    o1 = _run(aq, sa, bq, sb, 0, torch.float32)
    o2 = _run(aq, sa, bq, sb, 0, torch.float32)
    assert torch.equal(o1, o2)


def test_end_to_end_quantise_then_gemm():
    """GPU quantisers feeding the GPU GEMM vs oracle quantisers feeding the oracle GEMM."""
    g = _gen(21)
    M, K, N = 200, 768, 512
    x, w = inputs.act(M, K, g), inputs.weight(K, N, g)
    xq, sx = fp8fg.fp8_quant_act_1x128(x.to(DEV))
    wq, _, sw = fp8fg.fp8_quant_weight_128x128(w.to(DEV))
    y = fp8fg.fp8_gemm_blockscaled(xq, sx, wq, sw, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    aq, sa = oracle.quant_act_1x128(bits(x))
    bq, _, sb = oracle.quant_weight_128x128(bits(w))
    _compare(y, aq, sa, bq, sb, 0)


def test_full_size_fprop_dense():
    """X[8192, 2048] . W[2048, 7168] -> BF16: every row against the oracle."""
    wl = inputs.fprop_dense()
    aq, sa = oracle.quant_act_1x128(bits(wl.x))
    bq, _, sw = oracle.quant_weight_128x128(bits(wl.w))
    out = _run(aq, sa, bq, sw, 0, torch.bfloat16)
    _compare(out, aq, sa, bq, sw, 0)


def test_full_size_training_trio():
    """Fprop X.W, Dgrad dY.W^T (transposed block scales), Wgrad X^T.dY (row
    scales), each on 1024 rows that include the first and last row of every
    128-row M tile; every column (so every N block) of those rows."""
    wl = inputs.training_trio()
    xb, wb, dyb = bits(wl.x), bits(wl.w), bits(wl.dy)
    wq, wqT, sw = oracle.quant_weight_128x128(wb)
    # Fprop: [8192, 7168] . [7168, 4096] -> BF16
    aq, sa = oracle.quant_act_1x128(xb)
    out = _run(aq, sa, wq, sw, 0, torch.bfloat16)
    _compare(out, aq, sa, wq, sw, 0, rows=sample_rows(wl.M, 1024, seed=2))
    del aq, sa, out
    # Dgrad: dY [8192, 4096] . W^T -> dX [8192, 7168] BF16; B = W [7168, 4096] K-major
    dq, sd = oracle.quant_act_1x128(dyb)
    # sw is [N_out/128][K_hidden/128] = [K'/128][N'/128] of this GEMM: the BLOCK128_T layout
    out = _run(dq, sd, wqT, sw, 2, torch.bfloat16)
    _compare(out, dq, sd, wqT, sw, 2, rows=sample_rows(wl.M, 1024, seed=3))
    del dq, sd, out
    # Wgrad: X^T [7168, 8192] . dY [8192, 4096] -> dW FP32; both operands 128x1
    xqT, sxT = oracle.quant_act_128x1(xb)
    dqT, sdT = oracle.quant_act_128x1(dyb)
    out = _run(xqT, sxT, dqT, sdT, 1, torch.float32)
    _compare(out, xqT, sxT, dqT, sdT, 1, rows=sample_rows(wl.K, 1024, seed=4))

