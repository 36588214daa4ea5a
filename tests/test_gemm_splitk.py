"""fp8_gemm_blockscaled_ws: the split-K tail of the dense CTA-pair kernels.

Shapes whose last wave of 256 x 256 tiles leaves at least half of the SM
pairs idle, with at least 48 K blocks, get that wave's tiles cut along K and
reduced in chunk order.
Checked against the oracle (same bars as test_gemm_parity: the chunk sum is
another FP32 rounding order within the same error bound), bitwise repeatable,
and leaving the workspace's counters zero.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import bits, sample_rows
from test_gemm_parity import _compare, _operands

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ws():
    return torch.zeros(fp8fg.fp8_gemm_blockscaled_workspace_size(), dtype=torch.uint8, device=DEV)


def _pairs():
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


def _run(aq, sa, bq, sb, bmode, out_dtype, ws):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    out = fp8fg.fp8_gemm_blockscaled(t(aq), t(sa), t(bq), t(sb), bmode=bmode, out_dtype=out_dtype,
                                     workspace=ws)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    return out


@pytest.mark.parametrize("bmode,out_dtype", [(1, torch.float32), (0, torch.bfloat16),
                                             (2, torch.float32)])
def test_tail_split_matches_oracle_and_repeats(bmode, out_dtype):
    # one 256-row pair block with ragged rows, pairs + 2 column tiles: two
    # tail tiles split along K (48 K blocks: the shallowest that splits)
    M, N, K = 256 - 37, 256 * (_pairs() + 2), 6144
    aq, sa, bq, sb = _operands(M, N, K, bmode, seed=300 + bmode)
    ws = _ws()
    o1 = _run(aq, sa, bq, sb, bmode, out_dtype, ws)
    _compare(o1, aq, sa, bq, sb, bmode)
    o2 = _run(aq, sa, bq, sb, bmode, out_dtype, ws)
    assert torch.equal(o1.view(torch.int16) if out_dtype == torch.bfloat16 else o1.view(torch.int32),
                       o2.view(torch.int16) if out_dtype == torch.bfloat16 else o2.view(torch.int32))
    assert int(ws[:4096].view(torch.int32).abs().sum()) == 0  # counters back to zero


def test_split_and_unsplit_agree_within_bounds():
    """The same GEMM with and without the workspace: identical outside the
    tail tiles (the whole tiles run the same code), the tail within bounds."""
    M, N, K = 256, 256 * (_pairs() + 1), 8192
    aq, sa, bq, sb = _operands(M, N, K, 1, seed=77)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    plain = fp8fg.fp8_gemm_blockscaled(t(aq), t(sa), t(bq), t(sb), bmode=1, out_dtype=torch.float32)
    split = fp8fg.fp8_gemm_blockscaled(t(aq), t(sa), t(bq), t(sb), bmode=1, out_dtype=torch.float32,
                                       workspace=_ws())
    torch.cuda.synchronize()
    full_cols = 256 * _pairs()
    assert torch.equal(plain[:, :full_cols], split[:, :full_cols])
    assert not torch.equal(plain[:, full_cols:], split[:, full_cols:])  # the tail was split
    _compare(split, aq, sa, bq, sb, 1, rows=sample_rows(M, 64, seed=3))


def test_full_size_trio_dgrad_and_wgrad_with_workspace():
    """The trio's Dgrad (896 tiles) and Wgrad (448 tiles) both end in a short
    wave on 74 pairs; rows sampled from every row block, every column."""
    wl = inputs.training_trio()
    xb, wb, dyb = bits(wl.x), bits(wl.w), bits(wl.dy)
    ws = _ws()
    # Dgrad: dY [M, N] . W^T -> [M, K]
    dq, sd = oracle.quant_act_1x128(dyb)
    _, wqT, sw = oracle.quant_weight_128x128(wb)
    # BLOCK128_T reads the Fprop weight scales sw [N/128][K/128] as they are
    out = _run(dq, sd, wqT, sw, 2, torch.bfloat16, ws)
    _compare(out, dq, sd, wqT, sw, 2, rows=sample_rows(wl.M, 256, seed=1))
    # Wgrad: X^T [K, M] . dY -> [K, N]
    xqT, sxT = oracle.quant_act_128x1(xb)
    dqT, sdT = oracle.quant_act_128x1(dyb)
    out = _run(xqT, sxT, dqT, sdT, 1, torch.float32, ws)
    _compare(out, xqT, sxT, dqT, sdT, 1, rows=sample_rows(wl.K, 256, seed=2))
    assert int(ws[:4096].view(torch.int32).abs().sum()) == 0


def test_workspace_errors():
    aq = torch.zeros((256, 256), dtype=torch.uint8, device=DEV)
    sa = torch.ones((2, 256), dtype=torch.float32, device=DEV)
    bq = torch.zeros((256, 256), dtype=torch.uint8, device=DEV)
    sb = torch.ones((2, 2), dtype=torch.float32, device=DEV)
    small = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    with pytest.raises(fp8fg.Fp8Error) as e:
        fp8fg.fp8_gemm_blockscaled(aq, sa, bq, sb, workspace=small)
    assert e.value.status == 2  # FP8_ERR_SHAPE
    ws = _ws()
    with pytest.raises(fp8fg.Fp8Error) as e:
        fp8fg.fp8_gemm_blockscaled(aq, sa, bq, sb, workspace=ws[8:])
    assert e.value.status == 3  # FP8_ERR_ALIGN
