"""GPU grouped (per-expert) FP8 GEMM vs the CPU oracle.

Covers empty experts, single-token experts, experts spanning several 128-row
tiles with ragged tails, the prefill routing workload (top-8 of 256 experts,
32 local, skewed) and the decode workload (1-256 tokens per expert), plus the
device-side offset validation.
"""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import (bits, check_bf16, check_f32, check_f32_elementwise, group_rows, magnitude,
                    np_u8)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _quant_experts(w):
    """Oracle 128x128 quantisation of each expert weight [E, K, N] (threads over experts)."""
    E = w.shape[0]
    wb = [bits(w[e]) for e in range(E)]
    with cf.ThreadPoolExecutor(8) as ex:
        res = list(ex.map(lambda b: oracle.quant_weight_128x128(b), wb))
    bq = np.stack([r[0] for r in res])
    sb = np.stack([r[2] for r in res])
    return bq, sb


def _run(aq, sa, bq, sb, offsets, out_dtype, c=None):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    off = torch.from_numpy(np.asarray(offsets, np.int32)).to(DEV)
    out = fp8fg.fp8_grouped_gemm_moe(t(aq), t(sa), t(bq), t(sb), off, out_dtype=out_dtype, c=c)
    torch.cuda.synchronize()
    return out


def _compare(out, aq, sa, bq, sb, offsets, rows, bmode=oracle.BSCALE_BLOCK128):
    """The requested rows, elementwise, each against its expert's oracle product."""
    ref = oracle.grouped_gemm(aq, sa, bq, sb, offsets, rows=rows, bmode=bmode)
    K = aq.shape[1]
    expert_of = np.searchsorted(offsets, rows, side="right") - 1
    o = out.cpu()
    n_fallback = 0
    for e in np.unique(expert_of):
        sel = np.nonzero(expert_of == e)[0]
        sbe = sb[e] if bmode == oracle.BSCALE_BLOCK128 else sb[e].T
        sbm = np.repeat(sbe, 128, axis=0)  # [N, K/128]
        S = lambda idx, e=e, sel=sel, sbm=sbm: magnitude(aq, sa, bq[e], sbm, rows[sel][idx])
        if o.dtype == torch.float32:
            got = o.numpy()[rows[sel]]
            check_f32(got, ref[sel])
            check_f32_elementwise(got, ref[sel], K, S)
        else:
            n_fallback += check_bf16(o.view(torch.int16).numpy().view(np.uint16)[rows[sel]],
                                     ref[sel], S=S, K=K)
    return n_fallback


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("counts", [[3, 0, 130, 1], [0, 0, 1], [128, 256, 127, 129, 5],
                                    [0, 300, 0],
                                    # fewer than 192 rows per expert on average: one CTA
                                    # per 128-row tile, experts ending on and around
                                    # tile edges and one spanning three tiles
                                    [16, 17, 33, 64, 65, 255, 257],
                                    # 192+ rows per expert on average, N = 256: CTA pairs
                                    # over 256-row blocks (ragged second halves, a
                                    # one-row expert, an empty one)
                                    [300, 0, 450], [1, 600, 7]])
def test_grouped_small(counts, out_dtype):
    g = torch.Generator().manual_seed(sum(counts) + len(counts))
    E, K, N = len(counts), 384, 256 if len(counts) % 2 else 384
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    T = int(offsets[-1])
    x = inputs.act(max(T, 1), K, g)[:T]
    w = torch.stack([inputs.weight(K, N, g) for _ in range(E)])
    aq, sa = oracle.quant_act_1x128(bits(x)) if T else (np.zeros((0, K), np.uint8),
                                                         np.zeros((K // 128, 0), np.float32))
    bq, sb = _quant_experts(w)
    c = torch.full((T, N), 3.0, dtype=out_dtype, device=DEV)
    _run(aq, sa, bq, sb, offsets, out_dtype, c=c)
    assert fp8fg.device_error() == 0
    if T:
        _compare(c, aq, sa, bq, sb, offsets, np.arange(T))


def test_uncovered_rows_untouched():
    """Rows past offsets[E] (< T) are not written."""
    g = torch.Generator().manual_seed(3)
    K, N, T = 256, 256, 200
    offsets = np.array([0, 70, 150])
    x = inputs.act(T, K, g)
    w = torch.stack([inputs.weight(K, N, g) for _ in range(2)])
    aq, sa = oracle.quant_act_1x128(bits(x))
    bq, sb = _quant_experts(w)
    c = torch.full((T, N), 5.0, dtype=torch.bfloat16, device=DEV)
    _run(aq, sa, bq, sb, offsets, torch.bfloat16, c=c)
    assert (c[150:].float() == 5.0).all()
    _compare(c, aq, sa, bq, sb, offsets, np.arange(150))


def test_bad_offsets_reported_on_device():
    K, N = 128, 128
    aq = np.zeros((64, K), np.uint8)
    sa = np.ones((1, 64), np.float32)
    bq = np.zeros((2, N, K), np.uint8)
    sb = np.ones((2, 1, 1), np.float32)
    c = torch.full((64, N), 9.0, dtype=torch.float32, device=DEV)
    _run(aq, sa, bq, sb, [0, 40, 30], torch.float32, c=c)  # decreasing
    assert fp8fg.device_error() == 7  # FP8_ERR_DEVICE_SHAPE
    assert (c == 9.0).all()
    _run(aq, sa, bq, sb, [0, 10, 65], torch.float32, c=c)  # beyond T
    assert fp8fg.device_error() == 7
    assert fp8fg.device_error() == 0  # cleared


def _workload_parity(wl, n_rows):
    """Grouped GEMM of a routing workload; rows: the first and last row of
    every expert and of every 128-row tile inside it, plus random rows up to
    n_rows (all rows when n_rows >= the row count)."""
    xb = bits(wl.x)
    aq, sa = oracle.quant_act_1x128(xb)
    bq, sb = _quant_experts(wl.w)
    out = _run(aq, sa, bq, sb, wl.offsets, torch.bfloat16)
    assert fp8fg.device_error() == 0
    rows = group_rows(wl.offsets, n_rows, seed=0)
    return _compare(out, aq, sa, bq, sb, wl.offsets, rows)


def test_moe_prefill_workload():
    """Top-8 of 256 routing, 32 local experts: 1024 rows covering every expert and tile edge."""
    wl = inputs.moe_prefill()
    counts = np.diff(wl.offsets)
    # the biased routing is skewed: empty experts next to experts with thousands of rows
    assert counts.min() == 0 and counts.max() > 1000
    _workload_parity(wl, 1024)


def test_moe_decode_workload():
    """1-256 tokens per expert, 32 experts: every row against the oracle."""
    wl = inputs.moe_decode()
    counts = np.diff(wl.offsets)
    assert counts.min() >= 1 and counts.max() <= 256
    _workload_parity(wl, int(wl.offsets[-1]))


def _quant_experts_T(w):
    """Oracle 128x128 quantisation of each expert weight: (wqT [E, K, N], sw [E, N/128, K/128])."""
    E = w.shape[0]
    wb = [bits(w[e]) for e in range(E)]
    with cf.ThreadPoolExecutor(8) as ex:
        res = list(ex.map(lambda b: oracle.quant_weight_128x128(b), wb))
    return np.stack([r[1] for r in res]), np.stack([r[2] for r in res])


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("counts", [[3, 0, 130, 1], [257, 0, 5], [0, 1]])
def test_grouped_dgrad_small(counts, out_dtype):
    """dX_e = dY_e . W_e^T with each expert's wqT codes and sw scales read transposed."""
    g = torch.Generator().manual_seed(7 * sum(counts) + len(counts))
    E, Kf, Nf = len(counts), 384, 256 if len(counts) % 2 else 512
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    T = int(offsets[-1])
    dy = inputs.grad(max(T, 1), Nf, g)[:T]
    w = torch.stack([inputs.weight(Kf, Nf, g) for _ in range(E)])
    dq, sd = oracle.quant_act_1x128(bits(dy))
    bqT, sw = _quant_experts_T(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    off = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    dx = fp8fg.fp8_grouped_gemm_moe_dgrad(t(dq), t(sd), t(bqT), t(sw), off, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    _compare(dx, dq, sd, bqT, sw, offsets, np.arange(T), bmode=oracle.BSCALE_BLOCK128_T)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_grouped_dgrad_pairs(out_dtype):
    """Dgrad with 512 output columns and 250 rows per expert: the CTA-pair path."""
    counts = [300, 0, 450]
    g = torch.Generator().manual_seed(41)
    E, Kf, Nf = len(counts), 512, 256
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    T = int(offsets[-1])
    dy = inputs.grad(T, Nf, g)
    w = torch.stack([inputs.weight(Kf, Nf, g) for _ in range(E)])
    dq, sd = oracle.quant_act_1x128(bits(dy))
    bqT, sw = _quant_experts_T(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    off = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    dx = fp8fg.fp8_grouped_gemm_moe_dgrad(t(dq), t(sd), t(bqT), t(sw), off, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    _compare(dx, dq, sd, bqT, sw, offsets, np.arange(T), bmode=oracle.BSCALE_BLOCK128_T)


def test_moe_prefill_dgrad_workload():
    """The prefill routing's backward: dY [rows, 4096] -> dX [rows, 7168] per expert."""
    wl = inputs.moe_prefill()
    T = int(wl.offsets[-1])
    dy = inputs.grad(T, wl.N, torch.Generator().manual_seed(8))
    dq, sd = oracle.quant_act_1x128(bits(dy))
    bqT, sw = _quant_experts_T(wl.w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    off = torch.from_numpy(np.asarray(wl.offsets, np.int32)).to(DEV)
    dx = fp8fg.fp8_grouped_gemm_moe_dgrad(t(dq), t(sd), t(bqT), t(sw), off)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    rows = group_rows(wl.offsets, 1024, seed=9)
    _compare(dx, dq, sd, bqT, sw, np.asarray(wl.offsets), rows, bmode=oracle.BSCALE_BLOCK128_T)
