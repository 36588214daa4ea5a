"""GPU MoE dispatch packing (fp8_moe_dispatch_quant) vs the CPU oracle.

Bit-exact: offsets, source token ids, E4M3 codes and scales of every packed
row; rows past the last used one stay untouched.  Then the packed operands
feed the grouped GEMM, compared with the oracle on 1024 rows that include
the first and last row of every expert and of every 128-row tile.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import bits, group_rows
from test_grouped_parity import _compare, _quant_experts as _oracle_weights

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(x, ids, begin, n_local, cap=None, workspace=None):
    xg = x.to(DEV)
    idg = torch.as_tensor(ids, dtype=torch.int32).to(DEV).contiguous()
    T, K = x.shape
    topk = idg.shape[1]
    cap = cap if cap is not None else T * min(topk, n_local)
    xq = torch.full((cap, K), 0xEE, dtype=torch.uint8, device=DEV)
    sx = torch.full((K // 128, cap), -3.0, dtype=torch.float32, device=DEV)
    tok = torch.full((cap,), -7, dtype=torch.int32, device=DEV)
    off = torch.full((n_local + 1,), -9, dtype=torch.int32, device=DEV)
    fp8fg.fp8_moe_dispatch_quant(xg, idg, begin, n_local, cap=cap, xq=xq, sx=sx, offsets=off,
                                 token_ids=tok, workspace=workspace)
    torch.cuda.synchronize()
    return xq.cpu().numpy(), sx.cpu().numpy(), off.cpu().numpy(), tok.cpu().numpy()


def _check(x, ids, begin, n_local, **kw):
    xq, sx, off, tok = _run(x, ids, begin, n_local, **kw)
    rxq, rsx, roff, rtok = oracle.moe_dispatch_quant(bits(x), np.asarray(ids), begin, n_local)
    R = int(roff[-1])
    assert np.array_equal(off, roff)
    assert np.array_equal(tok[:R], rtok)
    assert np.array_equal(xq[:R], rxq)
    assert np.array_equal(sx[:, :R].view(np.uint32), rsx.view(np.uint32))
    # untouched past the used rows
    assert np.all(xq[R:] == 0xEE) and np.all(sx[:, R:] == -3.0) and np.all(tok[R:] == -7)
    return R


CASES = [  # T, K, topk, n_experts (ids drawn from), expert_begin, n_local
    (1, 128, 1, 4, 0, 4), (63, 256, 2, 8, 0, 8), (64, 384, 8, 64, 16, 16),
    (65, 128, 8, 256, 32, 32), (200, 1024, 4, 40, 5, 30), (513, 640, 6, 12, 0, 12),
    (130, 256, 16, 1024, 0, 1024), (300, 128, 3, 3, 0, 1)]


@pytest.mark.parametrize("T,K,topk,n_exp,begin,n_local", CASES)
def test_random_routing(T, K, topk, n_exp, begin, n_local):
    g = torch.Generator().manual_seed(T * 7 + K + topk)
    x = inputs.act(T, K, g)
    # ids from a wider range than the local block, with repeats and negatives
    ids = torch.randint(-3, n_exp + 3, (T, topk), generator=g)
    R = _check(x, ids.numpy(), begin, n_local)
    assert R > 0 or T < 60


def test_repeats_and_single_expert_hot():
    T, K = 257, 256
    g = torch.Generator().manual_seed(11)
    x = inputs.act(T, K, g)
    ids = torch.full((T, 4), 5, dtype=torch.int64)  # every token: expert 5 four times
    ids[::3, 1] = 2
    _check(x, ids.numpy(), 0, 8)


def test_no_local_hits_and_no_tokens():
    T, K = 70, 128
    x = inputs.act(T, K, torch.Generator().manual_seed(12))
    xq, sx, off, tok = _run(x, np.full((T, 2), 500), 0, 8)
    assert off.tolist() == [0] * 9 and np.all(xq == 0xEE)
    x0 = torch.zeros((0, K), dtype=torch.bfloat16)
    xq, sx, off, tok = _run(x0, np.zeros((0, 2), np.int32), 0, 8, cap=0)
    assert off.tolist() == [0] * 9


def test_argument_checks():
    T, K = 10, 128
    x = inputs.act(T, K, torch.Generator().manual_seed(13)).to(DEV)
    ids = torch.zeros((T, 2), dtype=torch.int32, device=DEV)
    with pytest.raises(fp8fg.Fp8Error) as e:
        fp8fg.fp8_moe_dispatch_quant(x, ids, 0, 4, cap=T * 2 - 1)  # cap < T * min(topk, E)
    assert e.value.status == 2
    ws = torch.empty(fp8fg.fp8_moe_dispatch_workspace_size(T, 4) + 512, dtype=torch.uint8,
                     device=DEV)
    with pytest.raises(fp8fg.Fp8Error) as e:
        fp8fg.fp8_moe_dispatch_quant(x, ids, 0, 4, workspace=ws[4:])
    assert e.value.status == 3
    with pytest.raises(fp8fg.Fp8Error) as e:
        fp8fg.fp8_moe_dispatch_quant(x, torch.zeros((T, 17), dtype=torch.int32, device=DEV), 0, 4)
    assert e.value.status == 2


def test_more_chunks_than_resident_ctas():
    """40000 tokens make 625 chunks of 64: more (chunk, K slice) CTAs than fit on
    the GPU at once even with one K slice per chunk, so the pack launch runs in
    more than one wave; skewed top-8 routing over 256 experts, 32 local."""
    T, K = 40000, 256
    g = torch.Generator().manual_seed(15)
    x = inputs.act(T, K, g)
    ids = inputs.moe_topk(T, 256, 8, g)
    R = _check(x, ids.numpy(), 0, 32)
    assert R > 1000


def test_workspace_reused_without_initialisation():
    T, K = 400, 256
    g = torch.Generator().manual_seed(14)
    ws = torch.full((fp8fg.fp8_moe_dispatch_workspace_size(T, 16),), 0x5A, dtype=torch.uint8,
                    device=DEV)
    for _ in range(2):
        x = inputs.act(T, K, g)
        ids = torch.randint(0, 16, (T, 3), generator=g)
        _check(x, ids.numpy(), 0, 16, workspace=ws)


def test_prefill_workload_dispatch_then_grouped_gemm():
    """16384 tokens, top-8 of 256 experts, 32 local; K 7168 -> the grouped GEMM."""
    wl = inputs.moe_prefill()
    x_tok, order = wl.extra["x_tokens"], wl.extra["topk_ids"]
    T, K = x_tok.shape
    R = _check(x_tok, order.numpy(), 0, wl.E)
    assert R == int(wl.offsets[-1])
    # packed operands straight into the grouped GEMM
    xg = x_tok.to(DEV)
    idg = order.to(torch.int32).to(DEV).contiguous()
    xq, sx, off, tok = fp8fg.fp8_moe_dispatch_quant(xg, idg, 0, wl.E)
    cap = xq.shape[0]
    wq = torch.empty((wl.E, wl.N, K), dtype=torch.uint8, device=DEV)
    sw = torch.empty((wl.E, wl.N // 128, K // 128), dtype=torch.float32, device=DEV)
    for e in range(wl.E):
        fp8fg.fp8_quant_weight_128x128(wl.w[e].to(DEV), wq=wq[e], sw=sw[e])
    y = fp8fg.fp8_grouped_gemm_moe(xq, sx, wq, sw, off)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    rxq, rsx, roff, _ = oracle.moe_dispatch_quant(bits(x_tok), order.numpy(), 0, wl.E)
    rows = group_rows(roff, 1024, seed=5)
    # every operand of the oracle product comes from the oracle: the packed A
    # rows of its dispatch and its own 128x128 quantisation of each weight
    bq, sb = _oracle_weights(wl.w)
    _compare(y, rxq, rsx, bq, sb, roff, rows)
    assert cap >= R
