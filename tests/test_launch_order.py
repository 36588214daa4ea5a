"""The GEMMs are launched with programmatic stream serialisation: their CTAs
may start while the kernel before them on the stream is still running, and
they wait for it before reading any operand, scale or offset.

These tests run producer -> GEMM pairs back to back on one stream with no
host synchronisation, alternating two different inputs, so that every GEMM
follows a producer that is overwriting the very buffers it reads.  Each
result must be bitwise equal to the same pair run with a synchronisation in
between (the kernels are deterministic), and those reference results are
checked against the oracle on rows that include every tile and expert edge.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import b_scale_matrix, bits, check_bf16, group_rows, magnitude, sample_rows
from test_grouped_parity import _compare, _quant_experts as _oracle_weights

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_operand_quantiser_then_gemm_back_to_back():
    M, K, N = 4096, 4096, 1024
    g = torch.Generator().manual_seed(31)
    xs = [inputs.act(M, K, g).to(DEV) for _ in range(2)]
    ws = [inputs.weight(K, N, g).to(DEV) for _ in range(2)]
    xq = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    sx = torch.empty((K // 128, M), dtype=torch.float32, device=DEV)
    wq = torch.empty((N, K), dtype=torch.uint8, device=DEV)
    sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=DEV)

    def pair(j, y):
        fp8fg.fp8_quant_fprop_operands(xs[j], ws[j], xq=xq, sx=sx, wq=wq, sw=sw)
        fp8fg.fp8_gemm_blockscaled(xq, sx, wq, sw, out_dtype=torch.bfloat16, c=y)

    ref = []
    for j in range(2):
        y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        fp8fg.fp8_quant_fprop_operands(xs[j], ws[j], xq=xq, sx=sx, wq=wq, sw=sw)
        torch.cuda.synchronize()
        fp8fg.fp8_gemm_blockscaled(xq, sx, wq, sw, out_dtype=torch.bfloat16, c=y)
        torch.cuda.synchronize()
        ref.append(y)
        # the synchronised result against the oracle on sampled rows
        aq, sa = oracle.quant_act_1x128(bits(xs[j].cpu()))
        bq, _, sb = oracle.quant_weight_128x128(bits(ws[j].cpu()))
        rows = sample_rows(M, 256, seed=j)
        want = oracle.gemm_blockscaled(aq, sa, bq, sb, rows=rows)
        got = ref[j].cpu().view(torch.int16).numpy().view(np.uint16)[rows]
        sbm = b_scale_matrix(sb, oracle.BSCALE_BLOCK128, N, K)
        check_bf16(got, want, S=lambda idx: magnitude(aq, sa, bq, sbm, rows[idx]), K=K)

    outs = [torch.empty((M, N), dtype=torch.bfloat16, device=DEV) for _ in range(16)]
    for i, y in enumerate(outs):
        pair(i % 2, y)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    for i, y in enumerate(outs):
        assert torch.equal(y, ref[i % 2]), i


def test_dispatch_then_grouped_gemm_back_to_back():
    T, K, N, E, topk = 3000, 1024, 512, 8, 4
    g = torch.Generator().manual_seed(32)
    xs = [inputs.act(T, K, g).to(DEV) for _ in range(2)]
    ids = [torch.randint(0, E + 2, (T, topk), generator=g).to(torch.int32).to(DEV)
           for _ in range(2)]
    wq = torch.empty((E, N, K), dtype=torch.uint8, device=DEV)
    sw = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=DEV)
    w_host = [inputs.weight(K, N, g) for _ in range(E)]
    for e in range(E):
        fp8fg.fp8_quant_weight_128x128(w_host[e].to(DEV), wq=wq[e], sw=sw[e])
    cap = T * min(topk, E)
    xq = torch.empty((cap, K), dtype=torch.uint8, device=DEV)
    sx = torch.empty((K // 128, cap), dtype=torch.float32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    tok = torch.empty(cap, dtype=torch.int32, device=DEV)
    ws = fp8fg.moe_dispatch_workspace(T, E, torch.device(DEV))

    def pair(j, y):
        fp8fg.fp8_moe_dispatch_quant(xs[j], ids[j], 0, E, cap=cap, xq=xq, sx=sx, offsets=off,
                                     token_ids=tok, workspace=ws)
        fp8fg.fp8_grouped_gemm_moe(xq, sx, wq, sw, off, c=y)

    bq_ref, sb_ref = _oracle_weights(torch.stack(w_host))  # the oracle's own weight codes
    ref, rows_used = [], []
    for j in range(2):
        y = torch.zeros((cap, N), dtype=torch.bfloat16, device=DEV)
        fp8fg.fp8_moe_dispatch_quant(xs[j], ids[j], 0, E, cap=cap, xq=xq, sx=sx, offsets=off,
                                     token_ids=tok, workspace=ws)
        torch.cuda.synchronize()
        fp8fg.fp8_grouped_gemm_moe(xq, sx, wq, sw, off, c=y)
        torch.cuda.synchronize()
        R = int(off[-1].item())
        ref.append(y[:R].clone())
        rows_used.append(R)
        rxq, rsx, roff, _ = oracle.moe_dispatch_quant(bits(xs[j].cpu()), ids[j].cpu().numpy(),
                                                      0, E)
        assert int(roff[-1]) == R
        _compare(y, rxq, rsx, bq_ref, sb_ref, roff, group_rows(roff, 256, seed=j))
    assert rows_used[0] != rows_used[1]  # the two routings pack different row counts

    outs = [torch.zeros((cap, N), dtype=torch.bfloat16, device=DEV) for _ in range(12)]
    for i, y in enumerate(outs):
        pair(i % 2, y)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    for i, y in enumerate(outs):
        assert torch.equal(y[:rows_used[i % 2]], ref[i % 2]), i
