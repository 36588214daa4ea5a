"""Pins of the oracle's block-scaled GEMM (CPU only).

Pinned against:
  * brute force with integer arithmetic: every decoded E4M3 value times 2^9 is
    an integer, so each 128-wide block sum is formed exactly in int64 from
    torch's own decoding of the codes;
  * an independent dequantise-then-multiply path (numpy float64 matmul of
    dec(q) * s for both operands), which reaches the same value up to binary64
    rounding;
  * the unquantised float64 product of the original bfloat16 inputs, within
    the elementwise bound that the per-element dequantisation error implies.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import inputs

DEC = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(
    torch.float64).numpy()


def _bits(t):
    return inputs.bf16_bits(t)


def _int_codes(q):
    v = DEC[q] * 512.0
    assert np.all(v == np.round(v))
    return v.astype(np.int64)


def _b_scale_matrix(sb, bmode, N, K):
    """[N, K/128] per-(n, kb) B scales, indexed independently of the oracle."""
    KB = K // 128
    n = np.arange(N)[:, None]
    kb = np.arange(KB)[None, :]
    if bmode == oracle.BSCALE_BLOCK128:
        return sb[n // 128, kb].astype(np.float64)
    if bmode == oracle.BSCALE_ROW1x128:
        return sb[kb, n].astype(np.float64)
    return sb[kb, n // 128].astype(np.float64)


def _operands(M, N, K, bmode, seed):
    g = torch.Generator().manual_seed(seed)
    x = inputs.act(M, K, g)
    if bmode == oracle.BSCALE_ROW1x128:
        w = inputs.grad(N, K, g)  # B rows quantised 1x128 along K
        bq, sbT = oracle.quant_act_1x128(_bits(w))
        sb = sbT  # [K/128, N]
        wf = w.double().numpy().T  # [K, N]
    else:
        w = inputs.weight(K, N, g)
        bq, bqT, sw = oracle.quant_weight_128x128(_bits(w))
        sb = sw if bmode == oracle.BSCALE_BLOCK128 else np.ascontiguousarray(sw.T)
        wf = w.double().numpy()
    aq, sa = oracle.quant_act_1x128(_bits(x))
    return x.double().numpy(), wf, aq, sa, bq, sb


SHAPES = [(2, 128, 128), (2, 256, 256), (3, 384, 512), (5, 128, 384)]


@pytest.mark.parametrize("bmode", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_brute_force_integer(M, N, K, bmode):
    _, _, aq, sa, bq, sb = _operands(M, N, K, bmode, seed=M * 7 + N + K + bmode)
    c = oracle.gemm_blockscaled(aq, sa, bq, sb, bmode)
    ia, ib = _int_codes(aq), _int_codes(bq)
    sbm = _b_scale_matrix(sb, bmode, N, K)
    want = np.zeros((M, N))
    for kb in range(K // 128):
        blk = slice(kb * 128, kb * 128 + 128)
        p = (ia[:, blk] @ ib[:, blk].T).astype(np.float64) * 2.0 ** -18  # exact
        want += (sa[kb].astype(np.float64)[:, None] * sbm[None, :, kb]) * p
    np.testing.assert_array_equal(c, want)


@pytest.mark.parametrize("bmode", [0, 1, 2])
def test_dequantised_matmul_path(bmode):
    M, N, K = 37, 384, 640
    _, _, aq, sa, bq, sb = _operands(M, N, K, bmode, seed=100 + bmode)
    c = oracle.gemm_blockscaled(aq, sa, bq, sb, bmode)
    a_hat = DEC[aq] * np.repeat(sa.T.astype(np.float64), 128, axis=1)
    b_hat = DEC[bq] * np.repeat(_b_scale_matrix(sb, bmode, N, K), 128, axis=1)
    ref = a_hat @ b_hat.T
    mag = np.abs(a_hat) @ np.abs(b_hat).T
    assert np.all(np.abs(c - ref) <= 1e-12 * mag + 1e-300)


def _qerr(x64, s64):
    r = np.abs(x64 / s64)
    e = np.floor(np.log2(np.maximum(r, 2.0 ** -6)))
    return (0.5 * np.exp2(e - 3) + r * 2.0 ** -24) * s64


@pytest.mark.parametrize("bmode", [0, 1, 2])
def test_within_quantisation_bound_of_unquantised_product(bmode):
    M, N, K = 64, 256, 512
    xf, wf, aq, sa, bq, sb = _operands(M, N, K, bmode, seed=200 + bmode)
    c = oracle.gemm_blockscaled(aq, sa, bq, sb, bmode)
    exact = xf @ wf
    da = _qerr(xf, np.repeat(sa.T.astype(np.float64), 128, axis=1))
    db = _qerr(wf.T, np.repeat(_b_scale_matrix(sb, bmode, N, K), 128, axis=1))
    bound = np.abs(xf) @ db.T + da @ np.abs(wf) + da @ db.T
    assert np.all(np.abs(c - exact) <= bound * (1 + 1e-9) + 1e-300)
    # and the bound is not vacuous: the error is a small fraction of |x||w|
    assert np.linalg.norm(c - exact) < 0.1 * np.linalg.norm(exact)


def test_row_sampling_and_output_rounding():
    M, N, K = 40, 256, 384
    _, _, aq, sa, bq, sb = _operands(M, N, K, 0, seed=300)
    full = oracle.gemm_blockscaled(aq, sa, bq, sb)
    rows = np.array([39, 0, 17, 17, 5])
    np.testing.assert_array_equal(oracle.gemm_blockscaled(aq, sa, bq, sb, rows=rows), full[rows])
    np.testing.assert_array_equal(
        oracle.gemm_blockscaled(aq, sa, bq, sb, nthreads=3),
        oracle.gemm_blockscaled(aq, sa, bq, sb, nthreads=1))
    f32 = oracle.round_f32(full)
    np.testing.assert_array_equal(f32, full.astype(np.float32))
    bf = oracle.round_bf16(full)
    ref = torch.from_numpy(full.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    np.testing.assert_array_equal(bf, ref.view(np.uint16))


def test_grouped_equals_dense_per_expert():
    g = torch.Generator().manual_seed(400)
    K, N, E = 256, 256, 4
    counts = [3, 0, 130, 1]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    T = int(offsets[-1])
    x = inputs.act(T, K, g)
    ws = [inputs.weight(K, N, g) for _ in range(E)]
    aq, sa = oracle.quant_act_1x128(_bits(x))
    bq = np.stack([oracle.quant_weight_128x128(_bits(w))[0] for w in ws])
    sb = np.stack([oracle.quant_weight_128x128(_bits(w))[2] for w in ws])
    y = oracle.grouped_gemm(aq, sa, bq, sb, offsets)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        aq_e, sa_e = oracle.quant_act_1x128(_bits(x[lo:hi]))
        np.testing.assert_array_equal(
            y[lo:hi], oracle.gemm_blockscaled(aq_e, sa_e, bq[e], sb[e]))
    rows = np.array([T - 1, 0, 3, 132])
    np.testing.assert_array_equal(oracle.grouped_gemm(aq, sa, bq, sb, offsets, rows=rows), y[rows])


def test_grouped_dgrad_equals_dequantised_product():
    """Dgrad of the grouped GEMM (weights' transposed codes, scales read transposed)
    against dY_deq . W_deq^T formed from the Fprop-orientation codes and scales."""
    g = torch.Generator().manual_seed(500)
    K, N, E = 384, 256, 3  # Fprop W[K, N]; Dgrad contracts over N, outputs K columns
    counts = [5, 0, 131]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    T = int(offsets[-1])
    dy = inputs.grad(T, N, g)
    ws = [inputs.weight(K, N, g) for _ in range(E)]
    q = [oracle.quant_weight_128x128(_bits(w)) for w in ws]
    dq, sd = oracle.quant_act_1x128(_bits(dy))
    bqT = np.stack([r[1] for r in q])  # [E][K][N]
    sw = np.stack([r[2] for r in q])   # [E][N/128][K/128]
    dx = oracle.grouped_gemm(dq, sd, bqT, sw, offsets, bmode=oracle.BSCALE_BLOCK128_T)
    dy_hat = DEC[dq] * np.repeat(sd.T.astype(np.float64), 128, axis=1)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        wq, _, s = q[e]
        w_hat = DEC[wq].T * np.repeat(np.repeat(s.T.astype(np.float64), 128, axis=0), 128,
                                      axis=1)  # [K, N]
        ref = dy_hat[lo:hi] @ w_hat.T
        mag = np.abs(dy_hat[lo:hi]) @ np.abs(w_hat).T
        assert np.all(np.abs(dx[lo:hi] - ref) <= 1e-12 * mag + 1e-300)


def test_grouped_128x1_single_expert_is_the_dense_quantiser():
    g = torch.Generator().manual_seed(600)
    x = inputs.act(256, 192, g)
    xqT, sxT, pofs = oracle.quant_act_128x1_grouped(_bits(x), [0, 256])
    q, s = oracle.quant_act_128x1(_bits(x))
    assert pofs.tolist() == [0, 256]
    np.testing.assert_array_equal(xqT, q)
    np.testing.assert_array_equal(sxT, s)


def test_grouped_128x1_short_groups():
    """Short groups: zero codes in the padding, amax element at +-448, codes within the
    E4M3 rounding bound of x / s."""
    g = torch.Generator().manual_seed(601)
    counts = [5, 0, 130, 128]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    T, K = int(offsets[-1]), 128
    x = inputs.act(T, K, g)
    xqT, sxT, pofs = oracle.quant_act_128x1_grouped(_bits(x), offsets)
    assert pofs.tolist() == [0, 128, 128, 384, 512]
    xf = x.double().numpy()
    for e in range(len(counts)):
        t_e = counts[e]
        for grp in range((t_e + 127) // 128):
            col0 = int(pofs[e]) + 128 * grp
            n = min(128, t_e - 128 * grp)
            seg = xf[offsets[e] + 128 * grp:offsets[e] + 128 * grp + n]  # [n, K]
            codes = xqT[:, col0:col0 + 128]                                # [K, 128]
            assert np.all(codes[:, n:] == 0)
            s = sxT[col0 // 128].astype(np.float64)                        # [K]
            deq = DEC[codes[:, :n]].T * s[None, :]
            r = np.abs(seg / s[None, :])
            ulp = np.exp2(np.floor(np.log2(np.maximum(r, 2.0 ** -6))) - 3)
            assert np.all(np.abs(deq - seg) <= (0.5 * ulp + r * 2.0 ** -23) * s[None, :])
            amax_rows = np.abs(seg).argmax(axis=0)
            top = codes[np.arange(K), amax_rows] & 0x7F
            assert np.all((top == 0x7E) | (np.abs(seg).max(axis=0) == 0))


def test_grouped_wgrad_equals_dequantised_product():
    g = torch.Generator().manual_seed(602)
    counts = [3, 0, 200, 128]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    T, M, N = int(offsets[-1]), 256, 384  # M: Fprop inner dim, N: Fprop output dim
    x = inputs.act(T, M, g)
    dy = inputs.grad(T, N, g)
    xqT, sxT, pofs = oracle.quant_act_128x1_grouped(_bits(x), offsets)
    dqT, sdT, pofs2 = oracle.quant_act_128x1_grouped(_bits(dy), offsets)
    assert np.array_equal(pofs, pofs2)
    dw = oracle.grouped_wgrad(xqT, sxT, dqT, sdT, pofs)
    for e in range(len(counts)):
        lo, hi = int(pofs[e]), int(pofs[e + 1])
        if hi == lo:
            assert np.all(dw[e] == 0)
            continue
        a_hat = DEC[xqT[:, lo:hi]] * np.repeat(sxT[lo // 128:hi // 128].T.astype(np.float64), 128,
                                                 axis=1)
        b_hat = DEC[dqT[:, lo:hi]] * np.repeat(sdT[lo // 128:hi // 128].T.astype(np.float64), 128,
                                                 axis=1)
        ref = a_hat @ b_hat.T
        mag = np.abs(a_hat) @ np.abs(b_hat).T
        assert np.all(np.abs(dw[e] - ref) <= 1e-12 * mag + 1e-300)
        # and it approximates the unquantised X_e^T dY_e
        exact = x.double().numpy()[offsets[e]:offsets[e + 1]].T @ \
            dy.double().numpy()[offsets[e]:offsets[e + 1]]
        assert np.linalg.norm(dw[e] - exact) < 0.1 * np.linalg.norm(exact)
