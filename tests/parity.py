"""Comparison helpers shared by the GPU parity tests (CUDA path vs oracle)."""
import numpy as np
import torch

import oracle
from fp8_fine_grained_22_b300 import inputs

U32 = 2.0 ** -24  # binary32 unit roundoff


def bits(t):
    return inputs.bf16_bits(t)


def np_u8(t):
    return t.detach().cpu().numpy()


def bf16_to_f64(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(v64):
    """ulp of bfloat16 values (8 significant bits), smallest normal spacing at 0."""
    a = np.abs(v64)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def magnitude(aq, sa, bq, sb_matrix, rows):
    """S[i, n] = sum_kb |sa sb| sum_k |dec a||dec b| for the given rows (float64)."""
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    a = np.abs(dec[aq[rows]])
    b = np.abs(dec[bq])
    K = aq.shape[1]
    S = np.zeros((len(rows), bq.shape[0]))
    for kb in range(K // 128):
        blk = slice(kb * 128, kb * 128 + 128)
        S += (np.abs(sa[kb, rows])[:, None] * np.abs(sb_matrix[None, :, kb])) * (a[:, blk] @ b[:, blk].T)
    return S


def check_f32(gpu, ref64, tol=1e-5):
    """Relative Frobenius error of an FP32 GEMM output."""
    gpu = np.asarray(gpu, np.float64)
    err = np.linalg.norm(gpu - ref64) / max(np.linalg.norm(ref64), 1e-300)
    assert err <= tol, "relative Frobenius error %.3e > %.1e" % (err, tol)
    return err


def check_bf16(gpu_u16, ref64, S=None, K=None, max_fallback_frac=1e-3):
    """<= 1 bfloat16 ulp per element against RNE_bf16(fl32(C)).

    Where the GPU differs by more than that, the element must still be within
    1 ulp plus the FP32 accumulation bound u (K/128 + 128) S of the exact C (S
    the magnitude sum), and such elements must be rare.
    """
    g = bf16_to_f64(gpu_u16)
    o = bf16_to_f64(oracle.round_bf16(ref64))
    ulp = bf16_ulp(o)
    ok = np.abs(g - o) <= ulp
    bad = ~ok
    n_bad = int(bad.sum())
    if n_bad:
        assert S is not None, "%d elements beyond 1 bf16 ulp (first at %s)" % (
            n_bad, np.argwhere(bad)[0])
        bound = ulp + U32 * (K // 128 + 128) * S
        within = np.abs(g - ref64) <= bound
        assert np.all(within[bad]), "%d elements beyond 1 ulp + FP32 bound" % int((~within & bad).sum())
        assert n_bad <= max_fallback_frac * g.size, "%d of %d elements need the FP32 bound" % (
            n_bad, g.size)
    return n_bad


def b_scale_matrix(sb, bmode, N, K):
    KB = K // 128
    n = np.arange(N)[:, None]
    kb = np.arange(KB)[None, :]
    if bmode == oracle.BSCALE_BLOCK128:
        return sb[n // 128, kb].astype(np.float64)
    if bmode == oracle.BSCALE_ROW1x128:
        return sb[kb, n].astype(np.float64)
    return sb[kb, n // 128].astype(np.float64)


def sample_rows(M, n, seed=0, tile=128):
    """First/last rows of every 128-row tile (up to n) plus random rows."""
    rng = np.random.default_rng(seed)
    edges = []
    for t0 in range(0, M, tile):
        edges += [t0, min(t0 + tile, M) - 1]
    edges = np.unique(np.array(edges))
    if len(edges) > n // 2:
        edges = rng.choice(edges, n // 2, replace=False)
    rest = rng.choice(M, min(M, n - len(edges)), replace=False)
    return np.unique(np.concatenate([edges, rest, [0, M - 1]])).astype(np.int64)
