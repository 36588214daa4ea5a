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


def _rows_of(S, idx):
    """S for the local rows idx: S is an array [rows, N] or a callable(idx) -> [len(idx), N]."""
    return S(idx) if callable(S) else np.asarray(S)[idx]


def check_f32_elementwise(gpu, ref64, K, S):
    """|gpu - C| <= u (K/128 + 128) S per element (the FP32 accumulation bound).

    S (the magnitude sum, array or callable over local row indices) is only
    formed for the rows where the cheaper bound with |C| <= S in place of S
    does not already hold.
    """
    gpu = np.asarray(gpu, np.float64)
    gamma = U32 * (K // 128 + 128)
    d = np.abs(gpu - ref64)
    loose = d > gamma * np.abs(ref64)
    rows = np.nonzero(loose.any(axis=1))[0]
    if rows.size:
        Sr = _rows_of(S, rows)
        assert np.all(d[rows] <= gamma * Sr + 1e-300), "elements beyond the FP32 accumulation bound"
    return int(rows.size)


def check_bf16(gpu_u16, ref64, S=None, K=None, max_fallback_frac=1e-3):
    """<= 1 bfloat16 ulp per element against RNE_bf16(fl32(C)).

    Where the GPU differs by more than that, the element must still be within
    1 ulp plus the FP32 accumulation bound u (K/128 + 128) S of the exact C (S
    the magnitude sum, an array or a callable over local row indices, formed
    only for the rows that need it), and such elements must be rare.
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
        rows = np.nonzero(bad.any(axis=1))[0]
        Sr = _rows_of(S, rows)
        bound = ulp[rows] + U32 * (K // 128 + 128) * Sr
        within = np.abs(g[rows] - ref64[rows]) <= bound
        badr = bad[rows]
        assert np.all(within[badr]), "%d elements beyond 1 ulp + FP32 bound" % int(
            (~within & badr).sum())
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


def tile_edges(lo, hi, tile=128):
    """First and last row of every tile-row block of [lo, hi), blocks starting at lo."""
    out = []
    for t0 in range(lo, hi, tile):
        out += [t0, min(t0 + tile, hi) - 1]
    return out


def sample_rows(M, n, seed=0, tile=128):
    """Every 128-row tile's first and last row, plus random rows up to n in all."""
    rng = np.random.default_rng(seed)
    edges = np.unique(np.array(tile_edges(0, M, tile), np.int64))
    n_rest = max(0, min(M, n) - edges.size)
    pool = np.setdiff1d(np.arange(M), edges)
    rest = rng.choice(pool, min(n_rest, pool.size), replace=False) if n_rest else []
    return np.unique(np.concatenate([edges, rest])).astype(np.int64)


def group_rows(offsets, n, seed=0, tile=128):
    """Rows of an expert-grouped operand: the first and last row of every
    expert and of every 128-row tile inside each expert (tiles start at the
    expert's first row, as the grouped GEMM cuts them), plus random rows up to
    n in all."""
    rng = np.random.default_rng(seed)
    offsets = np.asarray(offsets, np.int64)
    edges = []
    for e in range(offsets.size - 1):
        edges += tile_edges(int(offsets[e]), int(offsets[e + 1]), tile)
    edges = np.unique(np.array(edges, np.int64))
    R = int(offsets[-1])
    n_rest = max(0, min(R, n) - edges.size)
    pool = np.setdiff1d(np.arange(R), edges)
    rest = rng.choice(pool, min(n_rest, pool.size), replace=False) if n_rest else []
    return np.unique(np.concatenate([edges, rest])).astype(np.int64)
