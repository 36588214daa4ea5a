"""CPU oracle for fine-grained FP8 quantisation and the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY.  The product path never imports this package; only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library.

The arithmetic lives in ``fp8_oracle.c`` (plain C, binary64 where the method
leaves precision open; see that file's header for the passages of the
DeepSeek-V3 Technical Report each step follows).  This module only marshals
numpy arrays into it.

Conventions: bfloat16 tensors are passed as ``uint16`` numpy arrays holding
the raw bfloat16 bit patterns; E4M3 codes are ``uint8`` arrays.

When the environment variable ``FP8FG_ORACLE_LIB`` names a library, that
library is loaded instead of the built ``liboracle.so``: the mutant tests use
it to run the oracle's pins against deliberately broken builds.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build as _build, LIB_PATH

_lib = None

BSCALE_BLOCK128 = 0    # sb[N/128][K/128]
BSCALE_ROW1x128 = 1    # sb[K/128][N]
BSCALE_BLOCK128_T = 2  # sb[K/128][N/128]


def _load():
    global _lib
    if _lib is None:
        path = os.environ.get("FP8FG_ORACLE_LIB")
        if not path:
            path = LIB_PATH
            if not os.path.exists(path):
                _build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.fo_e4m3_encode.restype = ctypes.c_uint8
        lib.fo_e4m3_encode.argtypes = [ctypes.c_float]
        lib.fo_e4m3_decode.restype = ctypes.c_double
        lib.fo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.fo_e4m3_encode_array.argtypes = [P, I64, P]
        lib.fo_e4m3_decode_array.argtypes = [P, I64, P]
        lib.fo_round_f32.argtypes = [P, I64, P]
        lib.fo_round_bf16.argtypes = [P, I64, P]
        lib.fo_group_scale.restype = ctypes.c_float
        lib.fo_group_scale.argtypes = [ctypes.c_float]
        lib.fo_quant_act_1x128.argtypes = [P, I64, I64, I64, P, I64, P]
        lib.fo_quant_act_128x1.argtypes = [P, I64, I64, I64, P, P]
        lib.fo_quant_weight_128x128.argtypes = [P, I64, I64, I64, P, P, P]
        lib.fo_e5m6_encode.restype = ctypes.c_uint16
        lib.fo_e5m6_encode.argtypes = [ctypes.c_float]
        lib.fo_e5m6_decode.restype = ctypes.c_double
        lib.fo_e5m6_decode.argtypes = [ctypes.c_uint16]
        lib.fo_e5m6_encode_array.argtypes = [P, I64, P]
        lib.fo_e5m6_decode_array.argtypes = [P, I64, P]
        lib.fo_group_scale_e5m6.restype = ctypes.c_float
        lib.fo_group_scale_e5m6.argtypes = [ctypes.c_float]
        lib.fo_quant_act_1x128_e5m6.argtypes = [P, I64, I64, I64, P, I64, P]
        lib.fo_pow2_exponent.restype = ctypes.c_int
        lib.fo_pow2_exponent.argtypes = [ctypes.c_float]
        lib.fo_quant_act_1x128_pow2.argtypes = [P, I64, I64, I64, P, I64, P]
        lib.fo_quant_weight_128x128_pow2.argtypes = [P, I64, I64, I64, P, P]
        lib.fo_gemm_blockscaled_rows.argtypes = [
            P, I64, P, I64, P, I64, P, I64, ctypes.c_int, I64, I64, I64, P, I64, P,
            ctypes.c_int]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


# ------------------------------------------------------------------ formats --
def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (RNE, saturating at 448) of binary32 values."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().fo_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_decode(c) -> np.ndarray:
    """binary64 values of E4M3 codes."""
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().fo_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def round_f32(c) -> np.ndarray:
    c = _c(c, np.float64)
    out = np.empty(c.shape, np.float32)
    _load().fo_round_f32(_ptr(c), c.size, _ptr(out))
    return out


def round_bf16(c) -> np.ndarray:
    """bfloat16 bit patterns of RNE_bf16(fl32(c))."""
    c = _c(c, np.float64)
    out = np.empty(c.shape, np.uint16)
    _load().fo_round_bf16(_ptr(c), c.size, _ptr(out))
    return out


def group_scale(amax: float) -> np.float32:
    return np.float32(_load().fo_group_scale(float(amax)))


def e5m6_encode(x) -> np.ndarray:
    """E5M6 codes (12-bit values in uint16; RNE, saturating at 65024) of binary32 values."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().fo_e5m6_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def e5m6_decode(c) -> np.ndarray:
    """binary64 values of E5M6 codes (low 12 bits of uint16)."""
    c = _c(c, np.uint16)
    out = np.empty(c.shape, np.float64)
    _load().fo_e5m6_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def group_scale_e5m6(amax: float) -> np.float32:
    return np.float32(_load().fo_group_scale_e5m6(float(amax)))


def pack_e5m6(codes) -> np.ndarray:
    """Storage layout of E5M6 rows: element i of a row occupies bits
    12 i .. 12 i + 11 of the row's bytes, least significant first, so two
    neighbours (c0, c1) fill three bytes: c0 & 0xFF, (c0 >> 8) | (c1 & 0xF) << 4,
    c1 >> 4.  codes uint16 [..., K] (K even) -> uint8 [..., 3 K / 2]."""
    c = _c(codes, np.uint16).astype(np.uint32)
    assert c.shape[-1] % 2 == 0
    c0, c1 = c[..., 0::2], c[..., 1::2]
    out = np.empty(c.shape[:-1] + (c.shape[-1] // 2, 3), np.uint8)
    out[..., 0] = c0 & 0xFF
    out[..., 1] = ((c0 >> 8) & 0xF) | ((c1 & 0xF) << 4)
    out[..., 2] = (c1 >> 4) & 0xFF
    return out.reshape(c.shape[:-1] + (3 * c.shape[-1] // 2,))


def unpack_e5m6(packed) -> np.ndarray:
    """Inverse of pack_e5m6: uint8 [..., 3 K / 2] -> uint16 codes [..., K]."""
    b = _c(packed, np.uint8)
    assert b.shape[-1] % 3 == 0
    t = b.reshape(b.shape[:-1] + (b.shape[-1] // 3, 3)).astype(np.uint16)
    c0 = t[..., 0] | ((t[..., 1] & 0xF) << 8)
    c1 = (t[..., 1] >> 4) | (t[..., 2] << 4)
    out = np.empty(b.shape[:-1] + (2 * (b.shape[-1] // 3),), np.uint16)
    out[..., 0::2] = c0
    out[..., 1::2] = c1
    return out


# ---------------------------------------------------------------- quantisers --
def quant_act_1x128(x_bf16: np.ndarray):
    """x: uint16 [M, K] bfloat16 bits -> (codes uint8 [M, K], scales f32 [K/128, M])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert K % 128 == 0
    xq = np.empty((M, K), np.uint8)
    sx = np.empty((K // 128, M), np.float32)
    _load().fo_quant_act_1x128(_ptr(x), M, K, K, _ptr(xq), K, _ptr(sx))
    return xq, sx


def quant_act_1x128_e5m6(x_bf16: np.ndarray):
    """x: uint16 [M, K] bfloat16 bits -> (E5M6 codes uint16 [M, K], scales f32 [K/128, M]),
    s = fl32(amax / 65024) per 1x128 group; pack_e5m6 gives the stored bytes."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint16)
    sx = np.empty((K // 128, M), np.float32)
    _load().fo_quant_act_1x128_e5m6(_ptr(x), M, K, K, _ptr(q), K, _ptr(sx))
    return q, sx


def pow2_exponent(amax: float) -> int:
    """e of the power-of-two scale 2^e: the smallest with amax / 2^e <= 448, in [-127, 127]."""
    return int(_load().fo_pow2_exponent(float(amax)))


def e8_scales(se8) -> np.ndarray:
    """float32 scales 2^(b - 127) of UE8M0 bytes b."""
    b = np.asarray(se8, dtype=np.int64)
    return np.ldexp(np.ones(b.shape, np.float64), b - 127).astype(np.float32)


def quant_act_1x128_pow2(x_bf16: np.ndarray):
    """x: uint16 [M, K] -> (codes uint8 [M, K], UE8M0 bytes uint8 [K/128, M]) with
    power-of-two 1x128 group scales."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert K % 128 == 0
    xq = np.empty((M, K), np.uint8)
    se8 = np.empty((K // 128, M), np.uint8)
    _load().fo_quant_act_1x128_pow2(_ptr(x), M, K, K, _ptr(xq), K, _ptr(se8))
    return xq, se8


def quant_weight_128x128_pow2(w_bf16: np.ndarray):
    """w: uint16 [K, N] -> (wq uint8 [N, K], UE8M0 bytes uint8 [K/128, N], one per row of
    wq, the block's exponent repeated over its 128 rows)."""
    w = _c(w_bf16, np.uint16)
    K, N = w.shape
    assert K % 128 == 0 and N % 128 == 0
    wq = np.empty((N, K), np.uint8)
    se8 = np.empty((K // 128, N), np.uint8)
    _load().fo_quant_weight_128x128_pow2(_ptr(w), K, N, N, _ptr(wq), _ptr(se8))
    return wq, se8


def quant_act_128x1(x_bf16: np.ndarray):
    """x: uint16 [M, K] -> (codes uint8 [K, M] transposed, scales f32 [M/128, K])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert M % 128 == 0
    xqT = np.empty((K, M), np.uint8)
    sxT = np.empty((M // 128, K), np.float32)
    _load().fo_quant_act_128x1(_ptr(x), M, K, K, _ptr(xqT), _ptr(sxT))
    return xqT, sxT


def quant_weight_128x128(w_bf16: np.ndarray):
    """w: uint16 [K, N] -> (wq uint8 [N, K], wqT uint8 [K, N], sw f32 [N/128, K/128])."""
    w = _c(w_bf16, np.uint16)
    K, N = w.shape
    assert K % 128 == 0 and N % 128 == 0
    wq = np.empty((N, K), np.uint8)
    wqT = np.empty((K, N), np.uint8)
    sw = np.empty((N // 128, K // 128), np.float32)
    _load().fo_quant_weight_128x128(_ptr(w), K, N, N, _ptr(wq), _ptr(wqT), _ptr(sw))
    return wq, wqT, sw


# --------------------------------------------------------------------- GEMM --
def gemm_blockscaled(aq, sa, bq, sb, bmode=BSCALE_BLOCK128, rows=None, nthreads=None):
    """binary64 C[rows, :] of the block-scaled product.

    aq: uint8 [M, K] codes, sa: f32 [K/128, M]; bq: uint8 [N, K] codes;
    sb: f32 laid out per ``bmode`` (BLOCK128 [N/128, K/128], ROW1x128
    [K/128, N], BLOCK128_T [K/128, N/128]).  ``rows``: the rows of C to form
    (default all).
    """
    aq = _c(aq, np.uint8)
    sa = _c(sa, np.float32)
    bq = _c(bq, np.uint8)
    sb = _c(sb, np.float32)
    M, K = aq.shape
    N, K2 = bq.shape
    assert K == K2 and K % 128 == 0 and N % 128 == 0
    assert sa.shape == (K // 128, M)
    expect = {BSCALE_BLOCK128: (N // 128, K // 128), BSCALE_ROW1x128: (K // 128, N),
              BSCALE_BLOCK128_T: (K // 128, N // 128)}[bmode]
    assert sb.shape == expect, (sb.shape, expect)
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = _c(rows, np.int64)
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < M)
    out = np.empty((rows.size, N), np.float64)
    if rows.size:
        _load().fo_gemm_blockscaled_rows(
            _ptr(aq), K, _ptr(sa), M, _ptr(bq), K, _ptr(sb), sb.shape[1], bmode, M, N, K,
            _ptr(rows), rows.size, _ptr(out), nthreads or default_threads())
    return out


def grouped_gemm(aq, sa, bq, sb, offsets, rows=None, nthreads=None, bmode=BSCALE_BLOCK128):
    """binary64 Y[rows, :] of the grouped (per-expert) block-scaled product.

    aq: uint8 [T, K] rows grouped by expert; sa: f32 [K/128, T];
    bq: uint8 [E, N, K]; sb: f32 [E, ...] per expert in the ``bmode`` layout
    (BLOCK128 [N/128, K/128]; BLOCK128_T [K/128, N/128] for the Dgrad GEMM);
    offsets: int [E+1], rows offsets[e]..offsets[e+1]-1 belong to expert e
    (rows at or past offsets[E] belong to no expert and may not be requested).
    Each row of Y is the dense product of that row with its expert's weight.
    """
    aq = _c(aq, np.uint8)
    sa = _c(sa, np.float32)
    bq = _c(bq, np.uint8)
    sb = _c(sb, np.float32)
    offsets = np.asarray(offsets, dtype=np.int64)
    T, K = aq.shape
    E, N, _ = bq.shape
    assert offsets.shape == (E + 1,) and offsets[0] == 0 and offsets[-1] <= T
    assert np.all(np.diff(offsets) >= 0)
    if rows is None:
        rows = np.arange(offsets[-1], dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, N), np.float64)
    assert rows.size == 0 or rows.max() < offsets[-1]
    expert_of = np.searchsorted(offsets, rows, side="right") - 1
    for e in range(E):
        sel = np.nonzero(expert_of == e)[0]
        if sel.size == 0:
            continue
        # each row only needs its own A row and A scales; pass the whole A
        # so that the row indices stay global.
        out[sel] = gemm_blockscaled(aq, sa, bq[e], sb[e], bmode,
                                    rows=rows[sel], nthreads=nthreads)
    return out


# ------------------------------------------------------------- MoE dispatch --
def moe_dispatch_quant(x_bf16, topk_ids, expert_begin, n_local):
    """FP8 dispatch of token rows to the local experts.

    Follows the DeepSeek-V3 Technical Report, section 3.3.3 (the activations
    sent to the MoE experts are quantised with the fine-grained 1x128 scheme
    and dispatched in FP8) and section 3.4 (each token goes to the experts of
    its top-k routing).  A token is routed to global expert g when g appears
    in its top-k row (a repeat counts once).  For every local expert
    e = 0 .. n_local-1 (global id expert_begin + e) the routed tokens are
    taken in ascending order; the packed rows are these token rows, expert
    after expert, quantised 1x128.

    x_bf16: uint16 [T, K] bfloat16 bits; topk_ids: int [T, topk].
    Returns (xq uint8 [R, K], sx f32 [K/128, R], offsets int64 [n_local+1],
    token_ids int64 [R]) with R = offsets[-1].
    """
    x = _c(x_bf16, np.uint16)
    ids = np.asarray(topk_ids, dtype=np.int64)
    ids = ids.reshape(x.shape[0], ids.shape[-1] if ids.ndim == 2 else -1)
    T, K = x.shape
    experts = expert_begin + np.arange(n_local, dtype=np.int64)
    # member[t, e]: token t routed to local expert e
    member = (ids[:, :, None] == experts[None, None, :]).any(axis=1)
    token_lists = [np.nonzero(member[:, e])[0] for e in range(n_local)]
    offsets = np.zeros(n_local + 1, np.int64)
    offsets[1:] = np.cumsum([len(tl) for tl in token_lists])
    token_ids = (np.concatenate(token_lists) if n_local else np.zeros(0)).astype(np.int64)
    if token_ids.size == 0:
        return (np.zeros((0, K), np.uint8), np.zeros((K // 128, 0), np.float32), offsets,
                token_ids)
    xq, sx = quant_act_1x128(x[token_ids])
    return xq, sx, offsets, token_ids



# ---------------------------------------------------------------- MoE Wgrad --
def quant_act_128x1_grouped(x_bf16, offsets):
    """128x1 quantisation of each expert's rows along its own tokens.

    DeepSeek-V3 Technical Report, sections 3.3.1-3.3.3 (Wgrad consumes the
    activations and gradients quantised along the tokens, the GEMM's inner
    dimension) applied per expert (section 3.4): expert e's rows
    offsets[e] .. offsets[e+1]-1 are cut into groups of 128 consecutive
    tokens; a short last group is completed with zero rows, which give zero
    codes and leave the group's amax unchanged.

    x_bf16: uint16 [T, K]; offsets: int [E+1].
    Returns (xqT uint8 [K, Tp], sxT f32 [Tp/128, K], pofs int64 [E+1]) with
    expert e in columns pofs[e] .. pofs[e+1]-1 and Tp = pofs[E].
    """
    x = _c(x_bf16, np.uint16)
    offsets = np.asarray(offsets, dtype=np.int64)
    T, K = x.shape
    E = offsets.size - 1
    padded = [((offsets[e + 1] - offsets[e] + 127) // 128) * 128 for e in range(E)]
    pofs = np.zeros(E + 1, np.int64)
    pofs[1:] = np.cumsum(padded)
    Tp = int(pofs[-1])
    xqT = np.zeros((K, Tp), np.uint8)
    sxT = np.zeros((Tp // 128, K), np.float32)
    for e in range(E):
        if padded[e] == 0:
            continue
        seg = np.zeros((padded[e], K), np.uint16)  # bfloat16 +0
        seg[:offsets[e + 1] - offsets[e]] = x[offsets[e]:offsets[e + 1]]
        q, sc = quant_act_128x1(seg)
        xqT[:, pofs[e]:pofs[e + 1]] = q
        sxT[pofs[e] // 128:pofs[e + 1] // 128] = sc
    return xqT, sxT, pofs


def grouped_wgrad(aqT, sa, bqT, sb, pofs, rows=None, nthreads=None):
    """binary64 dW[e][rows, :] for every expert: the per-expert product of the
    transposed operands over the expert's padded token columns, promoted per
    128-token block with the per-row A scale and the per-column B scale
    (section 3.3.2).  aqT uint8 [M, Tp], sa f32 [Tp/128, M], bqT uint8 [N, Tp],
    sb f32 [Tp/128, N], pofs int [E+1].  Returns [E, len(rows), N]."""
    aqT = _c(aqT, np.uint8)
    bqT = _c(bqT, np.uint8)
    pofs = np.asarray(pofs, dtype=np.int64)
    M = aqT.shape[0]
    N = bqT.shape[0]
    E = pofs.size - 1
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((E, rows.size, N))
    for e in range(E):
        lo, hi = int(pofs[e]), int(pofs[e + 1])
        if hi == lo:
            continue
        out[e] = gemm_blockscaled(aqT[:, lo:hi], sa[lo // 128:hi // 128], bqT[:, lo:hi],
                                  sb[lo // 128:hi // 128], BSCALE_ROW1x128, rows=rows,
                                  nthreads=nthreads)
    return out
