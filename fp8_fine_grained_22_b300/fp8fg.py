"""Thin ctypes binding of libfp8fg.so (include/fp8fg.h).

Argument marshalling only: every step runs in the CUDA kernels of the
library.  PyTorch supplies device memory (output tensors are allocated here
when the caller does not pass them) and the current CUDA stream.  There is no
fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH, build as _build

FP8_OK = 0
FP8_OUT_F32 = 0
FP8_OUT_BF16 = 1
FP8_BSCALE_BLOCK128 = 0
FP8_BSCALE_ROW1x128 = 1
FP8_BSCALE_BLOCK128_T = 2

# every entry point of include/fp8fg.h
EXPORTS = ("fp8_status_str", "fp8_device_error", "fp8_selftest_wait_timeout",
           "fp8_quant_act_1x128", "fp8_quant_act_1x128_e5m6", "fp8_quant_act_128x1",
           "fp8_quant_act_dual",
           "fp8_quant_weight_128x128",
           "fp8_quant_fprop_operands", "fp8_quant_act_1x128_pow2",
           "fp8_quant_weight_128x128_pow2", "fp8_gemm_mxfp8",
           "fp8_gemm_blockscaled", "fp8_gemm_blockscaled_ws", "fp8_gemm_blockscaled_workspace_size",
           "fp8_grouped_gemm_moe", "fp8_grouped_gemm_moe_dgrad",
           "fp8_gemm_blockscaled_bf16a", "fp8_grouped_gemm_moe_bf16a",
           "fp8_quant_act_128x1_grouped", "fp8_grouped_gemm_moe_wgrad",
           "fp8_moe_dispatch_workspace_size", "fp8_moe_dispatch_quant",
           "fp8_moe_dispatch_quant_noalloc")


class Fp8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, status_str(status), status))


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; builds it in-tree first if the sources are newer."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            _build()
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libfp8fg.so is missing: build it with "
                               "`python -m fp8_fine_grained_22_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
        L.fp8_status_str.restype = ctypes.c_char_p
        L.fp8_status_str.argtypes = [I]
        L.fp8_device_error.restype = I
        L.fp8_device_error.argtypes = [P]
        L.fp8_selftest_wait_timeout.restype = I
        L.fp8_selftest_wait_timeout.argtypes = [P]
        L.fp8_quant_act_1x128.restype = I
        L.fp8_quant_act_1x128.argtypes = [P, I64, I64, I64, P, I64, P, P]
        L.fp8_quant_act_1x128_e5m6.restype = I
        L.fp8_quant_act_1x128_e5m6.argtypes = [P, I64, I64, I64, P, I64, P, P]
        L.fp8_quant_act_1x128_pow2.restype = I
        L.fp8_quant_act_1x128_pow2.argtypes = [P, I64, I64, I64, P, I64, P, P]
        L.fp8_quant_weight_128x128_pow2.restype = I
        L.fp8_quant_weight_128x128_pow2.argtypes = [P, I64, I64, I64, P, P, P]
        L.fp8_gemm_blockscaled_bf16a.restype = I
        L.fp8_gemm_blockscaled_bf16a.argtypes = [P, I64, P, P, I, I64, I64, I64, P, I64, I, P]
        L.fp8_grouped_gemm_moe_bf16a.restype = I
        L.fp8_grouped_gemm_moe_bf16a.argtypes = [P, I64, P, P, P, I32, I64, I64, I64, P, I, P]
        L.fp8_gemm_mxfp8.restype = I
        L.fp8_gemm_mxfp8.argtypes = [P, P, P, P, I64, I64, I64, P, I64, I, P]
        L.fp8_quant_act_128x1.restype = I
        L.fp8_quant_act_128x1.argtypes = [P, I64, I64, I64, P, P, P]
        L.fp8_quant_act_dual.restype = I
        L.fp8_quant_act_dual.argtypes = [P, I64, I64, I64, P, I64, P, P, P, P]
        L.fp8_quant_weight_128x128.restype = I
        L.fp8_quant_weight_128x128.argtypes = [P, I64, I64, I64, P, P, P, P]
        L.fp8_quant_fprop_operands.restype = I
        L.fp8_quant_fprop_operands.argtypes = [P, I64, I64, I64, P, I64, P, P, I64, I64, P, P,
                                               P, P]
        L.fp8_gemm_blockscaled.restype = I
        L.fp8_gemm_blockscaled.argtypes = [P, P, P, P, I, I64, I64, I64, P, I64, I, P]
        L.fp8_gemm_blockscaled_ws.restype = I
        L.fp8_gemm_blockscaled_ws.argtypes = [P, P, P, P, I, I64, I64, I64, P, I64, I, P, I64, P]
        L.fp8_gemm_blockscaled_workspace_size.restype = I64
        L.fp8_gemm_blockscaled_workspace_size.argtypes = []
        L.fp8_grouped_gemm_moe.restype = I
        L.fp8_grouped_gemm_moe.argtypes = [P, P, P, P, P, I32, I64, I64, I64, P, I, P]
        L.fp8_quant_act_128x1_grouped.restype = I
        L.fp8_quant_act_128x1_grouped.argtypes = [P, I64, I64, I64, P, I32, P, P, I64, P, P]
        L.fp8_grouped_gemm_moe_wgrad.restype = I
        L.fp8_grouped_gemm_moe_wgrad.argtypes = [P, P, P, P, P, I32, I64, I64, I64, P, P]
        L.fp8_grouped_gemm_moe_dgrad.restype = I
        L.fp8_grouped_gemm_moe_dgrad.argtypes = [P, P, P, P, P, I32, I64, I64, I64, P, I, P]
        L.fp8_moe_dispatch_workspace_size.restype = I
        L.fp8_moe_dispatch_workspace_size.argtypes = [I64, I32, ctypes.POINTER(ctypes.c_size_t)]
        L.fp8_moe_dispatch_quant.restype = I
        L.fp8_moe_dispatch_quant.argtypes = [P, I64, I64, I64, P, I32, I32, I32, P, P, I64, P, P,
                                             P, ctypes.c_size_t, P]
        L.fp8_moe_dispatch_quant_noalloc.restype = I
        L.fp8_moe_dispatch_quant_noalloc.argtypes = [P, I64, I64, I64, P, I32, I32, I32, P, P,
                                                     I64, P, P, P]
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().fp8_status_str(int(status)).decode()


def _check(status: int, what: str):
    if status != FP8_OK:
        raise Fp8Error(status, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _cuda(t, name, dtype=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))


def selftest_wait_timeout(stream=None):
    """Launch the bounded-wait self-test (a wait nothing completes); device_error() then
    reports FP8_ERR_TIMEOUT (6)."""
    _check(lib().fp8_selftest_wait_timeout(_stream(stream)), "fp8_selftest_wait_timeout")


def device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device-side error status."""
    return lib().fp8_device_error(_stream(stream))


# --------------------------------------------------------------- quantisers --
def fp8_quant_act_1x128(x, xq=None, sx=None, stream=None):
    """x: bf16 [M, K] (row stride x.stride(0)) -> (xq uint8 [M, K], sx f32 [K/128, M])."""
    _cuda(x, "x", torch.bfloat16)
    assert x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    assert xq.stride(1) == 1 and sx.is_contiguous()
    _check(lib().fp8_quant_act_1x128(_p(x), M, K, x.stride(0), _p(xq), xq.stride(0), _p(sx),
                                     _stream(stream)), "fp8_quant_act_1x128")
    return xq, sx


def fp8_quant_act_1x128_e5m6(x, xq=None, sx=None, stream=None):
    """x: bf16 [M, K] -> (xq uint8 [M, 3K/2] packed 12-bit E5M6 codes, sx f32 [K/128, M])."""
    _cuda(x, "x", torch.bfloat16)
    assert x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, 3 * K // 2), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    assert xq.stride(1) == 1 and sx.is_contiguous()
    _check(lib().fp8_quant_act_1x128_e5m6(_p(x), M, K, x.stride(0), _p(xq), xq.stride(0),
                                          _p(sx), _stream(stream)), "fp8_quant_act_1x128_e5m6")
    return xq, sx


def fp8_quant_act_128x1(x, xqT=None, sxT=None, stream=None):
    """x: bf16 [M, K] -> (xqT uint8 [K, M], sxT f32 [M/128, K])."""
    _cuda(x, "x", torch.bfloat16)
    assert x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if xqT is None:
        xqT = torch.empty((K, M), dtype=torch.uint8, device=x.device)
    if sxT is None:
        sxT = torch.empty((M // 128, K), dtype=torch.float32, device=x.device)
    assert xqT.is_contiguous() and sxT.is_contiguous()
    _check(lib().fp8_quant_act_128x1(_p(x), M, K, x.stride(0), _p(xqT), _p(sxT),
                                     _stream(stream)), "fp8_quant_act_128x1")
    return xqT, sxT


def fp8_quant_act_dual(x, xq=None, sx=None, xqT=None, sxT=None, stream=None):
    """x: bf16 [M, K] -> (xq uint8 [M, K], sx f32 [K/128, M], xqT uint8 [K, M],
    sxT f32 [M/128, K]): fp8_quant_act_1x128 and fp8_quant_act_128x1 in one launch."""
    _cuda(x, "x", torch.bfloat16)
    assert x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    if xqT is None:
        xqT = torch.empty((K, M), dtype=torch.uint8, device=x.device)
    if sxT is None:
        sxT = torch.empty((M // 128, K), dtype=torch.float32, device=x.device)
    assert xq.stride(1) == 1 and sx.is_contiguous() and xqT.is_contiguous() and sxT.is_contiguous()
    _check(lib().fp8_quant_act_dual(_p(x), M, K, x.stride(0), _p(xq), xq.stride(0), _p(sx),
                                    _p(xqT), _p(sxT), _stream(stream)), "fp8_quant_act_dual")
    return xq, sx, xqT, sxT


def fp8_quant_weight_128x128(w, wq=None, wqT=None, sw=None, want_wq=True, want_wqT=False,
                             stream=None):
    """w: bf16 [K, N] -> (wq uint8 [N, K] or None, wqT uint8 [K, N] or None, sw f32 [N/128, K/128])."""
    _cuda(w, "w", torch.bfloat16)
    assert w.dim() == 2 and w.stride(1) == 1
    K, N = w.shape
    if wq is None and want_wq:
        wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if wqT is None and want_wqT:
        wqT = torch.empty((K, N), dtype=torch.uint8, device=w.device)
    if sw is None:
        sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    _check(lib().fp8_quant_weight_128x128(_p(w), K, N, w.stride(0), _p(wq), _p(wqT), _p(sw),
                                          _stream(stream)), "fp8_quant_weight_128x128")
    return wq, wqT, sw


def fp8_quant_fprop_operands(x, w, xq=None, sx=None, wq=None, wqT=None, sw=None, want_wq=True,
                             want_wqT=False, stream=None):
    """x: bf16 [M, K], w: bf16 [K, N] in one launch ->
    (xq uint8 [M, K], sx f32 [K/128, M], wq [N, K] or None, wqT [K, N] or None,
    sw f32 [N/128, K/128]); the same bits as fp8_quant_act_1x128 and
    fp8_quant_weight_128x128."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(w, "w", torch.bfloat16)
    assert x.dim() == 2 and x.stride(1) == 1 and w.dim() == 2 and w.stride(1) == 1
    M, K = x.shape
    K2, N = w.shape
    if K != K2:
        raise ValueError("x and w disagree on K: %d vs %d" % (K, K2))
    dev = x.device
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    if sx is None:
        sx = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    if wq is None and want_wq:
        wq = torch.empty((N, K), dtype=torch.uint8, device=dev)
    if wqT is None and want_wqT:
        wqT = torch.empty((K, N), dtype=torch.uint8, device=dev)
    if sw is None:
        sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
    assert xq.stride(1) == 1 and sx.is_contiguous() and sw.is_contiguous()
    assert (wq is None or wq.is_contiguous()) and (wqT is None or wqT.is_contiguous())
    _check(lib().fp8_quant_fprop_operands(_p(x), M, K, x.stride(0), _p(xq), xq.stride(0), _p(sx),
                                          _p(w), N, w.stride(0), _p(wq), _p(wqT), _p(sw),
                                          _stream(stream)), "fp8_quant_fprop_operands")
    return xq, sx, wq, wqT, sw


# -------------------------------------------------------------------- GEMMs --
def fp8_gemm_blockscaled_workspace_size():
    """Bytes of the split-K workspace on the current device."""
    n = lib().fp8_gemm_blockscaled_workspace_size()
    if n < 0:
        raise Fp8Error(5, "fp8_gemm_blockscaled_workspace_size")  # FP8_ERR_CUDA
    return n


def fp8_gemm_blockscaled(aq, sa, bq, sb, bmode=FP8_BSCALE_BLOCK128, out_dtype=torch.bfloat16,
                         c=None, stream=None, workspace=None):
    """C[M, N] of the block-scaled product; aq uint8 [M, K], bq uint8 [N, K].
    workspace: a zero-filled uint8 device tensor of
    fp8_gemm_blockscaled_workspace_size() bytes enables the split-K tail."""
    for t, n in ((aq, "aq"), (sa, "sa"), (bq, "bq"), (sb, "sb")):
        _cuda(t, n)
    M, K = aq.shape
    N = bq.shape[0]
    assert aq.is_contiguous() and bq.is_contiguous() and bq.shape[1] == K
    out_type = FP8_OUT_BF16 if out_dtype == torch.bfloat16 else FP8_OUT_F32
    if c is None:
        c = torch.empty((M, N), dtype=out_dtype, device=aq.device)
    assert c.stride(1) == 1
    if workspace is None:
        _check(lib().fp8_gemm_blockscaled(_p(aq), _p(sa), _p(bq), _p(sb), int(bmode), M, N, K,
                                          _p(c), c.stride(0), out_type, _stream(stream)),
               "fp8_gemm_blockscaled")
    else:
        _cuda(workspace, "workspace", torch.uint8)
        _check(lib().fp8_gemm_blockscaled_ws(_p(aq), _p(sa), _p(bq), _p(sb), int(bmode), M, N, K,
                                             _p(c), c.stride(0), out_type, _p(workspace),
                                             workspace.numel(), _stream(stream)),
               "fp8_gemm_blockscaled_ws")
    return c


# ------------------------------------------- activation quantisation fused in --
def fp8_gemm_blockscaled_bf16a(x, bq, sb, bmode=FP8_BSCALE_BLOCK128, out_dtype=torch.bfloat16,
                               c=None, stream=None):
    """C[M, N] from bf16 x [M, K] (quantised 1x128 inside the GEMM) and bq uint8 [N, K]."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(bq, "bq", torch.uint8)
    _cuda(sb, "sb", torch.float32)
    assert x.dim() == 2 and x.stride(1) == 1 and bq.is_contiguous()
    M, K = x.shape
    N = bq.shape[0]
    out_type = FP8_OUT_BF16 if out_dtype == torch.bfloat16 else FP8_OUT_F32
    if c is None:
        c = torch.empty((M, N), dtype=out_dtype, device=x.device)
    assert c.stride(1) == 1
    _check(lib().fp8_gemm_blockscaled_bf16a(_p(x), x.stride(0), _p(bq), _p(sb), int(bmode), M, N,
                                            K, _p(c), c.stride(0), out_type, _stream(stream)),
           "fp8_gemm_blockscaled_bf16a")
    return c


def fp8_grouped_gemm_moe_bf16a(x, bq, sb, offsets, out_dtype=torch.bfloat16, c=None,
                               stream=None):
    """Y[T, N] per expert from bf16 x [T, K] (quantised 1x128 inside the GEMM)."""
    _cuda(x, "x", torch.bfloat16)
    for t, n in ((bq, "bq"), (sb, "sb"), (offsets, "offsets")):
        _cuda(t, n)
    assert x.dim() == 2 and x.stride(1) == 1 and offsets.dtype == torch.int32
    T, K = x.shape
    E, N, _ = bq.shape
    out_type = FP8_OUT_BF16 if out_dtype == torch.bfloat16 else FP8_OUT_F32
    if c is None:
        c = torch.empty((T, N), dtype=out_dtype, device=x.device)
    assert c.is_contiguous()
    _check(lib().fp8_grouped_gemm_moe_bf16a(_p(x), x.stride(0), _p(bq), _p(sb), _p(offsets), E, T,
                                            N, K, _p(c), out_type, _stream(stream)),
           "fp8_grouped_gemm_moe_bf16a")
    return c


# ------------------------------------------------ MXFP8 (power-of-two) variant --
def fp8_quant_act_1x128_pow2(x, xq=None, se8=None, stream=None):
    """x: bf16 [M, K] -> (xq uint8 [M, K], se8 uint8 [K/128, M] UE8M0 exponents)."""
    _cuda(x, "x", torch.bfloat16)
    assert x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if se8 is None:
        se8 = torch.empty((K // 128, M), dtype=torch.uint8, device=x.device)
    assert xq.stride(1) == 1 and se8.is_contiguous()
    _check(lib().fp8_quant_act_1x128_pow2(_p(x), M, K, x.stride(0), _p(xq), xq.stride(0),
                                          _p(se8), _stream(stream)), "fp8_quant_act_1x128_pow2")
    return xq, se8


def fp8_quant_weight_128x128_pow2(w, wq=None, se8=None, stream=None):
    """w: bf16 [K, N] -> (wq uint8 [N, K], se8 uint8 [K/128, N] per-row UE8M0 exponents)."""
    _cuda(w, "w", torch.bfloat16)
    assert w.dim() == 2 and w.stride(1) == 1
    K, N = w.shape
    if wq is None:
        wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if se8 is None:
        se8 = torch.empty((K // 128, N), dtype=torch.uint8, device=w.device)
    assert wq.is_contiguous() and se8.is_contiguous()
    _check(lib().fp8_quant_weight_128x128_pow2(_p(w), K, N, w.stride(0), _p(wq), _p(se8),
                                               _stream(stream)), "fp8_quant_weight_128x128_pow2")
    return wq, se8


def fp8_gemm_mxfp8(aq, sa_e8, bq, sb_e8, out_dtype=torch.bfloat16, c=None, stream=None):
    """C[M, N] on the block-scaled tensor-core path; aq uint8 [M, K], sa_e8 uint8 [K/128, M],
    bq uint8 [N, K], sb_e8 uint8 [K/128, N]."""
    for t, n in ((aq, "aq"), (sa_e8, "sa_e8"), (bq, "bq"), (sb_e8, "sb_e8")):
        _cuda(t, n, torch.uint8)
    M, K = aq.shape
    N = bq.shape[0]
    assert aq.is_contiguous() and bq.is_contiguous() and bq.shape[1] == K
    assert sa_e8.is_contiguous() and sb_e8.is_contiguous()
    out_type = FP8_OUT_BF16 if out_dtype == torch.bfloat16 else FP8_OUT_F32
    if c is None:
        c = torch.empty((M, N), dtype=out_dtype, device=aq.device)
    assert c.stride(1) == 1
    _check(lib().fp8_gemm_mxfp8(_p(aq), _p(sa_e8), _p(bq), _p(sb_e8), M, N, K, _p(c), c.stride(0),
                                out_type, _stream(stream)), "fp8_gemm_mxfp8")
    return c


def _grouped(fn, name, aq, sa, bq, sb, offsets, out_dtype, c, stream):
    for t, n in ((aq, "aq"), (sa, "sa"), (bq, "bq"), (sb, "sb"), (offsets, "offsets")):
        _cuda(t, n)
    assert offsets.dtype == torch.int32
    T, K = aq.shape
    E, N, _ = bq.shape
    out_type = FP8_OUT_BF16 if out_dtype == torch.bfloat16 else FP8_OUT_F32
    if c is None:
        c = torch.empty((T, N), dtype=out_dtype, device=aq.device)
    assert c.is_contiguous()
    _check(fn(_p(aq), _p(sa), _p(bq), _p(sb), _p(offsets), E, T, N, K, _p(c), out_type,
              _stream(stream)), name)
    return c


def fp8_grouped_gemm_moe(aq, sa, bq, sb, offsets, out_dtype=torch.bfloat16, c=None,
                         stream=None):
    """Y[T, N] per expert; aq uint8 [T, K], bq uint8 [E, N, K], offsets int32 [E+1] (device)."""
    return _grouped(lib().fp8_grouped_gemm_moe, "fp8_grouped_gemm_moe", aq, sa, bq, sb, offsets,
                    out_dtype, c, stream)


def fp8_grouped_gemm_moe_dgrad(aq, sa, bqT, sw, offsets, out_dtype=torch.bfloat16, c=None,
                               stream=None):
    """dX[T, N] per expert from dY codes aq [T, K]; bqT uint8 [E, N, K] (each expert's wqT),
    sw f32 [E, K/128, N/128] (each expert's Fprop weight scales)."""
    return _grouped(lib().fp8_grouped_gemm_moe_dgrad, "fp8_grouped_gemm_moe_dgrad", aq, sa, bqT,
                    sw, offsets, out_dtype, c, stream)


# ------------------------------------------------------------- MoE dispatch --
def fp8_moe_dispatch_workspace_size(T, n_local) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().fp8_moe_dispatch_workspace_size(T, n_local, ctypes.byref(n)),
           "fp8_moe_dispatch_workspace_size")
    return n.value


def moe_dispatch_workspace(T, n_local, device="cuda"):
    """Device workspace for fp8_moe_dispatch_quant (uninitialised; None when T = 0)."""
    n = fp8_moe_dispatch_workspace_size(T, n_local)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def fp8_moe_dispatch_quant(x, topk_ids, expert_begin, n_local, cap=None, xq=None, sx=None,
                           offsets=None, token_ids=None, workspace=None, stream=None):
    """x bf16 [T, K], topk_ids int32 [T, topk] -> (xq uint8 [cap, K], sx f32 [K/128, cap],
    offsets int32 [n_local+1], token_ids int32 [cap]); rows of local expert e at
    offsets[e]:offsets[e+1], tokens ascending."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(topk_ids, "topk_ids", torch.int32)
    assert x.dim() == 2 and x.stride(1) == 1 and topk_ids.is_contiguous()
    T, K = x.shape
    topk = topk_ids.shape[1] if topk_ids.dim() == 2 else 1
    assert topk_ids.shape[0] == T
    if cap is None:
        cap = T * min(topk, n_local)
    dev = x.device
    if xq is None:
        xq = torch.empty((cap, K), dtype=torch.uint8, device=dev)
    if sx is None:
        sx = torch.empty((K // 128, cap), dtype=torch.float32, device=dev)
    if offsets is None:
        offsets = torch.empty(n_local + 1, dtype=torch.int32, device=dev)
    if token_ids is None:
        token_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = moe_dispatch_workspace(T, n_local, dev)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fp8_moe_dispatch_quant(_p(x), T, K, x.stride(0), _p(topk_ids), topk,
                                        expert_begin, n_local, _p(xq), _p(sx), cap, _p(offsets),
                                        _p(token_ids), _p(workspace), nbytes, _stream(stream)),
           "fp8_moe_dispatch_quant")
    return xq, sx, offsets, token_ids


def fp8_moe_dispatch_quant_noalloc(x, topk_ids, expert_begin, n_local, cap=None, xq=None,
                                   sx=None, offsets=None, token_ids=None, stream=None):
    """fp8_moe_dispatch_quant on the library's fixed device scratch (no workspace)."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(topk_ids, "topk_ids", torch.int32)
    assert x.dim() == 2 and x.stride(1) == 1 and topk_ids.is_contiguous()
    T, K = x.shape
    topk = topk_ids.shape[1] if topk_ids.dim() == 2 else 1
    assert topk_ids.shape[0] == T
    if cap is None:
        cap = T * min(topk, n_local)
    dev = x.device
    if xq is None:
        xq = torch.empty((cap, K), dtype=torch.uint8, device=dev)
    if sx is None:
        sx = torch.empty((K // 128, cap), dtype=torch.float32, device=dev)
    if offsets is None:
        offsets = torch.empty(n_local + 1, dtype=torch.int32, device=dev)
    if token_ids is None:
        token_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    _check(lib().fp8_moe_dispatch_quant_noalloc(_p(x), T, K, x.stride(0), _p(topk_ids), topk,
                                                expert_begin, n_local, _p(xq), _p(sx), cap,
                                                _p(offsets), _p(token_ids), _stream(stream)),
           "fp8_moe_dispatch_quant_noalloc")
    return xq, sx, offsets, token_ids


# ---------------------------------------------------------- MoE Wgrad path --
def padded_tokens(T, E):
    """Column capacity Tp that fp8_quant_act_128x1_grouped needs for T rows over E experts."""
    return ((T + 127 * E + 127) // 128) * 128


def fp8_quant_act_128x1_grouped(x, offsets, E, Tp=None, xqT=None, sxT=None, pofs=None,
                                stream=None):
    """x bf16 [T, K], offsets int32 [E+1] (device) -> (xqT uint8 [K, Tp], sxT f32 [Tp/128, K],
    pofs int32 [E+1]): per-expert 128-token groups, short groups zero-padded."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(offsets, "offsets", torch.int32)
    assert x.dim() == 2 and x.stride(1) == 1
    T, K = x.shape
    if Tp is None:
        Tp = padded_tokens(T, E)
    if xqT is None:
        xqT = torch.empty((K, Tp), dtype=torch.uint8, device=x.device)
    if sxT is None:
        sxT = torch.empty((Tp // 128, K), dtype=torch.float32, device=x.device)
    if pofs is None:
        pofs = torch.empty(E + 1, dtype=torch.int32, device=x.device)
    _check(lib().fp8_quant_act_128x1_grouped(_p(x), T, K, x.stride(0), _p(offsets), E, _p(xqT),
                                             _p(sxT), Tp, _p(pofs), _stream(stream)),
           "fp8_quant_act_128x1_grouped")
    return xqT, sxT, pofs


def fp8_grouped_gemm_moe_wgrad(aqT, sa, bqT, sb, pofs, c=None, stream=None):
    """dW [E, M, N] FP32 from aqT uint8 [M, Tp], sa [Tp/128, M], bqT uint8 [N, Tp],
    sb [Tp/128, N], pofs int32 [E+1] (device)."""
    for t, n in ((aqT, "aqT"), (sa, "sa"), (bqT, "bqT"), (sb, "sb"), (pofs, "pofs")):
        _cuda(t, n)
    M, Tp = aqT.shape
    N = bqT.shape[0]
    E = pofs.numel() - 1
    if c is None:
        c = torch.empty((E, M, N), dtype=torch.float32, device=aqT.device)
    assert c.is_contiguous() and c.dtype == torch.float32
    _check(lib().fp8_grouped_gemm_moe_wgrad(_p(aqT), _p(sa), _p(bqT), _p(sb), _p(pofs), E, Tp, M,
                                            N, _p(c), _stream(stream)),
           "fp8_grouped_gemm_moe_wgrad")
    return c
