"""fp8_moe_dispatch_quant_noalloc (fixed device scratch) against the
workspace entry point fp8_moe_dispatch_quant: identical outputs, two calls
in a row, and the size limit of the fixed scratch.

Collected last (file name) so that it also runs after every other GPU test;
it needs nothing from them and passes alone.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_22_b300 import fp8fg, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _both(x, ids, begin, n_local):
    xg = x.to(DEV)
    idg = torch.as_tensor(ids, dtype=torch.int32).to(DEV).contiguous()
    ref = fp8fg.fp8_moe_dispatch_quant(xg, idg, begin, n_local)
    got = fp8fg.fp8_moe_dispatch_quant_noalloc(xg, idg, begin, n_local)
    torch.cuda.synchronize()
    R = int(ref[2][-1].item())
    assert torch.equal(got[2], ref[2])                     # offsets
    assert torch.equal(got[3][:R], ref[3][:R])             # source tokens
    assert torch.equal(got[0][:R], ref[0][:R])             # codes
    assert torch.equal(got[1][:, :R].view(torch.int32), ref[1][:, :R].view(torch.int32))
    return R


def test_matches_workspace_entry_point_two_calls_in_a_row():
    g = torch.Generator().manual_seed(21)
    # first call: wide routing; second: a different shape and routing on the same scratch
    x1 = inputs.act(1000, 512, g)
    ids1 = torch.randint(-2, 70, (1000, 8), generator=g)
    x2 = inputs.act(333, 1024, g)
    ids2 = torch.randint(0, 9, (333, 2), generator=g)
    assert _both(x1, ids1.numpy(), 4, 32) > 0
    assert _both(x2, ids2.numpy(), 0, 8) > 0


def test_prefill_routing():
    wl = inputs.moe_prefill()
    R = _both(wl.extra["x_tokens"], wl.extra["topk_ids"].numpy(), 0, wl.E)
    assert R == int(wl.offsets[-1])


def test_rejects_problems_beyond_the_fixed_scratch():
    # 32 local experts: n_local * ceil(T / 64) + n_local must stay <= 65536
    T, K, E = 131072, 128, 32
    x = torch.zeros((T, K), dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros((T, 1), dtype=torch.int32, device=DEV)
    with pytest.raises(fp8fg.Fp8Error) as e:
        fp8fg.fp8_moe_dispatch_quant_noalloc(x, ids, 0, E)
    assert e.value.status == 4  # FP8_ERR_UNSUPPORTED, nothing launched
    # the largest T that fits still runs
    T = 64 * (65536 // E - 1)
    R = _both(torch.zeros((T, K), dtype=torch.bfloat16), np.zeros((T, 1), np.int32), 0, E)
    assert R == T


# ------------------------------------------- a second context on the device --
def _driver():
    import ctypes
    cu = ctypes.CDLL("libcuda.so.1")
    return ctypes, cu


def _ck(r, what):
    assert r == 0, "%s returned CUresult %d" % (what, r)


def test_call_in_another_context_of_the_device():
    """The scratch address is looked up per CUDA context.  A caller that makes
    its own context current (driver API) gets that context's address of the
    scratch, not the one cached from the primary context that torch uses;
    back in the primary context the next call uses the primary's address
    again.  Every buffer of the call in the second context is allocated in
    that context, so no pointer crosses contexts."""
    ctypes, cu = _driver()
    g = torch.Generator().manual_seed(5)
    T, K, topk, E, begin = 700, 384, 4, 16, 2
    x = inputs.act(T, K, g)
    ids = torch.randint(0, 24, (T, topk), generator=g).to(torch.int32)
    # primary context (torch): fills the cache, gives the expected outputs
    R = _both(x, ids.numpy(), begin, E)
    ref = fp8fg.fp8_moe_dispatch_quant(x.to(DEV), ids.to(DEV), begin, E)
    torch.cuda.synchronize()
    ref = [t.cpu() for t in ref]
    cap = T * min(topk, E)

    dev = ctypes.c_int(0)
    _ck(cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()), "cuDeviceGet")
    ctx = ctypes.c_void_p(0)
    if hasattr(cu, "cuCtxCreate_v2"):
        _ck(cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, dev), "cuCtxCreate_v2")
    else:
        _ck(cu.cuCtxCreate_v4(ctypes.byref(ctx), None, 0, dev), "cuCtxCreate_v4")
    bufs = []
    try:
        def alloc(nbytes):
            p = ctypes.c_uint64(0)
            _ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc_v2")
            bufs.append(p)
            return p.value

        xh = np.ascontiguousarray(inputs.bf16_bits(x))
        idh = np.ascontiguousarray(ids.numpy())
        d_x, d_ids = alloc(xh.nbytes), alloc(idh.nbytes)
        d_xq, d_sx = alloc(cap * K), alloc((K // 128) * cap * 4)
        d_off, d_tok = alloc((E + 1) * 4), alloc(cap * 4)
        for d, h in ((d_x, xh), (d_ids, idh)):
            _ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(d), h.ctypes.data_as(ctypes.c_void_p),
                                   ctypes.c_size_t(h.nbytes)), "cuMemcpyHtoD_v2")
        P = ctypes.c_void_p
        for _ in range(2):  # the second call reuses the second context's cached address
            st = fp8fg.lib().fp8_moe_dispatch_quant_noalloc(
                P(d_x), T, K, K, P(d_ids), topk, begin, E, P(d_xq), P(d_sx), cap, P(d_off),
                P(d_tok), P(0))
            assert st == 0, fp8fg.status_str(st)
        _ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
        out_off = np.empty(E + 1, np.int32)
        out_tok = np.empty(cap, np.int32)
        out_xq = np.empty((cap, K), np.uint8)
        out_sx = np.empty((K // 128, cap), np.float32)
        for h, d in ((out_off, d_off), (out_tok, d_tok), (out_xq, d_xq), (out_sx, d_sx)):
            _ck(cu.cuMemcpyDtoH_v2(h.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(d),
                                   ctypes.c_size_t(h.nbytes)), "cuMemcpyDtoH_v2")
    finally:
        for p in bufs:
            cu.cuMemFree_v2(p)
        popped = ctypes.c_void_p(0)
        _ck(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent_v2")
        _ck(cu.cuCtxDestroy_v2(ctx), "cuCtxDestroy_v2")
    assert np.array_equal(out_off, ref[2].numpy())
    assert np.array_equal(out_tok[:R], ref[3].numpy()[:R])
    assert np.array_equal(out_xq[:R], ref[0].numpy()[:R])
    assert np.array_equal(out_sx[:, :R].view(np.int32), ref[1][:, :R].view(torch.int32).numpy())
    # back in the primary context: the cached entry belongs to the second
    # context, so this call looks the primary's address up again
    assert _both(x, ids.numpy(), begin, E) == R
