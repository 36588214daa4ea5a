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
