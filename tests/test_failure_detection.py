"""Failure detection without a GPU fault: a bounded barrier wait that nothing
completes gives up after its limit (about two seconds), the kernel returns,
fp8_device_error() reports FP8_ERR_TIMEOUT, and the context stays usable."""
import time

import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_22_b300 import fp8fg, inputs
from parity import bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_bounded_wait_times_out_and_the_context_survives():
    assert fp8fg.device_error() == 0
    t0 = time.time()
    fp8fg.selftest_wait_timeout()
    status = fp8fg.device_error()  # synchronises
    dt = time.time() - t0
    assert status == 6, status  # FP8_ERR_TIMEOUT
    assert dt < 60
    assert fp8fg.device_error() == 0  # reading the word clears it
    # the context still runs kernels correctly
    wl = inputs.small_dense(seed=3)
    xq, sx = fp8fg.fp8_quant_act_1x128(wl.x.to(DEV))
    wq, _, sw = fp8fg.fp8_quant_weight_128x128(wl.w.to(DEV))
    y = fp8fg.fp8_gemm_blockscaled(xq, sx, wq, sw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fp8fg.device_error() == 0
    aq, sa = oracle.quant_act_1x128(bits(wl.x))
    bq, _, sb = oracle.quant_weight_128x128(bits(wl.w))
    ref = oracle.gemm_blockscaled(aq, sa, bq, sb)
    err = np.linalg.norm(y.cpu().numpy() - ref) / np.linalg.norm(ref)
    assert err <= 1e-5
