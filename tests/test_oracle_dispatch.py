"""Pins of the oracle's MoE dispatch packing (CPU).

The packing follows the DeepSeek-V3 Technical Report, section 3.3.3 (FP8
dispatch of the activations with 1x128 scales) and section 3.4 (top-k
routing to experts): rows of local expert e are the tokens routed to it in
ascending order, quantised 1x128.
"""
import numpy as np
import torch

import oracle
from fp8_fine_grained_22_b300 import inputs
from parity import bits


def _x(T, K, seed):
    return bits(inputs.act(T, K, torch.Generator().manual_seed(seed)))


def test_hand_worked_example():
    # global experts 1..3 are local (expert_begin 1, three experts).
    # token 0 -> {1, 3}; token 1 -> {0, 2}; token 2 -> {2, 1}; token 3 -> {3} (repeated);
    # token 4 -> {4, 0}: none local.  Local expert 0 (global 1): tokens 0, 2;
    # expert 1 (global 2): tokens 1, 2; expert 2 (global 3): tokens 0, 3.
    ids = np.array([[1, 3], [0, 2], [2, 1], [3, 3], [4, 0]])
    x = _x(5, 256, 1)
    xq, sx, offsets, token_ids = oracle.moe_dispatch_quant(x, ids, 1, 3)
    assert offsets.tolist() == [0, 2, 4, 6]
    assert token_ids.tolist() == [0, 2, 1, 2, 0, 3]
    assert xq.shape == (6, 256) and sx.shape == (2, 6)


def test_quantisation_commutes_with_the_gather():
    """1x128 groups are row-local: quantise-then-gather gives the same bits."""
    T, K = 300, 512
    x = _x(T, K, 2)
    ids = torch.randint(0, 40, (T, 4), generator=torch.Generator().manual_seed(3)).numpy()
    xq, sx, offsets, token_ids = oracle.moe_dispatch_quant(x, ids, 8, 16)
    xq_all, sx_all = oracle.quant_act_1x128(x)
    assert np.array_equal(xq, xq_all[token_ids])
    assert np.array_equal(sx, sx_all[:, token_ids])


def test_membership_counts_and_order():
    T = 257
    g = torch.Generator().manual_seed(4)
    ids = torch.randint(-5, 70, (T, 6), generator=g).numpy()  # repeats and non-local ids
    x = _x(T, 128, 5)
    begin, n_local = 10, 32
    _, _, offsets, token_ids = oracle.moe_dispatch_quant(x, ids, begin, n_local)
    for e in range(n_local):
        rows = token_ids[offsets[e]:offsets[e + 1]]
        brute = [t for t in range(T) if (begin + e) in set(ids[t].tolist())]
        assert rows.tolist() == brute
    assert np.all(np.diff(offsets) >= 0)


def test_matches_the_workload_routing():
    """The prefill workload's own gather (torch) and the oracle agree."""
    g = torch.Generator().manual_seed(0)
    order = inputs.moe_topk(2048, 256, 8, g)
    tok_ref, off_ref = inputs.local_routing(order, 32)
    x = _x(2048, 128, 6)
    _, _, offsets, token_ids = oracle.moe_dispatch_quant(x, order.numpy(), 0, 32)
    assert np.array_equal(offsets, off_ref)
    assert np.array_equal(token_ids, tok_ref.numpy())


def test_no_tokens_and_no_local_hits():
    x = np.zeros((0, 256), np.uint16)
    xq, sx, offsets, token_ids = oracle.moe_dispatch_quant(x, np.zeros((0, 2), np.int64), 0, 4)
    assert offsets.tolist() == [0] * 5 and xq.shape == (0, 256) and token_ids.size == 0
    x = _x(3, 128, 7)
    xq, sx, offsets, token_ids = oracle.moe_dispatch_quant(x, np.full((3, 2), 99), 0, 4)
    assert offsets.tolist() == [0] * 5 and xq.shape == (0, 128)
