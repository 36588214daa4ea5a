"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no FP8 arithmetic: it only draws bfloat16 tensors with the
shapes and value distributions of the workloads the DeepSeek-V3 Technical
Report trains and serves (section 3.3 FP8 Training; section 3.4.2 Decoding for
the small per-expert batches), and a skewed MoE routing.  Random numbers come
from ``torch.Generator`` seeded explicitly; every workload draws its tensors
from one generator in the order listed in its builder.

Distributions:
  activations  ACT(M, K): N(0, 1), with max(1, round(0.01 K)) randomly chosen
               K-channels multiplied by 100 (outlier channels), then bf16 (RNE).
  weights      W(K, N): N(0, 0.006^2) -> bf16.
  gradients    dY(M, N): N(0, 1e-3^2) -> bf16.
  routing      logits N(0,1) [T, 256], per-expert bias N(0, 0.5^2); score =
               sigmoid(logit) + bias; top-8 per token (ties: lower expert
               index); experts 0..31 are the local ones; each expert's tokens
               in ascending token order.
  decode       t_e uniform in [1, 256] per expert.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def act(M: int, K: int, g: torch.Generator, device="cpu") -> torch.Tensor:
    x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    n_out = max(1, int(round(0.01 * K)))
    idx = torch.randperm(K, generator=g, device=device)[:n_out]
    x[:, idx] *= 100.0
    return x.to(torch.bfloat16)


def weight(K: int, N: int, g: torch.Generator, device="cpu", std=0.006) -> torch.Tensor:
    return (torch.randn(K, N, generator=g, device=device, dtype=torch.float32) * std).to(
        torch.bfloat16)


def grad(M: int, N: int, g: torch.Generator, device="cpu") -> torch.Tensor:
    return (torch.randn(M, N, generator=g, device=device, dtype=torch.float32) * 1e-3).to(
        torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bfloat16 bit patterns of a (CPU or device) tensor as a uint16 numpy array."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def moe_topk(T: int, n_experts: int, topk: int, g: torch.Generator) -> torch.Tensor:
    """Top-k expert ids [T, topk] (int64) of a sigmoid-plus-bias router."""
    logits = torch.randn(T, n_experts, generator=g, dtype=torch.float32)
    bias = torch.randn(n_experts, generator=g, dtype=torch.float32) * 0.5
    score = torch.sigmoid(logits) + bias
    # stable descending sort: among equal scores the lower expert index wins
    return torch.sort(score, dim=1, descending=True, stable=True).indices[:, :topk]


def local_routing(order: torch.Tensor, n_local: int, expert_begin: int = 0):
    """Token ids per local expert (concatenated, expert-major, ascending) and offsets."""
    tokens, counts = [], []
    for e in range(n_local):
        tok = torch.nonzero((order == expert_begin + e).any(dim=1)).flatten()
        tokens.append(tok)
        counts.append(tok.numel())
    token_ids = torch.cat(tokens).to(torch.int64)
    offsets = np.zeros(n_local + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    return token_ids, offsets


def moe_routing(T: int, n_experts: int, topk: int, n_local: int, g: torch.Generator):
    """Token ids per local expert (concatenated, expert-major) and offsets [n_local+1]."""
    return local_routing(moe_topk(T, n_experts, topk, g), n_local)


def decode_counts(E: int, g: torch.Generator, lo=1, hi=256) -> np.ndarray:
    return torch.randint(lo, hi + 1, (E,), generator=g).numpy().astype(np.int64)


# --------------------------------------------------------------- workloads --
@dataclass
class Dense:
    """One dense GEMM Y[M, N] = X[M, K] . W[K, N] with its bf16 inputs."""
    name: str
    M: int
    N: int
    K: int
    x: torch.Tensor
    w: torch.Tensor
    out_f32: bool


@dataclass
class Trio:
    """Expert-MLP training trio: Fprop X.W, Dgrad dY.W^T, Wgrad X^T.dY."""
    name: str
    M: int
    K: int
    N: int
    x: torch.Tensor
    w: torch.Tensor
    dy: torch.Tensor


@dataclass
class Grouped:
    """Grouped per-expert GEMM over rows grouped by expert (offsets [E+1])."""
    name: str
    E: int
    N: int
    K: int
    x: torch.Tensor          # [T, K] bf16, rows grouped by expert
    w: torch.Tensor          # [E, K, N] bf16
    offsets: np.ndarray      # int64 [E+1]
    extra: dict = field(default_factory=dict)


def small_dense(seed=0, device="cpu") -> Dense:
    """M=128, N=256, K=512; activations 1x128, weights 128x128; FP32 output."""
    g = _gen(seed, device)
    x = act(128, 512, g, device)
    w = weight(512, 256, g, device)
    return Dense("gemm_m128_n256_k512_f32", 128, 256, 512, x, w, True)


def fprop_dense(seed=0, device="cpu") -> Dense:
    """Shared-expert down-projection: X[8192, 2048] . W[2048, 7168] -> BF16 Y."""
    g = _gen(seed, device)
    x = act(8192, 2048, g, device)
    w = weight(2048, 7168, g, device)
    return Dense("fprop_m8192_n7168_k2048_bf16", 8192, 7168, 2048, x, w, False)


def training_trio(seed=0, device="cpu", M=8192, K=7168, N=4096) -> Trio:
    """Fprop X[M,K].W[K,N], Dgrad dY[M,N].W^T, Wgrad X^T.dY."""
    g = _gen(seed, device)
    x = act(M, K, g, device)
    w = weight(K, N, g, device)
    dy = grad(M, N, g, device)
    return Trio("trio_m%d_k%d_n%d" % (M, K, N), M, K, N, x, w, dy)


def moe_prefill(seed=0, device="cpu", T=16384, K=7168, N=4096, n_experts=256, topk=8,
                n_local=32) -> Grouped:
    """Top-8-of-256 routing of T tokens, 32 local experts with W[K, N] each."""
    g = _gen(seed)  # routing is drawn on the host
    x_tok = act(T, K, g)
    order = moe_topk(T, n_experts, topk, g)
    token_ids, offsets = local_routing(order, n_local)
    gw = _gen(seed + 1, device)
    w = torch.stack([weight(K, N, gw, device) for _ in range(n_local)])
    x = x_tok[token_ids].to(device)
    return Grouped("moe_prefill_t%d_e%d_k%d_n%d" % (T, n_local, K, N), n_local, N, K, x, w,
                   offsets, {"token_ids": token_ids, "topk_ids": order, "x_tokens": x_tok})


def moe_decode(seed=0, device="cpu", E=32, K=7168, N=4096, max_tokens=256) -> Grouped:
    """E experts, each with t_e ~ U[1, max_tokens] rows; memory-bound regime."""
    g = _gen(seed)
    counts = decode_counts(E, g, 1, max_tokens)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    T = int(offsets[-1])
    x = act(T, K, g).to(device)
    gw = _gen(seed + 1, device)
    w = torch.stack([weight(K, N, gw, device) for _ in range(E)])
    return Grouped("moe_decode_e%d_k%d_n%d_tmax%d" % (E, K, N, max_tokens), E, N, K, x, w,
                   offsets)
