"""Seeded synthetic inputs with the shapes and value distributions of the
workloads the method is measured on.  This module holds none of the method's
arithmetic (no quantisation, no dequantisation, no products): it only draws
random tensors and routing patterns, so that the GPU path and the CPU oracle can
be fed the very same inputs.

Distributions (those of the benchmark workloads): weights ~ N(0, 0.02) fp32, activations
and output gradients ~ N(0, 1) rounded to bf16, MoE router logits ~ U(0, 1).
Everything is drawn from a CPU ``torch.Generator`` in a fixed order, then moved
to the device by the caller.
"""
from __future__ import annotations

import torch

WEIGHT_STD = 0.02

# Projection shapes (name, K = in_features, N = out_features).
LLAMA8B_PROJ = [("q", 4096, 4096), ("k", 4096, 1024), ("v", 4096, 1024), ("o", 4096, 4096),
                ("gate", 4096, 14336), ("up", 4096, 14336), ("down", 14336, 4096)]
QWEN32B_PROJ = [("q", 5120, 5120), ("k", 5120, 1024), ("v", 5120, 1024), ("o", 5120, 5120),
                ("gate", 5120, 27648), ("up", 5120, 27648), ("down", 27648, 5120)]
M_SWEEP = [1, 8, 32, 128, 512, 1536, 2048, 4096, 8192]
OLMOE = dict(experts=64, hidden=2048, inter=1024, tokens=512, topk=8)


def generator(seed: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def weight(N: int, K: int, g: torch.Generator, std: float = WEIGHT_STD) -> torch.Tensor:
    """fp32 [N, K] ~ N(0, std^2)."""
    return torch.randn(N, K, generator=g, dtype=torch.float32) * std


def activation(M: int, K: int, g: torch.Generator) -> torch.Tensor:
    """bf16 [M, K] ~ N(0, 1)."""
    return torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)


def routing(tokens: int, experts: int, topk: int, g: torch.Generator):
    """Top-k routing from U(0,1) logits (ties to the lower expert index), then a
    stable sort of the (token, expert) pairs by expert.

    Returns (row_token int64 [tokens*topk], offsets int32 [experts+1]): grouped row
    r holds token row_token[r], and rows offsets[e]..offsets[e+1]-1 go to expert e."""
    logits = torch.rand(tokens, experts, generator=g, dtype=torch.float32)
    order = torch.sort(-logits, dim=1, stable=True).indices[:, :topk]  # [tokens, topk]
    tok = torch.arange(tokens).unsqueeze(1).expand(tokens, topk).reshape(-1)
    exp = order.reshape(-1)
    perm = torch.sort(exp, stable=True).indices
    row_token = tok[perm].contiguous()
    counts = torch.bincount(exp, minlength=experts)
    offsets = torch.zeros(experts + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    return row_token, offsets
