"""Codebooks used by the library, derived in fp64 with torch and rounded once to
fp32.

``nf4_code4``: the 16 NormalFloat levels (QLoRA, Dettmers et al. 2023, section 3):
standard-normal quantiles at probabilities spaced evenly from 1 - delta down to
1/2 -- eight on the positive side, seven mirrored on the negative side -- plus an
exact zero, all divided by the largest so the extremes are exactly -1 and +1;
delta = (1/30 + 1/32) / 2.  The pages name the type ("nf4", bitsandbytes issue
"MatMul4Bit keeps B and quant_state on ctx", "Minimal reproducer") without
printing it.

``dynamic_code8``: the signed 8-bit dynamic tree map (Dettmers et al. 2022,
"8-bit Optimizers via Block-wise Quantization") for the nested absmax codes:
decimal exponent groups 10**(e-6), e = 0..6, holding 2**e linear fraction values
each (bin midpoints of [0.1, 1]), both signs, plus 0 and 1.
"""
from __future__ import annotations

import torch

_DELTA = (1.0 / 30.0 + 1.0 / 32.0) / 2.0


def nf4_code4() -> torch.Tensor:
    hi = 1.0 - _DELTA
    p_pos = torch.linspace(hi, 0.5, 9, dtype=torch.float64)[:-1]
    p_neg = torch.linspace(hi, 0.5, 8, dtype=torch.float64)[:-1]
    levels = torch.cat([torch.special.ndtri(p_pos), -torch.special.ndtri(p_neg),
                        torch.zeros(1, dtype=torch.float64)])
    levels, _ = torch.sort(levels)
    return (levels / levels.max()).to(torch.float32)


def dynamic_code8() -> torch.Tensor:
    parts = []
    for e in range(7):
        edges = torch.linspace(0.1, 1.0, 2 ** e + 1, dtype=torch.float64)
        parts.append((edges[:-1] + edges[1:]) / 2.0 * (10.0 ** (e - 6)))
    mags = torch.cat(parts)
    levels = torch.cat([mags, -mags, torch.tensor([0.0, 1.0], dtype=torch.float64)])
    levels, _ = torch.sort(levels)
    return levels.to(torch.float32)
