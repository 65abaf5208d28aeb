"""Codebooks used by the library, derived in fp64 with torch and rounded once to
fp32.

``nf4_code4``: the 16 NormalFloat levels (QLoRA, Dettmers et al. 2023, section 3):
standard-normal quantiles at probabilities spaced evenly from 1 - delta down to
1/2 -- eight on the positive side, seven mirrored on the negative side -- plus an
exact zero, all divided by the largest so the extremes are exactly -1 and +1;
delta = (1/30 + 1/32) / 2.  The pages name the type ("nf4", bitsandbytes issue
"MatMul4Bit keeps B and quant_state on ctx", "Minimal reproducer") without
printing it.

``fp4_code4``: the "fp4" quant_type that the pages list beside nf4 for the same
packed 4-bit path (fork PR "Experts trainability", commit 1, quant_type table),
read as the E2M1 4-bit float (sign, 2-bit exponent with bias 1, 1-bit mantissa,
subnormals at exponent 0) scaled by 1/6 so its extremes are +-1, in ascending
order with -0 before +0.

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


def fp4_code4() -> torch.Tensor:
    bits = torch.arange(16, dtype=torch.int64)
    sign = torch.where(bits >= 8, -1.0, 1.0).to(torch.float64)
    exp = (bits >> 1) & 3
    man = (bits & 1).to(torch.float64)
    mag = torch.where(exp == 0, man * 0.5,
                      (1.0 + man * 0.5) * torch.pow(2.0, (exp - 1).to(torch.float64)))
    vals = sign * mag / 6.0
    # The magnitude grows with the low three bits, so ascending order (-0 before
    # +0) is codes 15 down to 8, then 0 up to 7.
    order = torch.cat([torch.arange(15, 7, -1), torch.arange(0, 8)])
    return vals[order].to(torch.float32)


def code4_for(quant_type: str) -> torch.Tensor:
    """The 16-entry codebook of a 4-bit quant_type ("nf4" or "fp4")."""
    if quant_type == "nf4":
        return nf4_code4()
    if quant_type == "fp4":
        return fp4_code4()
    raise ValueError(f"unknown 4-bit quant_type {quant_type!r} (expected 'nf4' or 'fp4')")


def dynamic_code8() -> torch.Tensor:
    parts = []
    for e in range(7):
        edges = torch.linspace(0.1, 1.0, 2 ** e + 1, dtype=torch.float64)
        parts.append((edges[:-1] + edges[1:]) / 2.0 * (10.0 ** (e - 6)))
    mags = torch.cat(parts)
    levels = torch.cat([mags, -mags, torch.tensor([0.0, 1.0], dtype=torch.float64)])
    levels, _ = torch.sort(levels)
    return levels.to(torch.float32)
