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

``e4m3_code8``: the "fp8" 8-bit weight storage ("e4m3 codebook", fork PR
"Experts trainability", commit 1, quant_type table), read as all 256 codes of a
1-4-3 float (exponent bias 7, subnormals at exponent 0, no special codes) scaled
by 1/480 so its extremes are +-1, ascending with -0 before +0.  The "int8"
storage of the same row uses ``dynamic_code8`` as its 256 levels.

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


def e4m3_code8() -> torch.Tensor:
    bits = torch.arange(256, dtype=torch.int64)
    sign = torch.where(bits >= 128, -1.0, 1.0).to(torch.float64)
    exp = (bits >> 3) & 15
    man = (bits & 7).to(torch.float64)
    mag = torch.where(exp == 0, man / 8.0 * 2.0 ** -6,
                      (1.0 + man / 8.0) * torch.pow(2.0, (exp - 7).to(torch.float64)))
    vals = sign * mag / 480.0
    # The magnitude grows with the low seven bits, so ascending order (-0 before
    # +0) is codes 255 down to 128, then 0 up to 127.
    order = torch.cat([torch.arange(255, 127, -1), torch.arange(0, 128)])
    return vals[order].to(torch.float32)


QUANT_TYPES = {"nf4": 4, "fp4": 4, "int8": 8, "fp8": 8}


def code_for(quant_type: str) -> torch.Tensor:
    """The value codebook of a quant_type: 16 levels for the packed 4-bit types
    ("nf4", "fp4"), 256 for the one-byte types ("int8": dynamic map, "fp8": e4m3)."""
    if quant_type == "nf4":
        return nf4_code4()
    if quant_type == "fp4":
        return fp4_code4()
    if quant_type == "int8":
        return dynamic_code8()
    if quant_type == "fp8":
        return e4m3_code8()
    raise ValueError(f"unknown quant_type {quant_type!r} (expected one of {sorted(QUANT_TYPES)})")


def code4_for(quant_type: str) -> torch.Tensor:
    """The 16-entry codebook of a 4-bit quant_type ("nf4" or "fp4")."""
    if QUANT_TYPES.get(quant_type) != 4:
        raise ValueError(f"unknown 4-bit quant_type {quant_type!r} (expected 'nf4' or 'fp4')")
    return code_for(quant_type)


def dynamic_code8() -> torch.Tensor:
    parts = []
    for e in range(7):
        edges = torch.linspace(0.1, 1.0, 2 ** e + 1, dtype=torch.float64)
        parts.append((edges[:-1] + edges[1:]) / 2.0 * (10.0 ** (e - 6)))
    mags = torch.cat(parts)
    levels = torch.cat([mags, -mags, torch.tensor([0.0, 1.0], dtype=torch.float64)])
    levels, _ = torch.sort(levels)
    return levels.to(torch.float32)
