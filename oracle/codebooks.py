"""Codebooks of the oracle, computed in fp64 from their definitions and rounded
once to fp32.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  The GPU package derives
its own tables with its own code; the tests check that the two agree bit for bit.

``nf4_code4`` -- the 4-bit NormalFloat levels.  The pages call the type "nf4"
(bitsandbytes issue "MatMul4Bit keeps B and quant_state on ctx", section
"Minimal reproducer": ``quantize_4bit(..., quant_type="nf4")``) but never print
its 16 values.  Reading: the NormalFloat construction of the QLoRA paper
(Dettmers et al., 2023, section 3, "4-bit NormalFloat"): levels are quantiles of
the standard normal, asymmetric so that an exact zero exists -- 8 positive levels
at the probabilities ``linspace(1 - delta, 1/2, 9)`` without the last point, 7
negative levels mirrored from ``linspace(1 - delta, 1/2, 8)`` without the last
point, plus 0 -- and the whole set divided by its largest value so that both
extremes are exactly +-1.  ``delta = (1/30 + 1/32) / 2``.

``fp4_code4`` -- the "fp4" quant_type, which the pages list beside nf4 as the
same packed 4-bit path (fork PR "Experts trainability", commit 1, quant_type
table, row "nf4 / fp4") without giving its levels.  Reading: the 16 codes of the
E2M1 4-bit float (1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit;
exponent 0 holds the subnormals 0 and 0.5), whose magnitudes are 0, 0.5, 1, 1.5,
2, 3, 4 and 6, divided by the largest (6) so that the extremes are exactly +-1,
and listed in ascending order with -0 before +0.  Because of that signed-zero
pair the table is non-decreasing rather than strictly increasing.  The midpoint
of the pair is 0, so a normalised value v quantises to index 7 (-0) when
-1/24 <= v <= 0 (an all-zero block included) and to index 8 (+0) when
0 < v <= 1/24 (the midpoint with 1/12 goes to the lower index).

``e4m3_code8`` -- the "fp8" 8-bit weight storage, which the pages describe as an
"e4m3 codebook" on the same blockwise path (fork PR "Experts trainability",
commit 1, quant_type table, row "fp8").  Reading: the 256 codes of a float with
1 sign bit, 4 exponent bits (bias 7) and 3 mantissa bits, exponent 0 holding the
subnormals, no code set aside for NaN or infinity; magnitudes m/8 * 2**-6 (e = 0)
and (1 + m/8) * 2**(e - 7) (e = 1..15), divided by the largest (480) so the
extremes are +-1, ascending with -0 before +0 (non-decreasing, as for fp4).  The
"int8" storage of the same table row uses ``dynamic_code8`` below as its 256
levels ("blockwise dynamic map").

``dynamic_code8`` -- the signed 8-bit dynamic ("tree") map used for the nested
absmax codes.  The pages name only "blockwise dynamic map" (fork PR "Experts
trainability", commit 1 table, int8 row); the nested statistics are 8-bit blockwise.
Reading: the dynamic tree quantisation of Dettmers et al., 2022 ("8-bit
Optimizers via Block-wise Quantization"): a sign, a run of leading zero bits that
sets a decimal exponent, an indicator bit, and the remaining bits a linear
fraction.  With 7 magnitude bits the exponent group e = 0..6 has 2**e fraction
values; each is the midpoint of one of 2**e equal bins of [0.1, 1], scaled by
10**(e - 6).  Both signs, plus an exact 0 and the value 1.0, give 256 levels.
"""
from __future__ import annotations

import numpy as np
from scipy.special import ndtri

NF4_DELTA = 0.5 * (1.0 / 30.0 + 1.0 / 32.0)


def nf4_code4_f64() -> np.ndarray:
    top = 1.0 - NF4_DELTA
    pos = ndtri(np.linspace(top, 0.5, 9)[:-1])  # 8 values, largest first
    neg = -ndtri(np.linspace(top, 0.5, 8)[:-1])  # 7 values
    levels = np.sort(np.concatenate([neg, [0.0], pos]))
    return levels / levels.max()


def nf4_code4() -> np.ndarray:
    """16 strictly increasing fp32 levels, code4[0] = -1, code4[7] = 0, code4[15] = 1."""
    return nf4_code4_f64().astype(np.float32)


def fp4_code4_f64() -> np.ndarray:
    mags = []
    for e in range(4):          # exponent field, bias 1
        for m in range(2):      # mantissa bit
            mags.append(m * 0.5 if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1))
    mags = np.array(mags) / max(mags)  # 0, 1/12, 1/6, 1/4, 1/3, 1/2, 2/3, 1
    return np.concatenate([-mags[::-1], mags])  # -1 ... -1/12, -0, +0, 1/12 ... 1


def fp4_code4() -> np.ndarray:
    """16 non-decreasing fp32 levels: -1 ... -1/12, -0, +0, 1/12 ... 1."""
    return fp4_code4_f64().astype(np.float32)


def e4m3_code8_f64() -> np.ndarray:
    mags = []
    for e in range(16):        # exponent field, bias 7
        for m in range(8):     # mantissa field
            mags.append(m / 8.0 * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    mags = np.array(mags) / max(mags)
    return np.concatenate([-mags[::-1], mags])


def e4m3_code8() -> np.ndarray:
    """256 non-decreasing fp32 levels: -1 ... -0, +0 ... 1."""
    return e4m3_code8_f64().astype(np.float32)


def dynamic_code8_f64() -> np.ndarray:
    mags = []
    for e in range(7):
        nbins = 2 ** e
        edges = np.linspace(0.1, 1.0, nbins + 1)
        mids = 0.5 * (edges[:-1] + edges[1:])
        mags.append(mids * 10.0 ** (e - 6))
    mags = np.concatenate(mags)  # 127 positive magnitudes
    levels = np.concatenate([-mags, mags, [0.0, 1.0]])
    return np.sort(levels)


def dynamic_code8() -> np.ndarray:
    """256 strictly increasing fp32 levels with an exact 0 and a largest level of 1."""
    return dynamic_code8_f64().astype(np.float32)


def linear_code8() -> np.ndarray:
    """A plain linear 8-bit map, (j - 128) / 128 for j = 0..255 (exact 0 at j = 128,
    -1 at j = 0); used by the tests so that kernel parity does not hinge on one
    choice of code8."""
    j = np.arange(256, dtype=np.float64)
    return ((j - 128.0) / 128.0).astype(np.float32)
