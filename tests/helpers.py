"""Shared helpers of the GPU parity tests: inputs come from the synthetic-input
module, expected values from the CPU oracle only."""
import numpy as np
import torch

import oracle
from oracle import codebooks as ocb

REL_FRO = 5e-3      # relative Frobenius error bound of the fused products
ELEM = 1e-2         # per-element bound: |err| <= ELEM * (|ref| + rms(ref))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_state(w32: torch.Tensor, dq: bool, code8=None):
    return oracle.quantize(w32.numpy(), ocb.nf4_code4(), 64, dq,
                           ocb.dynamic_code8() if code8 is None else code8, 256)


def parity(got: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), what
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(g - ref) / max(nref, 1e-300)
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e}"
    rms = np.sqrt(np.mean(ref ** 2))
    bad = np.abs(g - ref) > ELEM * (np.abs(ref) + rms)
    assert not bad.any(), f"{what}: {bad.sum()} elements out of bound, first at {np.argwhere(bad)[0]}"
    return rel
