"""Guard bands around the outputs of every product path.

Each output is a view into the middle of a larger buffer: rows before and after
it, and columns on both sides (the view's row pitch is wider than the output),
all filled with a sentinel bit pattern.  After the call the sentinel must be
untouched (no write past M, past the output width, or before the first element)
and the view itself must match the oracle.  The cases cover the token-tile
widths, ragged row and column tails, the split contraction with its reduction
kernel, stream-K, the small-M kernels, the one-byte codes, the fp16 dtype and the
grouped products with and without their epilogue.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import codebooks as ocb
import bit_nf4_quantized_linear_gb300 as nf4
from bit_nf4_quantized_linear_gb300 import _lib, ops, synth
from tests.helpers import bf16_bits, oracle_state, parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SENTINEL = 0x7FA5  # a NaN pattern no product writes
PAD_ROWS, PAD_COLS = 3, 8


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    nf4.device_status(clear=True)
    yield
    ops.set_stream_k(_lib.STREAM_K_AUTO)
    ops.set_small_m_path(_lib.SMALL_M_AUTO)
    assert nf4.device_status() == 0


def guarded(rows, cols, dtype=torch.bfloat16):
    """(buffer, view): the view [rows, cols] sits PAD_ROWS rows down and PAD_COLS
    columns in, inside a sentinel-filled buffer with row pitch cols + 2 PAD_COLS."""
    buf = torch.full((rows + 2 * PAD_ROWS, cols + 2 * PAD_COLS), 0, dtype=torch.int16, device=DEV)
    buf.fill_(SENTINEL)
    buf = buf.view(dtype)
    return buf, buf[PAD_ROWS:PAD_ROWS + rows, PAD_COLS:PAD_COLS + cols]


def check_guard(buf, rows, cols, what):
    bits = buf.view(torch.int16).cpu().numpy().view(np.uint16)
    inside = np.zeros(bits.shape, dtype=bool)
    inside[PAD_ROWS:PAD_ROWS + rows, PAD_COLS:PAD_COLS + cols] = True
    bad = (bits != SENTINEL) & ~inside
    assert not bad.any(), f"{what}: {bad.sum()} guard elements overwritten, first at {np.argwhere(bad)[0]}"


DENSE = [  # (M, N, K, stream_k, small_m): token tiles 16..256, ragged tails, every kernel
    (1, 200, 256, "auto", "auto"), (7, 384, 1024, "auto", "auto"), (12, 256, 512, "auto", "simt"),
    (9, 640, 1536, "off", "tiles"), (40, 328, 192, "auto", "auto"), (129, 392, 320, "force", "auto"),
    (300, 136, 2048, "off", "auto"), (700, 648, 1024, "force", "auto"), (1100, 1024, 512, "off", "auto"),
]
SK = {"off": _lib.STREAM_K_OFF, "auto": _lib.STREAM_K_AUTO, "force": _lib.STREAM_K_FORCE}
SM = {"auto": _lib.SMALL_M_AUTO, "simt": _lib.SMALL_M_SIMT, "tiles": _lib.SMALL_M_TILES}


@pytest.mark.parametrize("M,N,K,sk,small", DENSE)
def test_dense_products_stay_inside_their_output(M, N, K, sk, small):
    g = synth.generator(M + 3 * N + K)
    w32 = synth.weight(N, K, g)
    w = nf4.quantize(w32.to(DEV), double_quant=True)
    wb = oracle.dequantize(oracle_state(w32, True), "bf16")
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    try:
        ops.set_stream_k(SK[sk])
        ops.set_small_m_path(SM[small])
        ybuf, y = guarded(M, N)
        ops.linear_fwd(x.to(DEV), w, out=y)
        gbuf, gx = guarded(M, K)
        ops.linear_dgrad(gy.to(DEV), w, out=gx)
        torch.cuda.synchronize()
    finally:
        ops.set_stream_k(_lib.STREAM_K_AUTO)
        ops.set_small_m_path(_lib.SMALL_M_AUTO)
    check_guard(ybuf, M, N, f"fwd {M}x{N}x{K}")
    check_guard(gbuf, M, K, f"dgrad {M}x{N}x{K}")
    parity(y, oracle.linear_fwd(bf16_bits(x), wb), f"guarded fwd {M}x{N}x{K}")
    parity(gx, oracle.linear_dgrad(bf16_bits(gy), wb), f"guarded dgrad {M}x{N}x{K}")


@pytest.mark.parametrize("bt,M,N,K", [(64, 1100, 648, 1024), (128, 700, 136, 8192),
                                      (512, 1100, 648, 1024), (512, 700, 136, 8192)])
def test_fixed_token_tiles_stay_inside_their_output(bt, M, N, K):
    g = synth.generator(M + N)
    w32 = synth.weight(N, K, g)
    w = nf4.quantize(w32.to(DEV), double_quant=True)
    wb = oracle.dequantize(oracle_state(w32, True), "bf16")
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    try:
        ops.set_token_tile(bt)
        ybuf, y = guarded(M, N)
        ops.linear_fwd(x.to(DEV), w, out=y)
        gbuf, gx = guarded(M, K)
        ops.linear_dgrad(gy.to(DEV), w, out=gx)
        torch.cuda.synchronize()
    finally:
        ops.set_token_tile(0)
    check_guard(ybuf, M, N, f"tile {bt} fwd {M}x{N}x{K}")
    check_guard(gbuf, M, K, f"tile {bt} dgrad {M}x{N}x{K}")
    parity(y, oracle.linear_fwd(bf16_bits(x), wb), f"guarded tile {bt} fwd {M}x{N}x{K}")
    parity(gx, oracle.linear_dgrad(bf16_bits(gy), wb), f"guarded tile {bt} dgrad {M}x{N}x{K}")


@pytest.mark.parametrize("M", [3, 200])
def test_one_byte_codes_and_fp16_stay_inside_their_output(M):
    N, K = 264, 320
    g = synth.generator(90 + M)
    w32 = synth.weight(N, K, g)
    x = synth.activation(M, K, g)
    w8 = nf4.quantize(w32.to(DEV), double_quant=True, quant_type="int8")
    st8 = oracle.quantize(w32.numpy(), ocb.dynamic_code8(), 64, True, ocb.dynamic_code8(), 256)
    buf, y = guarded(M, N)
    ops.linear_fwd(x.to(DEV), w8, out=y)
    torch.cuda.synchronize()
    check_guard(buf, M, N, "int8 fwd")
    parity(y, oracle.linear_fwd(bf16_bits(x), oracle.dequantize(st8, "bf16")), "guarded int8 fwd")
    w4 = nf4.quantize(w32.to(DEV), double_quant=True)
    st4 = oracle_state(w32, True)
    xh = x.float().half()
    buf, yh = guarded(M, N, torch.float16)
    ops.linear_fwd(xh.to(DEV), w4, out=yh)
    torch.cuda.synchronize()
    check_guard(buf, M, N, "f16 fwd")
    xbits = xh.contiguous().view(torch.int16).numpy().view(np.uint16)
    parity(yh, oracle.linear_fwd(xbits, oracle.dequantize_f16(st4), dtype="f16"), "guarded f16 fwd")


@pytest.mark.parametrize("swiglu", [False, True])
def test_grouped_products_stay_inside_their_output(swiglu):
    E, N_e, K = 3, 256, 192
    counts = [17, 0, 70]
    g = synth.generator(95 + swiglu)
    if swiglu:
        w32 = nf4.interleave_gate_up(synth.weight(E * N_e // 2, K, g), synth.weight(E * N_e // 2, K, g), E)
    else:
        w32 = synth.weight(E * N_e, K, g)
    w = nf4.quantize(w32.to(DEV), double_quant=True)
    st = oracle_state(w32, True)
    wb = oracle.dequantize(st, "bf16").reshape(E, N_e, K)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offs[-1])
    x = synth.activation(T, K, g)
    gy = synth.activation(T, N_e, g)
    offs_d = torch.from_numpy(offs).to(DEV)
    width = N_e // 2 if swiglu else N_e
    buf, y = guarded(T, width)
    ops.grouped_fwd(x.to(DEV), offs_d, w, E, out=y, swiglu=swiglu)
    torch.cuda.synchronize()
    check_guard(buf, T, width, f"grouped fwd swiglu={swiglu}")
    parity(y, oracle.grouped_fwd_epilogue(bf16_bits(x), offs, wb, swiglu=swiglu), "guarded grouped fwd")
    if not swiglu:
        gbuf, gx = guarded(T, K)
        ops.grouped_dgrad(gy.to(DEV), offs_d, w, E, out=gx)
        torch.cuda.synchronize()
        check_guard(gbuf, T, K, "grouped dgrad")
        parity(gx, oracle.grouped_dgrad(bf16_bits(gy), offs, wb), "guarded grouped dgrad")
