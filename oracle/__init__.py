"""CPU oracle for the fused NF4 dequantise-and-multiply.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The GPU library never imports, links or calls it, and it never imports
the GPU library.

The arithmetic lives in plain C (``nf4_oracle.c``, fp64 sums, no fast-math, no
FMA contraction); this module only builds it, loads it with ctypes and moves
numpy arrays in and out.  Codebooks come from ``oracle.codebooks``.

Every function is pinned by the ``-m "not gpu"`` tests against values that the
definition fixes (codebook end points and zero, quantise/dequantise round trips of
codebook-aligned blocks, the absmax scaling invariant, hand-built packed bytes,
brute force and closed forms of the products).  Parity of the codebook values
and of the nibble order with bitsandbytes itself is unpinned: bitsandbytes is not
available and the pages print neither.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nf4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

MEAN_CHUNK = 1024  # chunk length of the fixed summation order of the mean offset


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            i32 = ctypes.c_int32
            L.oracle_quantize_nf4.argtypes = [P, i64, i32, P, P, P]
            L.oracle_double_quant.argtypes = [P, i64, i32, i32, P, P, P, P]
            L.oracle_decode_absmax.argtypes = [P, P, ctypes.c_float, i64, i32, P, P]
            L.oracle_dequantize_nf4.argtypes = [P, P, i64, i32, P, P, P]
            L.oracle_quantize_8bit.argtypes = [P, i64, i32, P, P, P]
            L.oracle_dequantize_8bit.argtypes = [P, P, i64, i32, P, P, P]
            L.oracle_linear_fwd.argtypes = [P, i64, i64, P, i64, P, i64, P]
            L.oracle_linear_dgrad.argtypes = [P, i64, i64, P, i64, P, i64, P]
            L.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
            L.oracle_bf16_from_f32.restype = ctypes.c_uint16
            L.oracle_f16_from_f32.argtypes = [ctypes.c_float]
            L.oracle_f16_from_f32.restype = ctypes.c_uint16
            L.oracle_f32_from_f16.argtypes = [ctypes.c_uint16]
            L.oracle_f32_from_f16.restype = ctypes.c_float
            L.oracle_f16_array.argtypes = [P, i64, P]
            L.oracle_bf16_array.argtypes = [P, i64, P]
            L.oracle_linear_fwd_f16.argtypes = [P, i64, i64, P, i64, P, i64, P]
            L.oracle_linear_dgrad_f16.argtypes = [P, i64, i64, P, i64, P, i64, P]
            L.oracle_num_threads.restype = ctypes.c_int
            for name in ("oracle_quantize_nf4", "oracle_double_quant", "oracle_decode_absmax",
                         "oracle_dequantize_nf4", "oracle_linear_fwd", "oracle_linear_dgrad",
                         "oracle_quantize_8bit", "oracle_dequantize_8bit", "oracle_f16_array",
                         "oracle_bf16_array",
                         "oracle_linear_fwd_f16", "oracle_linear_dgrad_f16"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def num_threads() -> int:
    return int(lib().oracle_num_threads())


# ------------------------------------------------------------------ bf16 ----

def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact widening)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns by round-to-nearest-even (the C oracle's rule)."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.zeros(f.shape, dtype=np.uint16)
    _check(lib().oracle_bf16_array(_p(f), f.size, _p(out)), "bf16_array")
    return out


# --------------------------------------------------------- quantisation ----

class QuantState:
    """Plain container of one quantised weight: the oracle's view of the pages'
    QuantState (packed bytes, fp32 absmax, and under double quantisation the 8-bit
    codes, nested absmax and offset)."""

    def __init__(self, shape, blocksize, packed, absmax, code4, double_quant=False,
                 absmax_q=None, nested_absmax=None, nested_offset=None, code8=None,
                 nested_blocksize=256, bits=4):
        self.bits = bits  # 4: two codes per byte, 16-level code4; 8: one code per byte, 256 levels
        self.shape = tuple(shape)
        self.blocksize = blocksize
        self.packed = packed
        self.absmax = absmax
        self.code4 = code4
        self.double_quant = double_quant
        self.absmax_q = absmax_q
        self.nested_absmax = nested_absmax
        self.nested_offset = nested_offset
        self.code8 = code8
        self.nested_blocksize = nested_blocksize

    @property
    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n


def quantize_nf4(w: np.ndarray, code4: np.ndarray, blocksize: int = 64):
    """Blockwise NF4 quantisation of a flat view of w (fp32).  Returns (packed, absmax)."""
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    code4 = np.ascontiguousarray(code4, dtype=np.float32)
    numel = w.size
    packed = np.zeros((numel + 1) // 2, dtype=np.uint8)
    absmax = np.zeros((numel + blocksize - 1) // blocksize, dtype=np.float32)
    _check(lib().oracle_quantize_nf4(_p(w), numel, blocksize, _p(code4), _p(packed), _p(absmax)),
           "quantize_nf4")
    return packed, absmax


def quantize_8bit(w: np.ndarray, code: np.ndarray, blocksize: int = 64):
    """Blockwise 8-bit quantisation of a flat view of w (fp32) with a 256-level
    codebook.  Returns (codes uint8 [numel], absmax)."""
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    code = np.ascontiguousarray(code, dtype=np.float32)
    assert code.size == 256
    numel = w.size
    q = np.zeros(numel, dtype=np.uint8)
    absmax = np.zeros((numel + blocksize - 1) // blocksize, dtype=np.float32)
    _check(lib().oracle_quantize_8bit(_p(w), numel, blocksize, _p(code), _p(q), _p(absmax)),
           "quantize_8bit")
    return q, absmax


def double_quant(absmax: np.ndarray, code8: np.ndarray, nested_blocksize: int = 256):
    """8-bit blockwise quantisation of the absmax array.  Returns (absmax_q, nested_absmax, offset)."""
    absmax = np.ascontiguousarray(absmax, dtype=np.float32).reshape(-1)
    code8 = np.ascontiguousarray(code8, dtype=np.float32)
    nb = absmax.size
    absmax_q = np.zeros(nb, dtype=np.uint8)
    nested = np.zeros((nb + nested_blocksize - 1) // nested_blocksize, dtype=np.float32)
    off = np.zeros(1, dtype=np.float32)
    _check(lib().oracle_double_quant(_p(absmax), nb, nested_blocksize, MEAN_CHUNK, _p(code8),
                                     _p(absmax_q), _p(nested), _p(off)), "double_quant")
    return absmax_q, nested, off


def decode_absmax(absmax_q, nested_absmax, offset, code8, nested_blocksize: int = 256):
    absmax_q = np.ascontiguousarray(absmax_q, dtype=np.uint8).reshape(-1)
    nested_absmax = np.ascontiguousarray(nested_absmax, dtype=np.float32)
    code8 = np.ascontiguousarray(code8, dtype=np.float32)
    out = np.zeros(absmax_q.size, dtype=np.float32)
    off = float(np.asarray(offset, dtype=np.float32).reshape(-1)[0])
    _check(lib().oracle_decode_absmax(_p(absmax_q), _p(nested_absmax), ctypes.c_float(off),
                                      absmax_q.size, nested_blocksize, _p(code8), _p(out)),
           "decode_absmax")
    return out


def quantize(w: np.ndarray, code4, blocksize: int = 64, double_quant_: bool = False,
             code8=None, nested_blocksize: int = 256) -> QuantState:
    """Blockwise quantisation with the value codebook `code4`: 16 levels give the
    packed 4-bit format, 256 levels the 8-bit format (one code per byte)."""
    code4 = np.asarray(code4, np.float32)
    if code4.size == 256:
        packed, absmax = quantize_8bit(w, code4, blocksize)
        st = QuantState(np.shape(w), blocksize, packed, absmax, code4, bits=8)
    else:
        packed, absmax = quantize_nf4(w, code4, blocksize)
        st = QuantState(np.shape(w), blocksize, packed, absmax, code4)
    if double_quant_:
        aq, nested, off = double_quant(absmax, code8, nested_blocksize)
        st.double_quant = True
        st.absmax_q, st.nested_absmax, st.nested_offset = aq, nested, off
        st.code8 = np.asarray(code8, np.float32)
        st.nested_blocksize = nested_blocksize
    return st


def block_scale(st: QuantState) -> np.ndarray:
    """The per-block fp32 scale the dequantisation multiplies by (absmax, or the
    decoded absmax under double quantisation)."""
    if st.double_quant:
        return decode_absmax(st.absmax_q, st.nested_absmax, st.nested_offset, st.code8,
                             st.nested_blocksize)
    return st.absmax


def dequantize(st: QuantState, dtype: str = "bf16") -> np.ndarray:
    """Dense dequantised weight: fp32 values, or bf16 bit patterns (uint16)."""
    scale = np.ascontiguousarray(block_scale(st), dtype=np.float32)
    n = st.numel
    fn = lib().oracle_dequantize_8bit if st.bits == 8 else lib().oracle_dequantize_nf4
    if dtype == "f32":
        out = np.zeros(n, dtype=np.float32)
        _check(fn(_p(st.packed), _p(scale), n, st.blocksize, _p(st.code4), _p(out), None),
               "dequantize")
    elif dtype == "bf16":
        out = np.zeros(n, dtype=np.uint16)
        _check(fn(_p(st.packed), _p(scale), n, st.blocksize, _p(st.code4), None, _p(out)),
               "dequantize")
    else:
        raise ValueError(dtype)
    return out.reshape(st.shape)


# ------------------------------------------------------------- products ----

def f16_bits(f: np.ndarray) -> np.ndarray:
    """fp32 values -> IEEE binary16 bit patterns (round to nearest, ties to even)."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.zeros(f.shape, dtype=np.uint16)
    _check(lib().oracle_f16_array(_p(f), f.size, _p(out)), "f16_array")
    return out


def dequantize_f16(st: QuantState) -> np.ndarray:
    """Dense dequantised weight rounded to fp16 (bit patterns): the operand of the
    fp16 compute dtype."""
    return f16_bits(dequantize(st, "f32"))


def linear_fwd(x_bf16: np.ndarray, wb_bf16: np.ndarray, rows=None, dtype: str = "bf16") -> np.ndarray:
    """y = x W^T in fp64 from 16-bit patterns x [M,K] and Wb [N,K] (bf16, or fp16 with
    dtype="f16"); only `rows` of y when given."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    wb = np.ascontiguousarray(wb_bf16, dtype=np.uint16)
    M, K = x.shape
    N, K2 = wb.shape
    assert K == K2
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = M if r is None else r.size
    y = np.zeros((nrows, N), dtype=np.float64)
    fn = lib().oracle_linear_fwd_f16 if dtype == "f16" else lib().oracle_linear_fwd
    _check(fn(_p(x), M, K, _p(wb), N, _p(r), nrows, _p(y)), "linear_fwd")
    return y


def linear_dgrad(gy_bf16: np.ndarray, wb_bf16: np.ndarray, rows=None, dtype: str = "bf16") -> np.ndarray:
    """grad_x = grad_y W in fp64 from 16-bit patterns gy [M,N] and Wb [N,K] (bf16, or
    fp16 with dtype="f16")."""
    gy = np.ascontiguousarray(gy_bf16, dtype=np.uint16)
    wb = np.ascontiguousarray(wb_bf16, dtype=np.uint16)
    M, N = gy.shape
    N2, K = wb.shape
    assert N == N2
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = M if r is None else r.size
    gx = np.zeros((nrows, K), dtype=np.float64)
    fn = lib().oracle_linear_dgrad_f16 if dtype == "f16" else lib().oracle_linear_dgrad
    _check(fn(_p(gy), M, N, _p(wb), K, _p(r), nrows, _p(gx)), "linear_dgrad")
    return gx


def grouped_fwd(x_bf16: np.ndarray, offsets, wb_stack_bf16: np.ndarray) -> np.ndarray:
    """Per-expert forward: rows offsets[e]..offsets[e+1] of x use expert e's weight
    wb_stack[e] ([E,N,K] bf16 bits).  Returns fp64 [T,N]."""
    E, N, K = wb_stack_bf16.shape
    T = x_bf16.shape[0]
    y = np.zeros((T, N), dtype=np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y[a:b] = linear_fwd(x_bf16[a:b], wb_stack_bf16[e])
    return y


def interleave_gate_up(gate: np.ndarray, up: np.ndarray, experts: int) -> np.ndarray:
    """Stack the gate and up projections of each expert ([E*H, K] each, H a multiple
    of 64) into one [E*2H, K] weight whose 128-row groups hold 64 gate rows then the
    64 up rows of the same output columns (the layout the fused SwiGLU epilogue reads)."""
    EH, K = gate.shape
    H = EH // experts
    g = gate.reshape(experts, H // 64, 64, K)
    u = up.reshape(experts, H // 64, 64, K)
    return np.stack([g, u], axis=2).reshape(experts * 2 * H, K)


def grouped_fwd_epilogue(x_bf16: np.ndarray, offsets, wb_stack_bf16: np.ndarray, bias=None,
                         row_scale=None, swiglu: bool = False) -> np.ndarray:
    """The grouped forward followed by the expert epilogue, in fp64 (Soup issue #842's
    expert path / fork PR "Experts trainability": the SwiGLU of gate and up, the
    routing-weight scaling and a bias that otherwise run in torch around the products):
      a = x_e W_e^T (+ bias[e, :], fp32 per weight row);
      swiglu: each 128-column group of a is (gate[64], up[64]) of 64 output columns,
              h = silu(gate) * up with silu(g) = g / (1 + exp(-g));
      row_scale: every output row times row_scale[t] (routing weights, sorted order)."""
    E, N, K = wb_stack_bf16.shape
    a = grouped_fwd(x_bf16, offsets, wb_stack_bf16)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float32).astype(np.float64).reshape(E, N)
        for e in range(E):
            a[int(offsets[e]):int(offsets[e + 1])] += b[e]
    if swiglu:
        return swiglu_forward(a, row_scale)
    if row_scale is not None:
        a = a * np.asarray(row_scale, dtype=np.float32).astype(np.float64)[:, None]
    return a


def _gate_up(a: np.ndarray):
    """Views of the gate and up columns of an interleaved [T, N] array (each 128-column
    group holds 64 gate columns, then the 64 up columns of the same outputs)."""
    T, N = a.shape
    grp = a.reshape(T, N // 128, 2, 64)
    return grp[:, :, 0, :], grp[:, :, 1, :]


def swiglu_forward(a: np.ndarray, row_scale=None) -> np.ndarray:
    """h = silu(g) * u (* row_scale[t]) in fp64 from interleaved pre-activations a
    [T, N]; silu(g) = g / (1 + exp(-g)).  Returns [T, N / 2]."""
    g, u = _gate_up(np.asarray(a, dtype=np.float64))
    h = (g / (1.0 + np.exp(-g)) * u).reshape(a.shape[0], a.shape[1] // 2)
    if row_scale is not None:
        h = h * np.asarray(row_scale, dtype=np.float32).astype(np.float64)[:, None]
    return h


def swiglu_backward(a: np.ndarray, dh: np.ndarray, row_scale=None):
    """Gradients of h = silu(g) * u * r (r = row_scale[t], or 1) in fp64, the chain
    rule of the fused expert SwiGLU written out (fork PR "Experts trainability",
    commit 2: the backward recomputes the expert products and needs no saved dense
    weight):
      s = 1 / (1 + exp(-g)),  silu(g) = g s,  silu'(g) = s (1 + g (1 - s));
      dg = dh r u silu'(g);   du = dh r silu(g);
      dr = sum over the row's outputs of silu(g) u dh.
    a: interleaved pre-activations [T, N] (bias included); dh: [T, N / 2].
    Returns (dgu [T, N] in the same interleaved layout, dr [T] or None)."""
    a = np.asarray(a, dtype=np.float64)
    T, N = a.shape
    g, u = _gate_up(a)
    d = np.asarray(dh, dtype=np.float64).reshape(T, N // 128, 64)
    r = None if row_scale is None else np.asarray(row_scale, dtype=np.float32).astype(np.float64)
    s = 1.0 / (1.0 + np.exp(-g))
    silu = g * s
    dr = None if r is None else (silu * u * d).reshape(T, -1).sum(axis=1)
    dd = d if r is None else d * r[:, None, None]
    dgu = np.empty((T, N // 128, 2, 64), dtype=np.float64)
    dgu[:, :, 0, :] = dd * u * (s * (1.0 + g * (1.0 - s)))
    dgu[:, :, 1, :] = dd * silu
    return dgu.reshape(T, N), dr


def grouped_swiglu_dgrad(x_bf16: np.ndarray, offsets, wb_stack_bf16: np.ndarray,
                         dh_bf16: np.ndarray, bias=None, row_scale=None):
    """Input gradient (and routing-weight gradient) of the fused expert SwiGLU over an
    interleaved gate/up weight, in the order the backward takes its steps:
      1. a = x_e W_e^T (+ bias), the exact fp64 product (grouped_fwd);
      2. (dgu, dr) = swiglu_backward(a, dh, row_scale);
      3. the gate/up gradient becomes an activation-dtype tensor: bf16(fp32(dgu)),
         round to nearest even (the operand of the frozen input-gradient product,
         as the activations are for the forward);
      4. gx = grouped_dgrad(that operand) in fp64.
    dh_bf16: bf16 bit patterns [T, N / 2].  Returns (gx fp64 [T, K], dr fp64 [T] or None)."""
    E, N, K = wb_stack_bf16.shape
    a = grouped_fwd(x_bf16, offsets, wb_stack_bf16)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float32).astype(np.float64).reshape(E, N)
        for e in range(E):
            a[int(offsets[e]):int(offsets[e + 1])] += b[e]
    dh = bf16_bits_to_f32(dh_bf16).astype(np.float64)
    dgu, dr = swiglu_backward(a, dh, row_scale)
    op = f32_to_bf16_bits(dgu.astype(np.float32))
    return grouped_dgrad(op, offsets, wb_stack_bf16), dr


def grouped_dgrad(gy_bf16: np.ndarray, offsets, wb_stack_bf16: np.ndarray) -> np.ndarray:
    E, N, K = wb_stack_bf16.shape
    T = gy_bf16.shape[0]
    gx = np.zeros((T, K), dtype=np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            gx[a:b] = linear_dgrad(gy_bf16[a:b], wb_stack_bf16[e])
    return gx


def moe_combine(rows_bf16: np.ndarray, token_rows: np.ndarray) -> np.ndarray:
    """Top-k combine of the grouped experts' output rows (fork PR "Experts
    trainability", commits 1-2: per-expert segments of a token-sorted batch; Soup
    issue #842, expert path): token t's output is the sum of the rows it was routed
    to, token_rows[t, j] (j = 0 .. k-1; -1 for an absent route).  rows_bf16: bf16
    bit patterns [R, H].  Returns the exact fp64 sums [tokens, H]."""
    rows = bf16_bits_to_f32(np.ascontiguousarray(rows_bf16, dtype=np.uint16)).astype(np.float64)
    tokens, k = token_rows.shape
    out = np.zeros((tokens, rows.shape[1]), dtype=np.float64)
    for t in range(tokens):
        for j in range(k):
            r = int(token_rows[t, j])
            if r >= 0:
                out[t] += rows[r]
    return out


def moe_combine_bwd(grad_bf16: np.ndarray, token_rows: np.ndarray, R: int) -> np.ndarray:
    """Backward of moe_combine: each row routed from token t receives grad[t]
    unchanged (bf16 bit patterns [R, H]; rows no route names stay 0)."""
    g = np.ascontiguousarray(grad_bf16, dtype=np.uint16)
    out = np.zeros((R, g.shape[1]), dtype=np.uint16)
    tokens, k = token_rows.shape
    for t in range(tokens):
        for j in range(k):
            r = int(token_rows[t, j])
            if r >= 0:
                out[r] = g[t]
    return out
