"""Torch-facing wrappers of the C ABI, one per entry point of ``include/nf4.h``.

PyTorch only supplies device memory and the current stream; every step of the
computation runs in the library's CUDA kernels.  Each wrapper checks that the
tensors it passes live on a CUDA device and have the layout the ABI expects, then
forwards raw pointers.  There is no CPU path.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib
from . import codebooks

BLOCKSIZE = 64
NESTED_BLOCKSIZE = 256


def _stream() -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need_cuda(name: str, *ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name}: tensors must be on a CUDA device (no CPU path exists)")


@dataclass
class NF4Weight:
    """A quantised frozen weight W [N, K]: the device tensors of the pages' quant
    state (packed codes, absmax or its 8-bit codes with the nested statistics, the
    codebooks) plus its shape."""
    packed: torch.Tensor
    absmax: Optional[torch.Tensor]
    absmax_q: Optional[torch.Tensor]
    nested_absmax: Optional[torch.Tensor]
    nested_offset: Optional[torch.Tensor]
    code4: torch.Tensor
    code8: Optional[torch.Tensor]
    N: int
    K: int
    double_quant: bool

    @property
    def bits(self) -> int:
        """Code width: 4 (packed nibbles, 16-level code4) or 8 (one code per byte,
        256-level code4)."""
        return 8 if self.code4.numel() == 256 else 4

    def struct(self) -> _lib.nf4_weight:
        return _lib.nf4_weight(
            _ptr(self.packed), _ptr(self.absmax) if not self.double_quant else None,
            _ptr(self.absmax_q) if self.double_quant else None,
            _ptr(self.nested_absmax) if self.double_quant else None,
            _ptr(self.nested_offset) if self.double_quant else None,
            _ptr(self.code4), _ptr(self.code8) if self.double_quant else None,
            self.N, self.K, BLOCKSIZE, NESTED_BLOCKSIZE, 1 if self.double_quant else 0,
            self.bits)

    def tensors(self) -> tuple:
        """The tensors a backward needs, in a fixed order (for save_for_backward)."""
        if self.double_quant:
            return (self.packed, None, self.absmax_q, self.nested_absmax, self.nested_offset,
                    self.code4, self.code8)
        return (self.packed, self.absmax, None, None, None, self.code4, None)

    @staticmethod
    def from_tensors(t: tuple, N: int, K: int, double_quant: bool) -> "NF4Weight":
        packed, absmax, absmax_q, nested_absmax, nested_offset, code4, code8 = t
        return NF4Weight(packed, absmax, absmax_q, nested_absmax, nested_offset, code4, code8,
                         N, K, double_quant)

    def nbytes(self) -> int:
        return sum(x.numel() * x.element_size() for x in self.tensors() if x is not None)


def workspace_size(op: int, M: int, N: int, K: int, E: int = 0) -> int:
    return int(_lib.lib().nf4_workspace_size(op, M, N, K, E))


def quantize(W: torch.Tensor, double_quant: bool = True, code4: Optional[torch.Tensor] = None,
             code8: Optional[torch.Tensor] = None, quant_type: str = "nf4") -> NF4Weight:
    """nf4_quantize / nf4_quantize_8bit: blockwise quantisation (+ double quantisation
    of the absmax) of a CUDA fp32/bf16 [N, K].  `quant_type` picks the storage and the
    default codebook: "nf4", "fp4" (packed 4-bit), "int8", "fp8" (one byte per
    value).  A given `code4` (16 or 256 levels) overrides the codebook."""
    _need_cuda("quantize", W)
    if W.dim() != 2 or not W.is_contiguous():
        raise ValueError("quantize: W must be a contiguous [N, K] tensor")
    if W.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("quantize: W must be fp32 or bf16")
    dev = W.device
    N, K = W.shape
    numel = N * K
    nblocks = (numel + BLOCKSIZE - 1) // BLOCKSIZE
    code4 = (_device_codebook(quant_type, dev, lambda: codebooks.code_for(quant_type)) if code4 is None
             else code4.to(dev, torch.float32).contiguous())
    if code4.numel() not in (16, 256):
        raise ValueError("quantize: the value codebook must have 16 or 256 levels")
    bits = 8 if code4.numel() == 256 else 4
    code8 = (_device_codebook("dynamic8", dev, codebooks.dynamic_code8) if code8 is None
             else code8.to(dev, torch.float32).contiguous())
    packed = torch.empty(numel if bits == 8 else (numel + 1) // 2, dtype=torch.uint8, device=dev)
    absmax = torch.empty(nblocks, dtype=torch.float32, device=dev)
    absmax_q = nested = offset = ws = None
    ws_bytes = 0
    if double_quant:
        absmax_q = torch.empty(nblocks, dtype=torch.uint8, device=dev)
        nested = torch.empty((nblocks + NESTED_BLOCKSIZE - 1) // NESTED_BLOCKSIZE,
                             dtype=torch.float32, device=dev)
        offset = torch.empty(1, dtype=torch.float32, device=dev)
        ws_bytes = workspace_size(_lib.OP_QUANTIZE, 0, N, K)
        ws = torch.empty(max(ws_bytes, 8), dtype=torch.uint8, device=dev)
    fn = _lib.lib().nf4_quantize_8bit if bits == 8 else _lib.lib().nf4_quantize
    rc = fn(
        _ptr(W), _lib.DTYPE_F32 if W.dtype == torch.float32 else _lib.DTYPE_BF16, N, K, BLOCKSIZE,
        1 if double_quant else 0, NESTED_BLOCKSIZE, _ptr(code4), _ptr(code8) if double_quant else None,
        _ptr(packed), _ptr(absmax), _ptr(absmax_q), _ptr(nested), _ptr(offset), _ptr(ws), ws_bytes,
        _stream())
    _lib.check(rc, "nf4_quantize")
    return NF4Weight(packed, absmax, absmax_q, nested, offset, code4,
                     code8 if double_quant else None, N, K, double_quant)


def dequantize(w: NF4Weight, dtype: torch.dtype = torch.bfloat16,
               out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """nf4_dequantize: dense [N, K] copy of the weight (checks and the unfused comparison
    arm; not the fused path).  `out`, when given, is a contiguous [N, K] tensor of `dtype`."""
    _need_cuda("dequantize", w.packed)
    if out is None:
        out = torch.empty(w.N, w.K, dtype=dtype, device=w.packed.device)
    elif out.shape != (w.N, w.K) or out.dtype != dtype or not out.is_contiguous():
        raise ValueError("dequantize: out must be a contiguous [N, K] tensor of the requested dtype")
    code = {torch.float32: _lib.DTYPE_F32, torch.bfloat16: _lib.DTYPE_BF16}[dtype]
    s = w.struct()
    _lib.check(_lib.lib().nf4_dequantize(ctypes.byref(s), _ptr(out), code, _stream()),
               "nf4_dequantize")
    return out


_CODEBOOKS = {}


def _device_codebook(kind: str, dev: torch.device, make) -> torch.Tensor:
    """One read-only device copy of a default codebook per device, shared by every
    weight quantised with it (so that weights can share a multi-product launch,
    which takes one codebook)."""
    key = (kind, str(dev))
    t = _CODEBOOKS.get(key)
    if t is None:
        t = make().to(dev, torch.float32).contiguous()
        _CODEBOOKS[key] = t
    return t


def _check_act(name, a: torch.Tensor, cols: int, f16_ok: bool = False):
    _need_cuda(name, a)
    dts = (torch.bfloat16, torch.float16) if f16_ok else (torch.bfloat16,)
    if a.dtype not in dts or a.dim() != 2 or a.shape[1] != cols or a.stride(1) != 1:
        kinds = "bf16 or fp16" if f16_ok else "bf16"
        raise ValueError(f"{name}: expected a {kinds} [rows, {cols}] tensor with unit column stride")


def linear_fwd(x: torch.Tensor, w: NF4Weight, out: Optional[torch.Tensor] = None,
               ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """nf4_linear_fwd (bf16) / nf4_linear_fwd_f16 (fp16): y = x W^T, x [M, K] -> y [M, N]
    in the activations' dtype."""
    _check_act("linear_fwd", x, w.K, f16_ok=True)
    M = x.shape[0]
    y = torch.empty(M, w.N, dtype=x.dtype, device=x.device) if out is None else out
    need = workspace_size(_lib.OP_LINEAR_FWD, M, w.N, w.K)
    if need and (ws is None or ws.numel() * ws.element_size() < need):
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    if y.dtype != x.dtype:
        raise ValueError("linear_fwd: out must have the activations' dtype")
    s = w.struct()
    fn = _lib.lib().nf4_linear_fwd_f16 if x.dtype == torch.float16 else _lib.lib().nf4_linear_fwd
    rc = fn(_ptr(x), M, x.stride(0), ctypes.byref(s), _ptr(y), y.stride(0),
            _ptr(ws) if need else None, need, _stream())
    _lib.check(rc, "nf4_linear_fwd")
    return y


def linear_dgrad(gy: torch.Tensor, w: NF4Weight, out: Optional[torch.Tensor] = None,
                 ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """nf4_linear_dgrad (bf16) / nf4_linear_dgrad_f16 (fp16): grad_x = grad_y W,
    gy [M, N] -> gx [M, K] in grad_y's dtype."""
    _check_act("linear_dgrad", gy, w.N, f16_ok=True)
    M = gy.shape[0]
    gx = torch.empty(M, w.K, dtype=gy.dtype, device=gy.device) if out is None else out
    need = workspace_size(_lib.OP_LINEAR_DGRAD, M, w.N, w.K)
    if need and (ws is None or ws.numel() * ws.element_size() < need):
        ws = torch.empty(need, dtype=torch.uint8, device=gy.device)
    if gx.dtype != gy.dtype:
        raise ValueError("linear_dgrad: out must have grad_y's dtype")
    s = w.struct()
    fn = _lib.lib().nf4_linear_dgrad_f16 if gy.dtype == torch.float16 else _lib.lib().nf4_linear_dgrad
    rc = fn(_ptr(gy), M, gy.stride(0), ctypes.byref(s), _ptr(gx),
            gx.stride(0), _ptr(ws) if need else None, need, _stream())
    _lib.check(rc, "nf4_linear_dgrad")
    return gx


def _multi(name, fn, acts, ws, outs, out_cols):
    n = len(ws)
    if not 1 <= n <= MAX_MULTI or len(acts) != n:
        raise ValueError(f"{name}: 1..{MAX_MULTI} products, one activation per weight")
    M = acts[0].shape[0]
    if outs is None:
        outs = [torch.empty(M, out_cols(w), dtype=torch.bfloat16, device=acts[0].device) for w in ws]
    if len(outs) != n:
        raise ValueError(f"{name}: one output per weight")
    structs = [w.struct() for w in ws]
    P = ctypes.c_void_p
    a_arr = (P * n)(*[a.data_ptr() for a in acts])
    o_arr = (P * n)(*[o.data_ptr() for o in outs])
    la = (ctypes.c_int64 * n)(*[a.stride(0) for a in acts])
    lo = (ctypes.c_int64 * n)(*[o.stride(0) for o in outs])
    w_arr = (P * n)(*[ctypes.addressof(st) for st in structs])
    rc = fn(n, a_arr, M, la, w_arr, o_arr, lo, _stream())
    _lib.check(rc, name)
    return outs


def route_rows(row_token: torch.Tensor, tokens: int, k: int) -> torch.Tensor:
    """The route table of the top-k combine from the grouped rows' token map
    (row r of the expert-sorted batch belongs to token row_token[r]): int32
    [tokens, k], token t's rows in ascending order.  Every token must hold exactly
    k rows (top-k routing)."""
    if row_token.numel() != tokens * k:
        raise ValueError("route_rows: expected tokens * k grouped rows")
    order = torch.argsort(row_token.to(torch.int64), stable=True)
    return order.to(torch.int32).reshape(tokens, k).contiguous()


def moe_combine(rows: torch.Tensor, token_rows: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """nf4_moe_combine: out[t] = sum over j of rows[token_rows[t, j]] (bf16 [R, H] ->
    [tokens, H]; fp32 sum in route order, rounded once)."""
    _check_act("moe_combine", rows, rows.shape[1] if rows.dim() == 2 else -1)
    _need_cuda("moe_combine", token_rows)
    if token_rows.dtype != torch.int32 or token_rows.dim() != 2 or not token_rows.is_contiguous():
        raise ValueError("moe_combine: token_rows must be a contiguous int32 [tokens, k] tensor")
    tokens, k = token_rows.shape
    R, H = rows.shape
    y = torch.empty(tokens, H, dtype=torch.bfloat16, device=rows.device) if out is None else out
    rc = _lib.lib().nf4_moe_combine(_ptr(rows), R, rows.stride(0), _ptr(token_rows), tokens, k, H, _ptr(y),
                                    y.stride(0), _stream())
    _lib.check(rc, "nf4_moe_combine")
    return y


def moe_combine_bwd(grad_out: torch.Tensor, token_rows: torch.Tensor, R: int,
                    out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """nf4_moe_combine_bwd: each routed row receives its token's gradient (bf16
    [tokens, H] -> [R, H]).  Rows no route names are zero in a new tensor, and left
    as they are in a given `out`."""
    _check_act("moe_combine_bwd", grad_out, grad_out.shape[1] if grad_out.dim() == 2 else -1)
    _need_cuda("moe_combine_bwd", token_rows)
    tokens, k = token_rows.shape
    H = grad_out.shape[1]
    g = torch.zeros(R, H, dtype=torch.bfloat16, device=grad_out.device) if out is None else out
    rc = _lib.lib().nf4_moe_combine_bwd(_ptr(grad_out), tokens, grad_out.stride(0), _ptr(token_rows), k, R, H,
                                        _ptr(g), g.stride(0), _stream())
    _lib.check(rc, "nf4_moe_combine_bwd")
    return g


MAX_MULTI = 4  # NF4_MAX_MULTI of include/nf4.h


def linear_fwd_multi(xs, ws, outs=None):
    """nf4_linear_fwd_multi: y[p] = xs[p] W[p]^T for up to four weights in one launch
    (bf16; the same M and K; xs may repeat one tensor).  Returns the list of y."""
    for x, w in zip(xs, ws):
        _check_act("linear_fwd_multi", x, w.K)
    return _multi("nf4_linear_fwd_multi", _lib.lib().nf4_linear_fwd_multi, xs, ws, outs, lambda w: w.N)


def linear_dgrad_multi(gys, ws, outs=None):
    """nf4_linear_dgrad_multi: gx[p] = gys[p] W[p] for up to four weights in one
    launch (bf16; the same M and K).  Returns the list of gx."""
    for gy, w in zip(gys, ws):
        _check_act("linear_dgrad_multi", gy, w.N)
    return _multi("nf4_linear_dgrad_multi", _lib.lib().nf4_linear_dgrad_multi, gys, ws, outs, lambda w: w.K)


def grouped_fwd(x: torch.Tensor, offsets: torch.Tensor, w: NF4Weight, experts: int,
                out: Optional[torch.Tensor] = None, bias: Optional[torch.Tensor] = None,
                row_scale: Optional[torch.Tensor] = None, swiglu: bool = False) -> torch.Tensor:
    """nf4_grouped_fwd: rows offsets[e]..offsets[e+1] of x through expert e.
    w is the stacked [E*N_e, K] weight; returns bf16 [T, N_e].
    With an epilogue (nf4_grouped_fwd_ep): `bias` fp32 [E*N_e] per weight row,
    `row_scale` fp32 [T] per output row (routing weights), `swiglu` for a weight whose
    expert rows interleave gate and up in groups of 64 (see `interleave_gate_up`):
    then y = silu(gate) * up, [T, N_e / 2]."""
    _check_act("grouped_fwd", x, w.K)
    _need_cuda("grouped_fwd", offsets, bias, row_scale)
    if offsets.dtype != torch.int32 or offsets.numel() != experts + 1:
        raise ValueError("grouped_fwd: offsets must be int32 [E+1]")
    N_e = w.N // experts
    T = x.shape[0]
    width = N_e // 2 if swiglu else N_e
    y = torch.empty(T, width, dtype=torch.bfloat16, device=x.device) if out is None else out
    s = w.struct()
    if bias is None and row_scale is None and not swiglu:
        rc = _lib.lib().nf4_grouped_fwd(_ptr(x), _ptr(offsets), experts, T, x.stride(0),
                                        ctypes.byref(s), N_e, _ptr(y), y.stride(0), _stream())
    else:
        for name, t, n in (("bias", bias, w.N), ("row_scale", row_scale, T)):
            if t is not None and (t.dtype != torch.float32 or t.numel() != n or not t.is_contiguous()):
                raise ValueError(f"grouped_fwd: {name} must be a contiguous fp32 tensor of {n} values")
        ep = _lib.nf4_epilogue(_ptr(bias), _ptr(row_scale), 1 if swiglu else 0)
        rc = _lib.lib().nf4_grouped_fwd_ep(_ptr(x), _ptr(offsets), experts, T, x.stride(0),
                                           ctypes.byref(s), N_e, ctypes.byref(ep), _ptr(y),
                                           y.stride(0), _stream())
    _lib.check(rc, "nf4_grouped_fwd")
    return y


def grouped_swiglu_bwd(x: torch.Tensor, offsets: torch.Tensor, w: NF4Weight, experts: int,
                       gh: torch.Tensor, bias: Optional[torch.Tensor] = None,
                       row_scale: Optional[torch.Tensor] = None, need_row_scale_grad: bool = False,
                       ws: Optional[torch.Tensor] = None):
    """nf4_grouped_swiglu_bwd: the backward of grouped_fwd(..., swiglu=True) over an
    interleaved gate/up weight.  x bf16 [T, K] (the forward input), gh bf16
    [T, N_e / 2].  Returns (grad_x bf16 [T, K], grad_row_scale fp32 [T] or None);
    the second needs `row_scale` and `need_row_scale_grad`."""
    _check_act("grouped_swiglu_bwd", x, w.K)
    N_e = w.N // experts
    _check_act("grouped_swiglu_bwd", gh, N_e // 2)
    _need_cuda("grouped_swiglu_bwd", offsets, bias, row_scale)
    if offsets.dtype != torch.int32 or offsets.numel() != experts + 1:
        raise ValueError("grouped_swiglu_bwd: offsets must be int32 [E+1]")
    T = x.shape[0]
    for name, t, n in (("bias", bias, w.N), ("row_scale", row_scale, T)):
        if t is not None and (t.dtype != torch.float32 or t.numel() != n or not t.is_contiguous()):
            raise ValueError(f"grouped_swiglu_bwd: {name} must be a contiguous fp32 tensor of {n} values")
    gx = torch.empty(T, w.K, dtype=torch.bfloat16, device=x.device)
    drw = (torch.empty(T, dtype=torch.float32, device=x.device)
           if need_row_scale_grad and row_scale is not None else None)
    need = workspace_size(_lib.OP_GROUPED_SWIGLU_BWD, T, N_e, w.K, experts)
    if ws is None or ws.numel() * ws.element_size() < need:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    ep = _lib.nf4_epilogue(_ptr(bias), _ptr(row_scale), 1)
    s = w.struct()
    rc = _lib.lib().nf4_grouped_swiglu_bwd(_ptr(x), _ptr(offsets), experts, T, x.stride(0),
                                           ctypes.byref(s), N_e, ctypes.byref(ep), _ptr(gh),
                                           gh.stride(0), _ptr(gx), gx.stride(0), _ptr(drw), _ptr(ws),
                                           need, _stream())
    _lib.check(rc, "nf4_grouped_swiglu_bwd")
    return gx, drw


def interleave_gate_up(gate: torch.Tensor, up: torch.Tensor, experts: int) -> torch.Tensor:
    """Stack per-expert gate and up weights ([E*H, K] each, H a multiple of 64) into
    the [E*2H, K] layout of the fused SwiGLU epilogue: each 128-row group holds 64
    gate rows, then the up rows of the same 64 output columns.  Done on the dense
    weight before quantisation."""
    EH, K = gate.shape
    H = EH // experts
    if up.shape != gate.shape or EH != experts * H or H % 64 != 0:
        raise ValueError("interleave_gate_up: gate and up must be [E*H, K] with H % 64 == 0")
    g = gate.reshape(experts, H // 64, 1, 64, K)
    u = up.reshape(experts, H // 64, 1, 64, K)
    return torch.cat([g, u], dim=2).reshape(experts * 2 * H, K).contiguous()


def grouped_dgrad(gy: torch.Tensor, offsets: torch.Tensor, w: NF4Weight, experts: int,
                  out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """nf4_grouped_dgrad: per-expert grad_x; gy bf16 [T, N_e] -> gx bf16 [T, K]."""
    N_e = w.N // experts
    _check_act("grouped_dgrad", gy, N_e)
    _need_cuda("grouped_dgrad", offsets)
    if offsets.dtype != torch.int32 or offsets.numel() != experts + 1:
        raise ValueError("grouped_dgrad: offsets must be int32 [E+1]")
    T = gy.shape[0]
    gx = torch.empty(T, w.K, dtype=torch.bfloat16, device=gy.device) if out is None else out
    s = w.struct()
    rc = _lib.lib().nf4_grouped_dgrad(_ptr(gy), _ptr(offsets), experts, T, gy.stride(0),
                                      ctypes.byref(s), N_e, _ptr(gx), gx.stride(0), _stream())
    _lib.check(rc, "nf4_grouped_dgrad")
    return gx


path_counters = _lib.path_counters
reset_path_counters = _lib.reset_path_counters
device_status = _lib.device_status
device_check = _lib.device_check
set_weight_prefetch = _lib.set_weight_prefetch
set_small_m_path = _lib.set_small_m_path
set_stream_k = _lib.set_stream_k
set_cluster_split = _lib.set_cluster_split
set_token_tile = _lib.set_token_tile
inject_stream_k_timeout = _lib.inject_stream_k_timeout
plan_query = _lib.plan_query
