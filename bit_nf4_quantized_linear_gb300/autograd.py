"""Autograd Functions over the fused kernels.

The backward of a frozen 4-bit Linear needs the packed weight and its statistics.
bitsandbytes' MatMul4Bit keeps them as plain ctx attributes, which activation
checkpointing cannot see, so a caller that re-materialises the weight into a
recycled buffer gets silently wrong gradients (bitsandbytes issue "MatMul4Bit
keeps B and quant_state on ctx ...", sections "Summary" and "Root cause").  Here
every tensor the backward reads -- the packed codes, the absmax or its 8-bit codes,
the nested absmax and offset, and both codebooks -- goes through
``ctx.save_for_backward`` (same issue, "Why save_for_backward fixes it"; Soup issue
#842, "Design sketch"); ctx holds Python ints only.  The backward computes only
grad_x (the base is frozen, Soup issue #842 "Scope") with the fused transposed
kernel; no dense weight is saved or materialised (fork PR "Experts trainability",
commit 2).
"""
from __future__ import annotations

import torch

from . import ops


class NF4LinearFn(torch.autograd.Function):
    """y = x W^T for a frozen NF4 weight; grad only for x."""

    @staticmethod
    def forward(ctx, x, packed, absmax, absmax_q, nested_absmax, nested_offset, code4, code8,
                N: int, K: int, double_quant: bool):
        w = ops.NF4Weight.from_tensors(
            (packed, absmax, absmax_q, nested_absmax, nested_offset, code4, code8), N, K,
            double_quant)
        lead = tuple(x.shape[:-1])
        y = ops.linear_fwd(x.reshape(-1, K).contiguous(), w)
        ctx.save_for_backward(packed, absmax, absmax_q, nested_absmax, nested_offset, code4, code8)
        ctx.N, ctx.K, ctx.double_quant = int(N), int(K), bool(double_quant)
        ctx.lead = lead
        return y.reshape(*lead, N)

    @staticmethod
    def backward(ctx, gy):
        saved = ctx.saved_tensors
        gx = None
        if ctx.needs_input_grad[0]:
            w = ops.NF4Weight.from_tensors(saved, ctx.N, ctx.K, ctx.double_quant)
            gx = ops.linear_dgrad(gy.reshape(-1, ctx.N).contiguous(), w).reshape(*ctx.lead, ctx.K)
        return gx, None, None, None, None, None, None, None, None, None, None


class NF4GroupedFn(torch.autograd.Function):
    """Per-expert y = x_e W_e^T over a stacked frozen NF4 weight; grad only for x."""

    @staticmethod
    def forward(ctx, x, offsets, packed, absmax, absmax_q, nested_absmax, nested_offset, code4,
                code8, experts: int, N: int, K: int, double_quant: bool):
        w = ops.NF4Weight.from_tensors(
            (packed, absmax, absmax_q, nested_absmax, nested_offset, code4, code8), N, K,
            double_quant)
        y = ops.grouped_fwd(x.contiguous(), offsets, w, experts)
        ctx.save_for_backward(offsets, packed, absmax, absmax_q, nested_absmax, nested_offset,
                              code4, code8)
        ctx.experts, ctx.N, ctx.K, ctx.double_quant = int(experts), int(N), int(K), bool(double_quant)
        return y

    @staticmethod
    def backward(ctx, gy):
        offsets, *rest = ctx.saved_tensors
        gx = None
        if ctx.needs_input_grad[0]:
            w = ops.NF4Weight.from_tensors(tuple(rest), ctx.N, ctx.K, ctx.double_quant)
            gx = ops.grouped_dgrad(gy.contiguous(), offsets, w, ctx.experts)
        return (gx,) + (None,) * 12


class NF4GroupedSwiGLUFn(torch.autograd.Function):
    """h = silu(x_e Wg_e^T) * (x_e Wu_e^T) * rw for grouped experts whose gate and up
    weights are interleaved (ops.interleave_gate_up) in one frozen 4-bit weight; the
    forward is one fused kernel (nf4_grouped_fwd_ep).  The backward is one library
    call (nf4_grouped_swiglu_bwd): the kernel recomputes gate and up, forms their
    gradients in its epilogue, and one grouped input-gradient product gives grad_x;
    the routing weights get their gradient (sum over the row of silu(g) u dh) when
    they require it.  Only the quantised weight (through save_for_backward), x and
    rw are kept."""

    @staticmethod
    def forward(ctx, x, offsets, row_scale, packed, absmax, absmax_q, nested_absmax,
                nested_offset, code4, code8, experts: int, N: int, K: int, double_quant: bool):
        w = ops.NF4Weight.from_tensors(
            (packed, absmax, absmax_q, nested_absmax, nested_offset, code4, code8), N, K,
            double_quant)
        h = ops.grouped_fwd(x.contiguous(), offsets, w, experts, row_scale=row_scale, swiglu=True)
        ctx.save_for_backward(x, offsets, row_scale, packed, absmax, absmax_q, nested_absmax,
                              nested_offset, code4, code8)
        ctx.experts, ctx.N, ctx.K, ctx.double_quant = int(experts), int(N), int(K), bool(double_quant)
        return h

    @staticmethod
    def backward(ctx, gh):
        x, offsets, rw, *wt = ctx.saved_tensors
        gx = grw = None
        need_rw = rw is not None and ctx.needs_input_grad[2]
        if ctx.needs_input_grad[0] or need_rw:
            w = ops.NF4Weight.from_tensors(tuple(wt), ctx.N, ctx.K, ctx.double_quant)
            gx, grw = ops.grouped_swiglu_bwd(x.contiguous(), offsets, w, ctx.experts,
                                             gh.contiguous(), row_scale=rw,
                                             need_row_scale_grad=need_rw)
            if not ctx.needs_input_grad[0]:
                gx = None
        return (gx, None, grw) + (None,) * 11


def nf4_grouped_swiglu(x: torch.Tensor, offsets: torch.Tensor, w: ops.NF4Weight, experts: int,
                       row_scale: torch.Tensor = None) -> torch.Tensor:
    """Fused expert SwiGLU over an interleaved gate/up weight (bf16 activations)."""
    return NF4GroupedSwiGLUFn.apply(x, offsets, row_scale, *w.tensors(), experts, w.N, w.K,
                                    w.double_quant)


class NF4MultiLinearFn(torch.autograd.Function):
    """y_p = x_p W_p^T for up to four frozen NF4 weights of the same in-features in
    one multi-product launch (nf4_linear_fwd_multi), and their input gradients in
    one nf4_linear_dgrad_multi launch.  Arguments: n, the weights' (N, double_quant)
    pairs, the n activations (the same tensor when the products share an input:
    autograd then adds their gradients), then the seven tensors of each weight, all
    saved through save_for_backward."""

    @staticmethod
    def forward(ctx, n: int, meta: tuple, K: int, *args):
        xs, tens = args[:n], args[n:]
        ws = [ops.NF4Weight.from_tensors(tuple(tens[7 * p:7 * p + 7]), meta[p][0], K, meta[p][1])
              for p in range(n)]
        lead = tuple(xs[0].shape[:-1])
        ys = ops.linear_fwd_multi([x.reshape(-1, K).contiguous() for x in xs], ws)
        ctx.save_for_backward(*tens)
        ctx.n, ctx.meta, ctx.K, ctx.lead = int(n), tuple((int(N), bool(dq)) for N, dq in meta), int(K), lead
        return tuple(y.reshape(*lead, meta[p][0]) for p, y in enumerate(ys))

    @staticmethod
    def backward(ctx, *gys):
        n, K = ctx.n, ctx.K
        saved = ctx.saved_tensors
        if not any(ctx.needs_input_grad[3:3 + n]):
            return (None,) * (3 + len(saved) + n)
        ws = [ops.NF4Weight.from_tensors(tuple(saved[7 * p:7 * p + 7]), ctx.meta[p][0], K, ctx.meta[p][1])
              for p in range(n)]
        gxs = ops.linear_dgrad_multi([g.reshape(-1, ctx.meta[p][0]).contiguous() for p, g in enumerate(gys)], ws)
        gxs = [gx.reshape(*ctx.lead, K) if ctx.needs_input_grad[3 + p] else None for p, gx in enumerate(gxs)]
        return (None, None, None, *gxs) + (None,) * len(saved)


def nf4_linear_multi(x: torch.Tensor, ws) -> tuple:
    """Frozen NF4 Linears that share their input (for instance q, k and v, or gate and
    up): one multi-product launch forward and one backward (bf16 compute; other
    input dtypes are cast to bf16 and the outputs cast back).  Returns one output
    per weight."""
    dt = x.dtype
    xb = x if dt == torch.bfloat16 else x.to(torch.bfloat16)
    K = ws[0].K
    meta = tuple((w.N, w.double_quant) for w in ws)
    tens = [t for w in ws for t in w.tensors()]
    ys = NF4MultiLinearFn.apply(len(ws), meta, K, *([xb] * len(ws)), *tens)
    return ys if dt == torch.bfloat16 else tuple(y.to(dt) for y in ys)


class NF4MoECombineFn(torch.autograd.Function):
    """The top-k combine of the grouped experts (nf4_moe_combine): token t's output
    is the sum of its routed rows; the backward (nf4_moe_combine_bwd) copies each
    token's gradient to its rows.  The route table goes through save_for_backward."""

    @staticmethod
    def forward(ctx, rows, token_rows):
        y = ops.moe_combine(rows.contiguous(), token_rows)
        ctx.save_for_backward(token_rows)
        ctx.R = int(rows.shape[0])
        return y

    @staticmethod
    def backward(ctx, gy):
        (token_rows,) = ctx.saved_tensors
        g = ops.moe_combine_bwd(gy.contiguous(), token_rows, ctx.R) if ctx.needs_input_grad[0] else None
        return g, None


def nf4_combine(rows: torch.Tensor, token_rows: torch.Tensor) -> torch.Tensor:
    """Sum each token's routed expert rows (bf16; see ops.route_rows for the table)."""
    return NF4MoECombineFn.apply(rows, token_rows)


def nf4_linear(x: torch.Tensor, w: ops.NF4Weight) -> torch.Tensor:
    """Frozen NF4 Linear: the compute dtype is the activations' half-precision type,
    bf16 or fp16 (the dtype handling of Linear4bit, which Soup issue #842's "Design
    sketch" keeps); other input dtypes are cast to bf16 and the output cast back (the
    casts are ordinary autograd ops)."""
    dt = x.dtype
    if dt == torch.float16 and w.bits == 4:
        return NF4LinearFn.apply(x, *w.tensors(), w.N, w.K, w.double_quant)
    xb = x if dt == torch.bfloat16 else x.to(torch.bfloat16)
    y = NF4LinearFn.apply(xb, *w.tensors(), w.N, w.K, w.double_quant)
    return y if dt == torch.bfloat16 else y.to(dt)


def nf4_grouped(x: torch.Tensor, offsets: torch.Tensor, w: ops.NF4Weight, experts: int) -> torch.Tensor:
    dt = x.dtype
    xb = x if dt == torch.bfloat16 else x.to(torch.bfloat16)
    y = NF4GroupedFn.apply(xb, offsets, *w.tensors(), experts, w.N, w.K, w.double_quant)
    return y if dt == torch.bfloat16 else y.to(dt)


class NF4Linear(torch.nn.Module):
    """A frozen NF4 Linear layer without bias (biases stay in native ops)."""

    def __init__(self, w: ops.NF4Weight):
        super().__init__()
        self.w = w

    @classmethod
    def from_float(cls, weight: torch.Tensor, double_quant: bool = True,
                   quant_type: str = "nf4") -> "NF4Linear":
        return cls(ops.quantize(weight.detach().contiguous(), double_quant=double_quant,
                                quant_type=quant_type))

    def forward(self, x):
        return nf4_linear(x, self.w)
