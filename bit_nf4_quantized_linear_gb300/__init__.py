"""Fused NF4 dequantise-and-multiply for a frozen 4-bit Linear on GB300 (sm_103a).

The compute lives in ``libnf4.so`` (hand-written CUDA, C ABI in ``include/nf4.h``);
this package is its thin binding plus the autograd Functions.  Importing it does
not load the library; the first call does, and fails loudly if it is not built.
"""
from .autograd import (NF4GroupedFn, NF4GroupedSwiGLUFn, NF4Linear, NF4LinearFn, NF4MoECombineFn,
                       NF4MultiLinearFn, nf4_combine, nf4_grouped, nf4_grouped_swiglu, nf4_linear,
                       nf4_linear_multi)
from .codebooks import code4_for, code_for, dynamic_code8, e4m3_code8, fp4_code4, nf4_code4
from .ops import (NF4Weight, dequantize, device_check, device_status, grouped_dgrad, grouped_fwd,
                  grouped_swiglu_bwd, interleave_gate_up,
                  linear_dgrad, linear_dgrad_multi, linear_fwd, linear_fwd_multi, moe_combine,
                  moe_combine_bwd, path_counters, quantize, reset_path_counters, route_rows,
                  workspace_size)

# The C-ABI names.
nf4_quantize = quantize
nf4_quantize_8bit = quantize
nf4_dequantize = dequantize
nf4_linear_fwd = linear_fwd
nf4_linear_dgrad = linear_dgrad
nf4_linear_fwd_multi = linear_fwd_multi
nf4_linear_dgrad_multi = linear_dgrad_multi
nf4_moe_combine = moe_combine
nf4_moe_combine_bwd = moe_combine_bwd
nf4_grouped_fwd = grouped_fwd
nf4_grouped_fwd_ep = grouped_fwd
nf4_grouped_dgrad = grouped_dgrad
nf4_grouped_swiglu_bwd = grouped_swiglu_bwd
nf4_workspace_size = workspace_size

__all__ = [
    "NF4Weight", "NF4Linear", "NF4LinearFn", "NF4GroupedFn", "NF4GroupedSwiGLUFn", "NF4MultiLinearFn",
    "nf4_linear", "nf4_linear_multi", "linear_fwd_multi", "linear_dgrad_multi", "nf4_linear_fwd_multi",
    "nf4_linear_dgrad_multi", "NF4MoECombineFn", "nf4_combine", "nf4_moe_combine", "nf4_moe_combine_bwd",
    "moe_combine", "moe_combine_bwd", "route_rows",
    "nf4_grouped", "nf4_grouped_swiglu",
    "nf4_code4", "fp4_code4", "e4m3_code8", "code4_for", "code_for", "dynamic_code8", "quantize", "dequantize", "linear_fwd", "linear_dgrad",
    "grouped_fwd", "grouped_dgrad", "grouped_swiglu_bwd", "interleave_gate_up", "workspace_size", "path_counters", "reset_path_counters",
    "device_status", "device_check", "nf4_quantize", "nf4_dequantize", "nf4_linear_fwd",
    "nf4_linear_dgrad", "nf4_grouped_fwd", "nf4_grouped_dgrad", "nf4_grouped_swiglu_bwd",
    "nf4_workspace_size",
]
