"""Autograd semantics of NF4LinearFn on the CPU, with the two product calls
replaced by a test double built on the CPU oracle (the library itself has no CPU
path).  What is checked here is the bookkeeping the bitsandbytes issue "MatMul4Bit
keeps B and quant_state on ctx" is about: every tensor the backward needs goes
through save_for_backward, so (1) nothing weight-shaped is saved, (2) an in-place
change of the saved packed weight is caught by the version counter, and (3) under
non-reentrant checkpointing with weights copied into recycled slots the gradients
equal the private-buffer run exactly, while a control that keeps the packed
weight as a ctx attribute gets the early layers wrong ("What it prints")."""
import numpy as np
import pytest
import torch
from torch.utils.checkpoint import checkpoint

import oracle
from oracle import codebooks as ocb
import bit_nf4_quantized_linear_gb300 as nf4
from bit_nf4_quantized_linear_gb300 import ops


def _dequant_bf16(w):
    st = oracle.QuantState((w.N, w.K), 64, w.packed.numpy(), None if w.absmax is None else w.absmax.numpy(),
                           w.code4.numpy(), w.double_quant,
                           None if w.absmax_q is None else w.absmax_q.numpy(),
                           None if w.nested_absmax is None else w.nested_absmax.numpy(),
                           None if w.nested_offset is None else w.nested_offset.numpy(),
                           None if w.code8 is None else w.code8.numpy(), 256)
    wb = oracle.dequantize(st, "bf16")
    return torch.from_numpy(oracle.bf16_bits_to_f32(wb).copy())


@pytest.fixture
def cpu_products(monkeypatch):
    def fwd(x, w, out=None, ws=None):
        return (x.float() @ _dequant_bf16(w).T).to(torch.bfloat16)

    def dgrad(gy, w, out=None, ws=None):
        return (gy.float() @ _dequant_bf16(w)).to(torch.bfloat16)

    monkeypatch.setattr(ops, "linear_fwd", fwd)
    monkeypatch.setattr(ops, "linear_dgrad", dgrad)


def _weight(N, K, seed, dq=True):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((N, K)) / 32).astype(np.float32)
    st = oracle.quantize(w, ocb.nf4_code4(), 64, dq, ocb.dynamic_code8(), 256)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a))
    return ops.NF4Weight(t(st.packed), t(st.absmax), t(st.absmax_q) if dq else None,
                         t(st.nested_absmax) if dq else None, t(st.nested_offset) if dq else None,
                         t(ocb.nf4_code4()), t(ocb.dynamic_code8()) if dq else None, N, K, dq)


def test_saved_tensors_are_the_quantised_weight_only(cpu_products):
    N, K = 96, 128
    w = _weight(N, K, 0)
    saved = []
    x = torch.randn(5, K).to(torch.bfloat16).requires_grad_(True)
    with torch.autograd.graph.saved_tensors_hooks(lambda t: (saved.append(t), t)[1], lambda t: t):
        y = nf4.nf4_linear(x, w)
    assert all(not (t.dtype.is_floating_point and tuple(t.shape) in ((N, K), (K, N))) for t in saved)
    ids = {id(t) for t in saved}
    for t in w.tensors():
        if t is not None:
            assert id(t) in ids or any(s.data_ptr() == t.data_ptr() for s in saved)
    y.float().sum().backward()
    ref = (torch.ones(5, N) @ _dequant_bf16(w)).to(torch.bfloat16)
    assert torch.equal(x.grad, ref)


def test_version_counter_catches_inplace_weight_change(cpu_products):
    w = _weight(64, 64, 1, dq=False)
    x = torch.randn(3, 64).to(torch.bfloat16).requires_grad_(True)
    y = nf4.nf4_linear(x, w)
    w.packed.add_(1)
    with pytest.raises(RuntimeError, match="modified by an inplace operation"):
        y.float().sum().backward()


class _CtxAttrFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w):
        ctx.w = w  # the MatMul4Bit pattern: invisible to checkpointing
        return ops.linear_fwd(x, w)

    @staticmethod
    def backward(ctx, gy):
        return ops.linear_dgrad(gy, ctx.w), None


def _run(layers, x0, scales, arm):
    slots = [torch.empty_like(layers[0].packed) for _ in range(2)] if arm != "private" else None
    cursor = [0]
    params = [s.clone().requires_grad_(True) for s in scales]

    def body(i):
        def fn(h, scale):
            h = h * scale
            w = layers[i]
            if slots is not None:
                slot = slots[cursor[0] % 2]
                cursor[0] += 1
                slot.copy_(w.packed)
                w = ops.NF4Weight(slot, w.absmax, w.absmax_q, w.nested_absmax, w.nested_offset,
                                  w.code4, w.code8, w.N, w.K, w.double_quant)
            if arm == "control":
                return _CtxAttrFn.apply(h, w)
            return nf4.nf4_linear(h, w)
        return fn

    h = x0.clone().requires_grad_(True)
    for i in range(len(layers)):
        h = checkpoint(body(i), h, params[i], use_reentrant=False)
    h.float().pow(2).mean().backward()
    return [p.grad.float().clone() for p in params]


def test_checkpoint_recycled_slots_exact_and_ctx_control_wrong(cpu_products):
    D, L, M = 128, 6, 16
    layers = [_weight(D, D, 10 + i) for i in range(L)]
    g = torch.Generator().manual_seed(0)
    x0 = torch.randn(M, D, generator=g).to(torch.bfloat16)
    scales = [(1 + 0.01 * torch.randn(D, generator=g)).to(torch.bfloat16) for _ in range(L)]
    ref = _run(layers, x0, scales, "private")
    got = _run(layers, x0, scales, "recycled")
    ctl = _run(layers, x0, scales, "control")
    for i in range(L):
        assert torch.equal(got[i], ref[i]), i
    wrong = [i for i in range(L) if not torch.equal(ctl[i], ref[i])]
    assert wrong[:L - 2] == list(range(L - 2)), wrong


def test_swiglu_function_returns_input_and_routing_weight_gradients(monkeypatch):
    # NF4GroupedSwiGLUFn with the two library calls replaced by oracle-backed test
    # doubles: the Function passes the saved x, offsets and routing weights to the
    # backward call, and returns its grad_x and routing-weight gradient.
    E, H, K = 2, 64, 64
    rng = np.random.default_rng(5)
    gate = (rng.standard_normal((E * H, K)) * 0.1).astype(np.float32)
    up = (rng.standard_normal((E * H, K)) * 0.1).astype(np.float32)
    w32 = oracle.interleave_gate_up(gate, up, E)
    w = _weight_from(w32)
    wb = oracle.dequantize(oracle.quantize(w32, ocb.nf4_code4(), 64, False), "bf16").reshape(E, 2 * H, K)
    offs = np.array([0, 3, 7], np.int32)
    bits = lambda t: t.detach().contiguous().view(torch.int16).numpy().view(np.uint16)
    calls = {}

    def fwd(x, offsets, w_, experts, out=None, bias=None, row_scale=None, swiglu=False):
        h = oracle.grouped_fwd_epilogue(bits(x), offsets.numpy(), wb,
                                        row_scale=None if row_scale is None else row_scale.numpy(),
                                        swiglu=swiglu)
        return torch.from_numpy(h).to(torch.bfloat16)

    def bwd(x, offsets, w_, experts, gh, bias=None, row_scale=None, need_row_scale_grad=False, ws=None):
        calls["need_rw"] = need_row_scale_grad
        gx, dr = oracle.grouped_swiglu_dgrad(bits(x), offsets.numpy(), wb, bits(gh),
                                             row_scale=None if row_scale is None else row_scale.numpy())
        return (torch.from_numpy(gx).to(torch.bfloat16),
                torch.from_numpy(dr).float() if need_row_scale_grad else None)

    monkeypatch.setattr(ops, "grouped_fwd", fwd)
    monkeypatch.setattr(ops, "grouped_swiglu_bwd", bwd)
    x = torch.from_numpy(rng.standard_normal((7, K)).astype(np.float32)).to(torch.bfloat16)
    rw = torch.from_numpy(rng.random(7).astype(np.float32))
    gh = torch.from_numpy(rng.standard_normal((7, H)).astype(np.float32)).to(torch.bfloat16)
    xr, rwr = x.clone().requires_grad_(True), rw.clone().requires_grad_(True)
    h = nf4.nf4_grouped_swiglu(xr, torch.from_numpy(offs), w, E, row_scale=rwr)
    h.backward(gh)
    assert calls["need_rw"] is True
    gx_ref, dr_ref = oracle.grouped_swiglu_dgrad(bits(x), offs, wb, bits(gh), row_scale=rw.numpy())
    assert torch.equal(xr.grad, torch.from_numpy(gx_ref).to(torch.bfloat16))
    assert torch.equal(rwr.grad, torch.from_numpy(dr_ref).float())
    # routing weights that need no gradient are not asked for one
    xr2 = x.clone().requires_grad_(True)
    nf4.nf4_grouped_swiglu(xr2, torch.from_numpy(offs), w, E, row_scale=rw).backward(gh)
    assert calls["need_rw"] is False and torch.equal(xr2.grad, xr.grad)


def _weight_from(w32):
    st = oracle.quantize(w32, ocb.nf4_code4(), 64, False)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return ops.NF4Weight(t(st.packed), t(st.absmax), None, None, None, t(ocb.nf4_code4()), None,
                         w32.shape[0], w32.shape[1], False)
