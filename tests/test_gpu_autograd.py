"""The autograd Functions on the GPU: gradients through the fused kernels match
the oracle, only save_for_backward carries the weight (no dense weight saved), an
in-place change of the saved packed weight is caught by autograd's version
counter, and under non-reentrant activation checkpointing with recycled weight
buffers the gradients equal the private-buffer run bit for bit while a control
that keeps the weight as a ctx attribute gets them wrong (bitsandbytes issue
"MatMul4Bit keeps B and quant_state on ctx", "Minimal reproducer" and "What it
prints"; Soup issue #842, "Acceptance criteria": aliasing control)."""
import numpy as np
import pytest
import torch
from torch.utils.checkpoint import checkpoint

import oracle
import bit_nf4_quantized_linear_gb300 as nf4
from bit_nf4_quantized_linear_gb300 import ops, synth
from tests.helpers import bf16_bits, oracle_state, parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    nf4.device_status(clear=True)


def test_function_grad_matches_oracle():
    g = synth.generator(7)
    N, K, M = 384, 512, 48
    w32 = synth.weight(N, K, g)
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    w = nf4.quantize(w32.to(DEV), double_quant=True)
    xd = x.to(DEV).requires_grad_(True)
    y = nf4.nf4_linear(xd.view(4, 12, K), w)
    assert y.shape == (4, 12, N)
    y.backward(gy.to(DEV).view(4, 12, N))
    wb = oracle.dequantize(oracle_state(w32, True), "bf16")
    parity(y.reshape(M, N), oracle.linear_fwd(bf16_bits(x), wb), "fn fwd")
    parity(xd.grad, oracle.linear_dgrad(bf16_bits(gy), wb), "fn dgrad")


def test_fp32_input_is_cast():
    g = synth.generator(8)
    w = nf4.quantize(synth.weight(128, 128, g).to(DEV))
    x = torch.randn(5, 128, device=DEV, requires_grad=True)
    y = nf4.nf4_linear(x, w)
    assert y.dtype == torch.float32
    y.sum().backward()
    assert x.grad.dtype == torch.float32 and torch.isfinite(x.grad).all()


def test_saves_no_weight_shaped_tensor():
    g = synth.generator(9)
    N, K, M = 256, 384, 16
    w = nf4.quantize(synth.weight(N, K, g).to(DEV), double_quant=True)
    saved = []

    def pack(t):
        saved.append((tuple(t.shape), t.dtype, t.numel() * t.element_size()))
        return t

    x = synth.activation(M, K, g).to(DEV).requires_grad_(True)
    with torch.autograd.graph.saved_tensors_hooks(pack, lambda t: t):
        y = nf4.nf4_linear(x, w)
    y.float().sum().backward()
    for shape, dtype, _ in saved:
        assert not (dtype.is_floating_point and shape in ((N, K), (K, N))), shape
    assert sum(b for _, _, b in saved) <= w.nbytes()
    # a plain dequantise + linear control does save a weight-shaped tensor
    saved.clear()
    with torch.autograd.graph.saved_tensors_hooks(pack, lambda t: t):
        wd = nf4.dequantize(w)
        torch.nn.functional.linear(x, wd)
    assert any(s in ((N, K), (K, N)) for s, _, _ in saved)


def test_inplace_change_of_saved_weight_is_caught():
    g = synth.generator(10)
    w = nf4.quantize(synth.weight(128, 128, g).to(DEV))
    x = synth.activation(4, 128, g).to(DEV).requires_grad_(True)
    y = nf4.nf4_linear(x, w)
    w.packed.add_(1)
    with pytest.raises(RuntimeError, match="modified by an inplace operation"):
        y.float().sum().backward()


class _CtxAttrFn(torch.autograd.Function):
    """Negative control: the packed weight is kept as a ctx attribute (the
    MatMul4Bit pattern), invisible to checkpointing."""

    @staticmethod
    def forward(ctx, x, w_tensors, N, K, dq):
        w = ops.NF4Weight.from_tensors(w_tensors, N, K, dq)
        ctx.w = w
        return ops.linear_fwd(x.contiguous(), w)

    @staticmethod
    def backward(ctx, gy):
        return ops.linear_dgrad(gy.contiguous(), ctx.w), None, None, None, None


class SlotPool:
    def __init__(self, n, like):
        self.slots = [torch.empty_like(like) for _ in range(n)]
        self.cursor = 0

    def acquire(self, src):
        s = self.slots[self.cursor % len(self.slots)]
        self.cursor += 1
        s.copy_(src)
        return s


def _aliasing_run(layers, x0, scales, arm):
    recycle = arm in ("recycled", "control")
    pool = SlotPool(2, layers[0].packed) if recycle else None
    params = [s.clone().requires_grad_(True) for s in scales]

    def body(i):
        def fn(h, scale):
            h = h * scale
            packed = pool.acquire(layers[i].packed) if recycle else layers[i].packed
            wt = list(layers[i].tensors())
            wt[0] = packed
            if arm == "control":
                return _CtxAttrFn.apply(h, tuple(wt), layers[i].N, layers[i].K, layers[i].double_quant)
            return nf4.NF4LinearFn.apply(h, *wt, layers[i].N, layers[i].K, layers[i].double_quant)
        return fn

    h = x0.clone().requires_grad_(True)
    for i in range(len(layers)):
        h = checkpoint(body(i), h, params[i], use_reentrant=False)
    h.float().pow(2).mean().backward()
    return [p.grad.float().clone() for p in params]


def test_checkpoint_recycled_buffers_exact_and_control_wrong():
    # 8 layers of 4096 x 4096 NF4 (double quant), M = 256, two recycled slots.
    g = synth.generator(12)
    D, L, M = 4096, 8, 256
    layers = [nf4.quantize((torch.randn(D, D, generator=g) / 32).to(DEV), double_quant=True)
              for _ in range(L)]
    x0 = synth.activation(M, D, g).to(DEV)
    scales = [(1 + 0.01 * torch.randn(D, generator=g)).to(DEV, torch.bfloat16) for _ in range(L)]
    ref = _aliasing_run(layers, x0, scales, "private")
    got = _aliasing_run(layers, x0, scales, "recycled")
    ctl = _aliasing_run(layers, x0, scales, "control")
    for i in range(L):
        assert torch.equal(got[i], ref[i]), f"layer {i}: recycled != private"
    wrong = [i for i in range(L) if not torch.equal(ctl[i], ref[i])]
    assert wrong[:L - 2] == list(range(L - 2)), f"control arm should be wrong on early layers: {wrong}"


def test_grouped_function_grad():
    g = synth.generator(13)
    E, N_e, K, tokens, topk = 8, 128, 256, 64, 2
    w32 = synth.weight(E * N_e, K, g)
    row_token, offsets = synth.routing(tokens, E, topk, g)
    x = synth.activation(tokens, K, g)[row_token].contiguous()
    gy = synth.activation(x.shape[0], N_e, g)
    w = nf4.quantize(w32.to(DEV), double_quant=False)
    xd = x.to(DEV).requires_grad_(True)
    y = nf4.nf4_grouped(xd, offsets.to(DEV), w, E)
    y.backward(gy.to(DEV))
    wb = oracle.dequantize(oracle_state(w32, False), "bf16").reshape(E, N_e, K)
    offs = offsets.numpy()
    parity(y, oracle.grouped_fwd(bf16_bits(x), offs, wb), "grouped fn fwd")
    parity(xd.grad, oracle.grouped_dgrad(bf16_bits(gy), offs, wb), "grouped fn dgrad")
