"""The 32B-class layer stack streamed through recycled weight slots, at its stated
size: hidden 5120, intermediate 27648, k/v width 1024, M = 4096 tokens, eight
layers of NF4 (double quantisation) q/k/v/o/gate/up/down weights of about 240 MiB
per layer, above the ~165 MiB per layer from which Soup issue #842's
"Acceptance criteria" ask for the aliasing control.

Every layer runs under non-reentrant activation checkpointing, and inside the
checkpointed region its quantised tensors are copied into one of two device slot
sets used in turn (bitsandbytes issue "MatMul4Bit keeps B and quant_state on
ctx", "Minimal reproducer": weights re-materialised into recycled buffers).
Layer body (the stack's reading: a trainable per-layer scale s upstream of the
projections, as the weight of an RMS normalisation of the layer input, which keeps
eight layers of N(0, 0.02) weights in range):
    h = x / rms(x) * s;  a = h + o(q(h));  kv = mean(k(h) * v(h));
    z = silu(gate(a)) * up(a);  out = a + down(z);
    loss = mean(out^2) + sum over layers of kv.
Checks: the gradients of every s and of x equal those of a run on private
buffers bit for bit; a Function that keeps the weight as a ctx attribute (the
MatMul4Bit pattern) gets the early layers wrong ("What it prints").  A further
test compares one projection of these shapes with the CPU oracle on sampled rows.
"""
import itertools

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.utils.checkpoint import checkpoint

import oracle
import bit_nf4_quantized_linear_gb300 as nf4
from bit_nf4_quantized_linear_gb300 import ops, synth
from tests.helpers import bf16_bits, oracle_state, parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
HIDDEN, M, LAYERS = 5120, 4096, 8


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    nf4.device_status(clear=True)
    yield
    assert nf4.device_status() == 0


class _KeepOnCtx(torch.autograd.Function):
    """Negative control: the quantised weight rides on ctx as a plain attribute,
    which activation checkpointing neither saves nor re-materialises."""

    @staticmethod
    def forward(ctx, x, w):
        ctx.weight = w
        return ops.linear_fwd(x.contiguous(), w)

    @staticmethod
    def backward(ctx, gy):
        return ops.linear_dgrad(gy.contiguous(), ctx.weight), None


def _apply(x, w, arm):
    if arm == "control":
        return _KeepOnCtx.apply(x, w)
    return nf4.NF4LinearFn.apply(x, *w.tensors(), w.N, w.K, w.double_quant)


class RecycledSlots:
    """Device buffers for every quantised tensor of one layer, `count` sets of them;
    `load(layer)` writes a layer into the next set (cycling) and returns weights
    that view that set."""

    def __init__(self, like: dict, count: int):
        self.sets = [{name: [None if t is None else torch.empty_like(t) for t in w.tensors()]
                      for name, w in like.items()} for _ in range(count)]
        self.order = itertools.cycle(range(count))

    def load(self, layer: dict) -> dict:
        dst = self.sets[next(self.order)]
        views = {}
        for name, w in layer.items():
            bufs = dst[name]
            for b, t in zip(bufs, w.tensors()):
                if b is not None:
                    b.copy_(t)
            views[name] = ops.NF4Weight.from_tensors(tuple(bufs), w.N, w.K, w.double_quant)
        return views


def _rms_scale(x, s):
    """x / sqrt(mean(x^2) + 1e-6) * s over the hidden dimension, in fp32, then bf16."""
    xf = x.float()
    return (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + 1e-6) * s.float()).to(torch.bfloat16)


def _stack_grads(layers, x0, scales, arm):
    """Gradients of every layer's scale and of the input for one arm: "private"
    (each layer reads its own tensors), "recycled" (copies into two slot sets
    inside the checkpointed regions) or "control" (recycled, weight on ctx)."""
    slots = RecycledSlots(layers[0], 2) if arm != "private" else None
    s_params = [s.clone().requires_grad_(True) for s in scales]
    x = x0.clone().requires_grad_(True)

    def block(i):
        def run(x_in, s):
            w = layers[i] if slots is None else slots.load(layers[i])
            p = lambda t, name: _apply(t, w[name], arm)
            h = _rms_scale(x_in, s)
            a = h + p(p(h, "q"), "o")
            kv = (p(h, "k").float() * p(h, "v").float()).mean()
            z = F.silu(p(a, "gate")) * p(a, "up")
            return a + p(z, "down"), kv
        return run

    h, kv_total = x, 0.0
    for i in range(len(layers)):
        h, kv = checkpoint(block(i), h, s_params[i], use_reentrant=False)
        kv_total = kv_total + kv
    (h.float().pow(2).mean() + kv_total).backward()
    return [s.grad.clone() for s in s_params] + [x.grad.clone()]


def _stack_weights(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    layers = []
    for _ in range(LAYERS):
        layer = {}
        for name, K, N in synth.QWEN32B_PROJ:
            w32 = torch.randn(N, K, generator=g, device=DEV) * synth.WEIGHT_STD
            layer[name] = nf4.quantize(w32, double_quant=True)
            del w32
        layers.append(layer)
    return layers


def test_qwen32b_stack_recycled_slots_bit_equal_and_ctx_control_wrong():
    layers = _stack_weights(50)
    per_layer = sum(w.nbytes() for w in layers[0].values())
    assert per_layer > 165 * 2 ** 20, per_layer
    g = torch.Generator(device=DEV)
    g.manual_seed(51)
    x0 = torch.randn(M, HIDDEN, generator=g, device=DEV).to(torch.bfloat16)
    scales = [(1 + 0.01 * torch.randn(HIDDEN, generator=g, device=DEV)).to(torch.bfloat16)
              for _ in range(LAYERS)]
    ref = _stack_grads(layers, x0, scales, "private")
    got = _stack_grads(layers, x0, scales, "recycled")
    ctl = _stack_grads(layers, x0, scales, "control")
    assert all(torch.isfinite(t.float()).all() for t in ref)
    for i, (a, b) in enumerate(zip(got, ref)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"gradient {i}: recycled != private"
    wrong = [i for i in range(LAYERS) if not torch.equal(ctl[i], ref[i])]
    assert wrong[:LAYERS - 2] == list(range(LAYERS - 2)), f"control should be wrong early: {wrong}"
    assert not torch.equal(ctl[-1], ref[-1]), "control: the input gradient should be wrong"


def test_qwen32b_down_projection_sampled_against_oracle():
    # The widest contraction of the stack (down: K = 27648 -> N = 5120) at M = 4096:
    # quantisation bit-exact with the oracle, products on sampled rows.
    name, K, N = synth.QWEN32B_PROJ[-1]
    g = synth.generator(52)
    w32 = synth.weight(N, K, g)
    w = nf4.quantize(w32.to(DEV), double_quant=True)
    st = oracle_state(w32, True)
    assert np.array_equal(w.packed.cpu().numpy(), st.packed)
    assert np.array_equal(w.absmax_q.cpu().numpy(), st.absmax_q)
    wb = oracle.dequantize(st, "bf16")
    x = synth.activation(M, K, g)
    gy = synth.activation(M, N, g)
    rows = np.array([0, 1, 1777, 2048, M - 1], dtype=np.int64)
    y = nf4.linear_fwd(x.to(DEV), w)
    gx = nf4.linear_dgrad(gy.to(DEV), w)
    r = torch.from_numpy(rows).to(DEV)
    parity(y[r], oracle.linear_fwd(bf16_bits(x), wb, rows), "qwen32b down fwd")
    parity(gx[r], oracle.linear_dgrad(bf16_bits(gy), wb, rows), "qwen32b down dgrad")
