"""The autograd Functions on the GPU: gradients through the fused kernels match
the oracle, only save_for_backward carries the weight (no dense weight saved), and
an in-place change of the saved packed weight is caught by autograd's version
counter (bitsandbytes issue "MatMul4Bit keeps B and quant_state on ctx", "Why
save_for_backward fixes it").  The checkpointed stack with recycled weight slots
and its ctx-attribute control run at full size in test_gpu_stack.py."""
import pytest
import torch

import oracle
import bit_nf4_quantized_linear_gb300 as nf4
from bit_nf4_quantized_linear_gb300 import synth
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


def test_multi_linear_function_grad_matches_oracle():
    """q/k/v-shaped weights sharing their input through nf4_linear_multi: one
    multi-product launch each way; each output and the summed input gradient (the
    engine adds the products' gradients) against the oracle."""
    M, K, Ns = 48, 256, (256, 128, 128)
    g = synth.generator(17)
    ws, wbs = [], []
    for N in Ns:
        w32 = synth.weight(N, K, g)
        ws.append(nf4.quantize(w32.to(DEV), double_quant=True))
        wbs.append(oracle.dequantize(oracle_state(w32, True), "bf16"))
    x = synth.activation(M, K, g)
    gys = [synth.activation(M, N, g) for N in Ns]
    xd = x.to(DEV).requires_grad_(True)
    nf4.reset_path_counters()
    ys = nf4.nf4_linear_multi(xd, ws)
    torch.autograd.backward(ys, [gy.to(DEV) for gy in gys])
    c = nf4.path_counters()
    assert c["multi"] == 2 and c["linear_fwd"] == 0 and c["linear_dgrad"] == 0, c
    for y, wb, N in zip(ys, wbs, Ns):
        assert y.shape == (M, N)
        parity(y, oracle.linear_fwd(bf16_bits(x), wb), f"multi fwd {N}")
    ref = sum(oracle.linear_dgrad(bf16_bits(gy), wb) for gy, wb in zip(gys, wbs))
    parity(xd.grad, ref, "multi grad_x (sum over the products)")


def test_multi_linear_function_saves_no_weight_shaped_tensor():
    K, Ns = 256, (256, 128)
    g = synth.generator(18)
    ws = [nf4.quantize(synth.weight(N, K, g).to(DEV), double_quant=True) for N in Ns]
    x = synth.activation(8, K, g).to(DEV).requires_grad_(True)
    ys = nf4.nf4_linear_multi(x, ws)
    fn = ys[0].grad_fn
    assert type(fn).__name__.startswith("NF4MultiLinearFn")
    saved = [t for t in fn.saved_tensors if t is not None]
    for t in saved:
        assert t.shape != (Ns[0], K) and t.shape != (Ns[1], K)
    assert not [k for k, v in vars(fn).items() if isinstance(v, torch.Tensor)]
