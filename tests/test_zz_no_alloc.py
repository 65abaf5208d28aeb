"""The allocation-free forward (nf4_linear_fwd_noalloc) through the C ABI.

It exists for callers that cannot allocate device memory themselves (code under
an allocator that owns all device memory, or a plugin handed only its inputs and
outputs): its split-contraction partials sit in a fixed device array inside the
library.  The test compares it with nf4_linear_fwd, which takes a caller-owned
workspace, on two calls in a row (the second must not be disturbed by what the
first left in the shared array), and checks that a shape needing more than the
fixed array is refused.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import bit_nf4_quantized_linear_gb300 as nf4
from bit_nf4_quantized_linear_gb300 import _lib, ops, synth
from tests.helpers import parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _noalloc(x, w, y):
    s = w.struct()
    return _lib.lib().nf4_linear_fwd_noalloc(
        x.data_ptr(), x.shape[0], x.stride(0), ctypes.byref(s), y.data_ptr(), y.stride(0),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("M,N,K", [(16, 4096, 4096), (24, 1024, 2048), (4, 4096, 4096),
                                   (200, 640, 512)])
def test_noalloc_matches_workspace_entry_point_twice(M, N, K):
    g = synth.generator(M + N)
    w = nf4.quantize(synth.weight(N, K, g).to(DEV), double_quant=True)
    for call in range(2):
        x = synth.activation(M, K, g).to(DEV)
        ref = ops.linear_fwd(x, w)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        before = nf4.path_counters()
        assert _noalloc(x, w, y) == 0, _lib.lib().nf4_last_cuda_error()
        torch.cuda.synchronize()
        after = nf4.path_counters()
        assert after["total"] > before["total"]
        parity(y, ref.double().cpu().numpy(), f"noalloc call {call} M={M}")
        # a small-M call on the tiled kernel really exercises the scratch (split
        # contraction, summed by the reduction kernel)
        if M <= 32 and after["linear_fwd"] > before["linear_fwd"]:
            assert after["splitk_reduce"] > before["splitk_reduce"]


def test_noalloc_refuses_shapes_beyond_its_scratch():
    M, N, K = 32, 9728, 8192
    need = ops.workspace_size(_lib.OP_LINEAR_FWD, M, N, K)
    g = synth.generator(5)
    w = nf4.quantize(synth.weight(N, K, g).to(DEV), double_quant=False)
    x = synth.activation(M, K, g).to(DEV)
    y = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    rc = _noalloc(x, w, y)
    torch.cuda.synchronize()
    if need > _lib.NOALLOC_SCRATCH_BYTES:
        assert rc == 4  # NF4_ERR_WORKSPACE, nothing launched
        assert torch.count_nonzero(y) == 0
    else:
        assert rc == 0
        parity(y, ops.linear_fwd(x, w).double().cpu().numpy(), "noalloc large")
