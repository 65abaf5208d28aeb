"""The allocation-free forward (nf4_linear_fwd_noalloc) through the C ABI.

Some callers cannot allocate device memory: code running under a framework
allocator that owns every device byte and forbids direct allocation, or a plugin
that is handed only its input and output buffers.  For them the forward keeps its
split-contraction partials in a fixed device array inside the library instead of
a caller workspace.  The test runs shapes whose plans really write and read that
array (a split contraction summed by the reduction kernel; the small-M cases with
the tiled kernel forced), two calls in a row on each, and checks every output
against nf4_linear_fwd with a caller workspace (the same plan and kernels, so bit
for bit) and against the CPU oracle within the products' tolerance.  A shape whose
partials exceed the array is refused.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import bit_nf4_quantized_linear_gb300 as nf4
from bit_nf4_quantized_linear_gb300 import _lib, ops, synth
from tests.helpers import bf16_bits, oracle_state, parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    nf4.device_status(clear=True)
    yield
    assert nf4.device_status() == 0


def _noalloc(x, w, y):
    s = w.struct()
    return _lib.lib().nf4_linear_fwd_noalloc(
        x.data_ptr(), x.shape[0], x.stride(0), ctypes.byref(s), y.data_ptr(), y.stride(0),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


# (M, N, K, force_tiles): every plan splits the contraction into the scratch array.
CASES = [(24, 1024, 2048, False), (48, 512, 8192, False), (16, 4096, 4096, True),
         (4, 4096, 4096, True), (9, 640, 1536, True)]


@pytest.mark.parametrize("M,N,K,force_tiles", CASES)
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(M, N, K, force_tiles):
    g = synth.generator(M + N + K)
    w32 = synth.weight(N, K, g)
    w = nf4.quantize(w32.to(DEV), double_quant=True)
    wb = oracle.dequantize(oracle_state(w32, True), "bf16")
    try:
        # The allocation-free call never takes the stream-K schedule (its partial
        # tiles outgrow the array); the reference call is given the same plan, and
        # both skip the cluster split, whose partials never leave shared memory, so
        # that the split partials go through the array.
        ops.set_stream_k(_lib.STREAM_K_OFF)
        ops.set_cluster_split(_lib.CLUSTER_SPLIT_OFF)
        ops.set_small_m_path(_lib.SMALL_M_TILES if force_tiles else _lib.SMALL_M_AUTO)
        plan = ops.plan_query(_lib.OP_LINEAR_FWD, M, N, K, nf4.device_check())
        assert plan["kernel"] == "fused" and plan["splits"] > 1 and not plan["stream_k"], plan
        assert 0 < plan["workspace_bytes"] <= _lib.NOALLOC_SCRATCH_BYTES
        for call in range(2):
            x = synth.activation(M, K, g)
            xd = x.to(DEV)
            ref = ops.linear_fwd(xd, w)
            y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
            before = nf4.path_counters()
            assert _noalloc(xd, w, y) == 0, _lib.lib().nf4_last_cuda_error()
            torch.cuda.synchronize()
            after = nf4.path_counters()
            # the fused kernel ran and its split partials were summed from the array
            assert after["linear_fwd"] == before["linear_fwd"] + 1
            assert after["splitk_reduce"] == before["splitk_reduce"] + 1
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), f"call {call}"
            parity(y, oracle.linear_fwd(bf16_bits(x), wb), f"noalloc call {call} M={M}")
    finally:
        ops.set_small_m_path(_lib.SMALL_M_AUTO)
        ops.set_stream_k(_lib.STREAM_K_AUTO)
        ops.set_cluster_split(_lib.CLUSTER_SPLIT_AUTO)


def test_noalloc_small_m_kernels_need_no_scratch():
    # M <= 16 on the default plan: the warp-MMA kernels, no partials at all.
    M, N, K = 8, 2048, 1024
    g = synth.generator(77)
    w32 = synth.weight(N, K, g)
    w = nf4.quantize(w32.to(DEV), double_quant=False)
    x = synth.activation(M, K, g)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    assert _noalloc(x.to(DEV), w, y) == 0
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ops.linear_fwd(x.to(DEV), w).view(torch.int16))
    parity(y, oracle.linear_fwd(bf16_bits(x), oracle.dequantize(oracle_state(w32, False), "bf16")),
           "noalloc small M")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    M, N, K = 32, 9728, 8192
    try:
        ops.set_stream_k(_lib.STREAM_K_OFF)
        ops.set_cluster_split(_lib.CLUSTER_SPLIT_OFF)
        plan = ops.plan_query(_lib.OP_LINEAR_FWD, M, N, K, nf4.device_check())
        g = synth.generator(5)
        w = nf4.quantize(synth.weight(N, K, g).to(DEV), double_quant=False)
        x = synth.activation(M, K, g).to(DEV)
        y = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
        rc = _noalloc(x, w, y)
        torch.cuda.synchronize()
        ref = ops.linear_fwd(x, w)
    finally:
        ops.set_stream_k(_lib.STREAM_K_AUTO)
        ops.set_cluster_split(_lib.CLUSTER_SPLIT_AUTO)
    if plan["workspace_bytes"] > _lib.NOALLOC_SCRATCH_BYTES:
        assert rc == 4  # NF4_ERR_WORKSPACE, nothing launched
        assert torch.count_nonzero(y) == 0
    else:
        assert rc == 0
        parity(y, ref.double().cpu().numpy(), "noalloc large")
