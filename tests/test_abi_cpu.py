"""The C-ABI library builds, loads without a GPU, exports every function that
include/nf4.h declares, and rejects bad arguments on the host before any launch."""
import ctypes

import pytest

from bit_nf4_quantized_linear_gb300 import _lib, build


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.lib()


def test_exports_every_declared_symbol(L):
    names = _lib.header_functions()
    assert {"nf4_quantize", "nf4_dequantize", "nf4_linear_fwd", "nf4_linear_dgrad",
            "nf4_grouped_fwd", "nf4_grouped_dgrad", "nf4_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_checked_build_loads_and_exports_every_declared_symbol(L):
    """The checked debug build (NF4_CHECKED=1: in-kernel index checks) is the same
    C ABI; it reports itself as such and the normal build does not."""
    path = build.build(checked=True)
    C = ctypes.CDLL(path)
    for n in _lib.header_functions():
        assert hasattr(C, n), n
    C.nf4_checked_build.restype = ctypes.c_int32
    assert C.nf4_checked_build() == 1
    assert L.nf4_checked_build() == 0


def test_status_strings(L):
    for code in range(10):
        s = L.nf4_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0 and s != b"unknown status"
    assert L.nf4_status_string(0) == b"ok"


def _weight(N=128, K=128, dq=0, blocksize=64):
    # Non-null dummy host addresses: validation must fail before anything is read.
    dummy = ctypes.c_void_p(0x1000)
    return _lib.nf4_weight(dummy, dummy, dummy, dummy, dummy, dummy, dummy, N, K, blocksize, 256, dq)


def test_host_validation_rejects_before_launch(L):
    w = _weight(K=100)
    x = ctypes.c_void_p(0x1000)
    assert L.nf4_linear_fwd(x, 4, 128, ctypes.byref(w), x, 128, None, 0, None) == 2  # K % 64
    w = _weight(blocksize=32)
    assert L.nf4_linear_fwd(x, 4, 128, ctypes.byref(w), x, 128, None, 0, None) == 7
    assert L.nf4_linear_fwd(x, 4, 128, None, x, 128, None, 0, None) == 1
    w = _weight()
    assert L.nf4_linear_fwd(x, -1, 128, ctypes.byref(w), x, 128, None, 0, None) == 1
    assert L.nf4_linear_fwd(x, 4, 64, ctypes.byref(w), x, 128, None, 0, None) == 1  # ldx < K
    # M == 0 is a no-op that touches nothing
    assert L.nf4_linear_fwd(None, 0, 128, ctypes.byref(w), None, 128, None, 0, None) == 0
    assert L.nf4_linear_dgrad(None, 0, 128, ctypes.byref(w), None, 128, None, 0, None) == 0
    # misaligned activation pointer / leading dimension
    bad = ctypes.c_void_p(0x1002)
    assert L.nf4_linear_fwd(bad, 4, 128, ctypes.byref(w), x, 128, None, 0, None) == 3
    assert L.nf4_linear_fwd(x, 4, 132, ctypes.byref(w), x, 128, None, 0, None) == 3
    # grouped: N must be E * N_e, E in range, offsets non-null
    off = ctypes.c_void_p(0x1000)
    assert L.nf4_grouped_fwd(x, off, 3, 10, 128, ctypes.byref(w), 64, x, 64, None) == 1
    assert L.nf4_grouped_fwd(x, None, 2, 10, 128, ctypes.byref(w), 64, x, 64, None) == 1
    assert L.nf4_grouped_fwd(x, off, 0, 10, 128, ctypes.byref(w), 64, x, 64, None) == 1
    assert L.nf4_grouped_fwd(x, off, 2, 0, 128, ctypes.byref(w), 64, None, 64, None) == 0
    # double quant without its tensors
    wd = _lib.nf4_weight(x, None, None, None, None, x, None, 128, 128, 64, 256, 1)
    assert L.nf4_linear_fwd(x, 4, 128, ctypes.byref(wd), x, 128, None, 0, None) == 1
    # quantize: bad block size, missing workspace for double quantisation
    assert L.nf4_quantize(x, 0, 4, 64, 32, 0, 256, x, x, x, x, x, x, x, None, 0, None) == 7
    assert L.nf4_quantize(x, 0, 4, 64, 64, 1, 256, x, x, x, x, x, x, x, None, 0, None) == 4
    assert L.nf4_quantize(x, 9, 4, 64, 64, 0, 256, x, x, x, x, x, x, x, None, 0, None) == 1
    assert L.nf4_quantize_8bit(x, 0, 4, 64, 32, 0, 256, x, x, x, x, x, x, x, None, 0, None) == 7
    assert L.nf4_quantize_8bit(x, 0, 4, 64, 64, 1, 256, x, x, x, x, x, x, x, None, 0, None) == 4
    # code width other than 4 or 8
    w3 = _lib.nf4_weight(x, x, None, None, None, x, None, 128, 128, 64, 256, 0, 3)
    assert L.nf4_linear_fwd(x, 4, 128, ctypes.byref(w3), x, 128, None, 0, None) == 1
    # fp16 entry points share the host checks
    w = _weight(K=100)
    assert L.nf4_linear_fwd_f16(x, 4, 128, ctypes.byref(w), x, 128, None, 0, None) == 2
    w = _weight()
    assert L.nf4_linear_dgrad_f16(None, 0, 128, ctypes.byref(w), None, 128, None, 0, None) == 0
    # grouped epilogue: required struct, SwiGLU needs N_e % 128 == 0 and N_e/2 output columns
    ep = _lib.nf4_epilogue(None, None, 1)
    assert L.nf4_grouped_fwd_ep(x, off, 2, 10, 128, ctypes.byref(w), 64, None, x, 64, None) == 1
    assert L.nf4_grouped_fwd_ep(x, off, 2, 10, 128, ctypes.byref(w), 64, ctypes.byref(ep), x, 64, None) == 2
    ep_bad = _lib.nf4_epilogue(None, None, 2)
    assert L.nf4_grouped_fwd_ep(x, off, 1, 10, 128, ctypes.byref(w), 128, ctypes.byref(ep_bad), x, 64, None) == 1
    assert L.nf4_grouped_fwd_ep(x, off, 1, 10, 128, ctypes.byref(w), 128, ctypes.byref(ep), x, 32, None) == 1
    assert L.nf4_grouped_fwd_ep(x, off, 1, 0, 128, ctypes.byref(w), 128, ctypes.byref(ep), x, 64, None) == 0


def test_quantize_workspace_size(L):
    assert L.nf4_workspace_size(0, 0, 4096, 4096, 0) == ((4096 * 4096 // 64 + 1023) // 1024) * 8
    assert L.nf4_workspace_size(0, 0, 1, 64, 0) == 8


def test_path_counters_start_at_zero(L):
    _lib.reset_path_counters()
    assert all(v == 0 for v in _lib.path_counters().values())


def test_swiglu_backward_host_validation(L):
    x = ctypes.c_void_p(0x1000)
    off = ctypes.c_void_p(0x1000)
    w = _weight(N=256, K=128)
    ep = _lib.nf4_epilogue(None, x, 1)
    T, N_e = 10, 256
    need = L.nf4_workspace_size(_lib.OP_GROUPED_SWIGLU_BWD, T, N_e, 128, 1)
    # dg / du in bf16 (padded to 256 bytes), then N_e / 64 fp32 partials per row
    assert need == (T * N_e * 2 + 255) // 256 * 256 + (N_e // 64) * T * 4
    ws = ctypes.c_void_p(0x10000)
    call = lambda ep_, drw, ws_, nbytes, ldgh=128, gh=x: L.nf4_grouped_swiglu_bwd(
        x, off, 1, T, 128, ctypes.byref(w), N_e, ep_, gh, ldgh, x, 128, drw, ws_, nbytes, None)
    assert call(None, None, ws, need) == 1                                   # epilogue required
    assert call(ctypes.byref(_lib.nf4_epilogue(None, x, 0)), None, ws, need) == 1  # swiglu must be 1
    no_scale = _lib.nf4_epilogue(None, None, 1)
    assert call(ctypes.byref(no_scale), x, ws, need) == 1   # routing-weight grad without weights
    assert call(ctypes.byref(ep), x, None, 0) == 4          # workspace missing
    assert call(ctypes.byref(ep), x, ws, need - 4) == 4     # workspace too small
    assert call(ctypes.byref(ep), x, ctypes.c_void_p(0x10010), need) == 3  # not 256-byte aligned
    assert call(ctypes.byref(ep), x, ws, need, ldgh=64) == 1              # ldgh < N_e / 2
    assert call(ctypes.byref(ep), x, ws, need, ldgh=132) == 3             # ldgh % 8
    assert call(ctypes.byref(ep), x, ws, need, gh=ctypes.c_void_p(0x1008)) == 3
    # T == 0 is a no-op
    assert L.nf4_grouped_swiglu_bwd(x, off, 1, 0, 128, ctypes.byref(w), N_e, ctypes.byref(ep), None,
                                    128, None, 128, None, None, 0, None) == 0


def test_multi_product_host_validation(L):
    """nf4_linear_*_multi reject bad arguments on the host, before any device call."""
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    dummy = 0x1000

    def call(ws, M=4, ld=256, nprod=None, aligned=True, fn=L.nf4_linear_fwd_multi):
        n = len(ws) if nprod is None else nprod
        k = max(n, len(ws), 1)
        ptr = dummy if aligned else dummy + 2
        acts = (P * k)(*([ptr] * k))
        outs = (P * k)(*([ptr] * k))
        lds = (I64 * k)(*([ld] * k))
        warr = (P * k)(*([ctypes.addressof(w) for w in ws] + [None] * (k - len(ws))))
        return fn(n, acts, M, lds, warr, outs, lds, None)

    a, b = _weight(N=128, K=128), _weight(N=256, K=128)
    assert call([a, b], nprod=0) == 1
    assert call([a] * 5) == 1                     # more than NF4_MAX_MULTI products
    assert call([a, _weight(N=128, K=192)]) == 1  # different K
    assert call([a, _weight(N=128, K=128, dq=1)]) == 1  # different double_quant
    w8 = _weight(N=128, K=128)
    w8.bits = 8
    assert call([a, w8]) == 7                     # one-byte codes
    assert call([_weight(N=128, K=100)] * 2, ld=256) == 2  # K % 64
    assert call([a, b], ld=64) == 1               # leading dimension below the width
    assert call([a, b], aligned=False) == 3       # misaligned activations / outputs
    assert call([a, b], M=0) == 0                 # M == 0: nothing to do
    assert call([a, b], ld=256, fn=L.nf4_linear_dgrad_multi, aligned=False) == 3


def test_moe_combine_host_validation(L):
    x = ctypes.c_void_p(0x1000)
    assert L.nf4_moe_combine(x, 8, 64, x, 4, 0, 64, x, 64, None) == 1      # k < 1
    assert L.nf4_moe_combine(x, 8, 64, x, 4, 2, 60, x, 64, None) == 2      # H % 8
    assert L.nf4_moe_combine(x, 8, 32, x, 4, 2, 64, x, 64, None) == 1      # pitch below H
    assert L.nf4_moe_combine(ctypes.c_void_p(0x1002), 8, 64, x, 4, 2, 64, x, 64, None) == 3  # misaligned
    assert L.nf4_moe_combine(x, 8, 64, x, 0, 2, 64, x, 64, None) == 0      # no tokens
    assert L.nf4_moe_combine_bwd(x, 4, 64, x, 2, 8, 64, ctypes.c_void_p(0x1002), 64, None) == 3
