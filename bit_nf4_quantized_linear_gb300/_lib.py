"""ctypes binding of ``libnf4.so`` (the C ABI declared in ``include/nf4.h``).

Argument marshalling only.  Loading fails loudly when the library has not been
built: there is no fallback path of any kind.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
# NF4_CHECKED=1 selects the checked debug build (in-kernel index checks).
LIB_PATH = os.path.join(PKG, "libnf4_checked.so" if os.environ.get("NF4_CHECKED") == "1" else "libnf4.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "nf4.h")

NF4_OK = 0
NOALLOC_SCRATCH_BYTES = 2 << 20  # NF4_NOALLOC_SCRATCH_BYTES of include/nf4.h
STATUS_NAMES = {
    0: "NF4_OK", 1: "NF4_ERR_INVALID_ARG", 2: "NF4_ERR_UNSUPPORTED_SHAPE", 3: "NF4_ERR_ALIGNMENT",
    4: "NF4_ERR_WORKSPACE", 5: "NF4_ERR_CUDA", 6: "NF4_ERR_TIMEOUT", 7: "NF4_ERR_UNSUPPORTED",
    8: "NF4_ERR_BAD_OFFSETS", 9: "NF4_ERR_BOUNDS",
}
DTYPE_F32, DTYPE_BF16 = 0, 1
OP_QUANTIZE, OP_LINEAR_FWD, OP_LINEAR_DGRAD, OP_GROUPED_FWD, OP_GROUPED_DGRAD, OP_GROUPED_SWIGLU_BWD = range(6)
PATHS = ["linear_fwd", "linear_dgrad", "splitk_reduce", "grouped_fwd", "grouped_dgrad",
         "dequantize", "quantize", "total", "gemv_fwd", "gemv_dgrad", "skinny_fwd",
         "skinny_dgrad", "stream_k", "cluster_split", "multi", "moe_combine"]


class NF4Error(RuntimeError):
    def __init__(self, what: str, code: int):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}")
        self.code = code


class nf4_weight(ctypes.Structure):
    _fields_ = [
        ("packed", ctypes.c_void_p),
        ("absmax", ctypes.c_void_p),
        ("absmax_q", ctypes.c_void_p),
        ("nested_absmax", ctypes.c_void_p),
        ("nested_offset", ctypes.c_void_p),
        ("code4", ctypes.c_void_p),
        ("code8", ctypes.c_void_p),
        ("N", ctypes.c_int64),
        ("K", ctypes.c_int64),
        ("blocksize", ctypes.c_int32),
        ("nested_blocksize", ctypes.c_int32),
        ("double_quant", ctypes.c_int32),
        ("bits", ctypes.c_int32),
    ]


class nf4_epilogue(ctypes.Structure):
    _fields_ = [
        ("bias", ctypes.c_void_p),
        ("row_scale", ctypes.c_void_p),
        ("swiglu", ctypes.c_int32),
    ]


class nf4_plan_info(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int32),
        ("token_tile", ctypes.c_int32),
        ("splits", ctypes.c_int32),
        ("stream_k", ctypes.c_int32),
        ("grid", ctypes.c_int32),
        ("items", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_uint64),
        ("cluster_split", ctypes.c_int32),
        ("tail_tokens", ctypes.c_int32),
        ("tail_token_tile", ctypes.c_int32),
    ]


PLAN_KERNELS = {0: "fused", 1: "small_m_mma", 2: "simt_gemv"}

_lock = threading.Lock()
_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/nf4.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nf4_[a-z_0-9]+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        W = ctypes.POINTER(nf4_weight)
        sig = {
            "nf4_quantize": [P, I32, I64, I64, I32, I32, I32, P, P, P, P, P, P, P, P, SZ, P],
            "nf4_quantize_8bit": [P, I32, I64, I64, I32, I32, I32, P, P, P, P, P, P, P, P, SZ, P],
            "nf4_dequantize": [W, P, I32, P],
            "nf4_linear_fwd": [P, I64, I64, W, P, I64, P, SZ, P],
            "nf4_linear_dgrad": [P, I64, I64, W, P, I64, P, SZ, P],
            "nf4_linear_fwd_multi": [I32, P, I64, P, P, P, P, P],
            "nf4_moe_combine": [P, I64, I64, P, I64, I32, I64, P, I64, P],
            "nf4_moe_combine_bwd": [P, I64, I64, P, I32, I64, I64, P, I64, P],
            "nf4_linear_dgrad_multi": [I32, P, I64, P, P, P, P, P],
            "nf4_linear_fwd_f16": [P, I64, I64, W, P, I64, P, SZ, P],
            "nf4_linear_dgrad_f16": [P, I64, I64, W, P, I64, P, SZ, P],
            "nf4_grouped_fwd": [P, P, I32, I64, I64, W, I64, P, I64, P],
            "nf4_grouped_dgrad": [P, P, I32, I64, I64, W, I64, P, I64, P],
            "nf4_grouped_fwd_ep": [P, P, I32, I64, I64, W, I64, ctypes.POINTER(nf4_epilogue), P, I64, P],
            "nf4_grouped_swiglu_bwd": [P, P, I32, I64, I64, W, I64, ctypes.POINTER(nf4_epilogue), P, I64,
                                       P, I64, P, P, SZ, P],
            "nf4_workspace_size": [I32, I64, I64, I64, I32],
            "nf4_status_string": [I32],
            "nf4_checked_build": [],
            "nf4_inject_bounds_failure": [],
            "nf4_get_path_counters": [P],
            "nf4_reset_path_counters": [],
            "nf4_device_status": [P, I32],
            "nf4_device_check": [P],
            "nf4_last_cuda_error": [],
            "nf4_linear_fwd_noalloc": [P, I64, I64, W, P, I64, P],
            "nf4_set_weight_prefetch": [I32],
            "nf4_set_small_m_path": [I32],
            "nf4_set_stream_k": [I32],
            "nf4_set_cluster_split": [I32],
            "nf4_set_token_tile": [I32],
            "nf4_inject_stream_k_timeout": [],
            "nf4_plan_query": [I32, I64, I64, I64, I32, I32, I32, ctypes.POINTER(nf4_plan_info)],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.nf4_workspace_size.restype = ctypes.c_size_t
        L.nf4_status_string.restype = ctypes.c_char_p
        L.nf4_last_cuda_error.restype = ctypes.c_char_p
        L.nf4_get_path_counters.restype = None
        L.nf4_reset_path_counters.restype = None
        L.nf4_set_weight_prefetch.restype = None
        L.nf4_set_small_m_path.restype = None
        L.nf4_set_stream_k.restype = None
        L.nf4_set_cluster_split.restype = None
        L.nf4_set_token_tile.restype = None
        L.nf4_inject_stream_k_timeout.restype = None
        L.nf4_inject_bounds_failure.restype = None
        _lib = L
        return _lib


def check(rc: int, what: str):
    if rc != NF4_OK:
        if rc == 5:
            what = f"{what} ({lib().nf4_last_cuda_error().decode()})"
        raise NF4Error(what, rc)


def path_counters() -> dict:
    arr = (ctypes.c_uint64 * len(PATHS))()
    lib().nf4_get_path_counters(ctypes.cast(arr, ctypes.c_void_p))
    return {name: int(v) for name, v in zip(PATHS, arr)}


def reset_path_counters():
    lib().nf4_reset_path_counters()


def device_status(clear: bool = False) -> int:
    v = ctypes.c_int32(0)
    check(lib().nf4_device_status(ctypes.byref(v), 1 if clear else 0), "nf4_device_status")
    return int(v.value)


SMALL_M_AUTO, SMALL_M_SIMT, SMALL_M_TILES = 0, 1, 2


def set_small_m_path(path: int):
    lib().nf4_set_small_m_path(int(path))


STREAM_K_OFF, STREAM_K_AUTO, STREAM_K_FORCE = 0, 1, 2


def inject_bounds_failure():
    """Checked build only: the next fused-kernel product's statistics-load index
    checks fail (loads skipped, NF4_ERR_BOUNDS recorded); see
    nf4_inject_bounds_failure."""
    lib().nf4_inject_bounds_failure()


def checked_build() -> bool:
    """True when the loaded library is the checked debug build."""
    return bool(lib().nf4_checked_build())


def set_stream_k(mode: int):
    lib().nf4_set_stream_k(int(mode))


CLUSTER_SPLIT_OFF, CLUSTER_SPLIT_AUTO, CLUSTER_SPLIT_FORCE = 0, 1, 2


def set_cluster_split(mode: int):
    lib().nf4_set_cluster_split(int(mode))


def set_token_tile(tokens: int):
    """Fixed token tile of the fused kernel (64, 128 or 256), 0 for the planner's."""
    lib().nf4_set_token_tile(int(tokens))


def plan_query(op: int, M: int, N: int, K: int, sms: int, bits: int = 4, f16: bool = False) -> dict:
    """The launch plan of a dense product (host only, no device needed)."""
    r = nf4_plan_info()
    check(lib().nf4_plan_query(int(op), int(M), int(N), int(K), int(sms), int(bits),
                               1 if f16 else 0, ctypes.byref(r)), "nf4_plan_query")
    d = {name: getattr(r, name) for name, _ in nf4_plan_info._fields_}
    d["kernel"] = PLAN_KERNELS[d["kernel"]]
    return d


def inject_stream_k_timeout():
    """Failure-path test hook: the next stream-K launch's bounded waits run out
    (NF4_ERR_TIMEOUT in the device status word); see nf4_inject_stream_k_timeout."""
    lib().nf4_inject_stream_k_timeout()


def set_weight_prefetch(enabled: bool):
    lib().nf4_set_weight_prefetch(1 if enabled else 0)


def device_check() -> int:
    sms = ctypes.c_int32(0)
    check(lib().nf4_device_check(ctypes.byref(sms)), "nf4_device_check")
    return int(sms.value)
