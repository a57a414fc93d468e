"""ctypes view of libmoe.so (the C ABI declared in include/moe.h). Marshalling only.

Importing this module does not need a GPU; calling a compute entry point does. If the
library has not been built, load() raises: there is no fallback implementation.
"""
import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "moe.h")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_DEVICE_TIMEOUT = -4
MOE_ERR_DEVICE_BOUNDS = -5
MOE_F32 = 0
MOE_BF16 = 1
MOE_ROW_ALIGN = 128
MOE_MAX_EXPERTS = 256
MOE_MAX_K = 8
MOE_MAX_WINDOW = 4096


class MoeConfig(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
        ("d_ff", ctypes.c_int32), ("capacity_factor", ctypes.c_float),
        ("temperature", ctypes.c_float), ("aux_loss_weight", ctypes.c_float),
        ("has_gate_bias", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("noise_std", ctypes.c_float), ("noise_seed", ctypes.c_uint32),
        ("capacity", ctypes.c_int32), ("rows_capacity", ctypes.c_int32),
        ("row_align", ctypes.c_int32),
    ]

    def __repr__(self):
        return "MoeConfig(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({status_str(status)})")


_P = ctypes.c_void_p
_CFG = ctypes.POINTER(MoeConfig)
_SIGS = {
    "moe_config_init": (ctypes.c_int, [_CFG]),
    "moe_workspace_bytes": (ctypes.c_size_t, [_CFG]),
    "moe_route": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_soft_balance": (ctypes.c_int, [_CFG, _P, ctypes.c_float, _P, _P, _P, _P]),
    "moe_soft_balance_backward": (ctypes.c_int, [_CFG, _P, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_expert_ffn": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_combine": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P]),
    "moe_backward": (ctypes.c_int, [_CFG] + [_P] * 26),
    "moe_coselect": (ctypes.c_int, [_CFG, _P, _P, _P]),
    "moe_get_error": (ctypes.c_int, [_P]),
    "moe_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_kernel_launches": (ctypes.c_uint64, []),
    "moe_version": (ctypes.c_char_p, []),
    "moe_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int64, _P, _P, _P]),
    "moe_soft_balance_window": (ctypes.c_int, [_CFG, _P, ctypes.c_float, ctypes.c_int32, _P, _P, _P, _P, _P,
                                               _P, _P]),
    "moe_soft_balance_window_backward": (ctypes.c_int, [_CFG, _P, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P,
                                                        _P, _P]),
    "moe_dispatch_noalloc": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_trace_begin": (ctypes.c_int, [ctypes.c_int32]),
    "moe_trace_end": (ctypes.c_int32, []),
    "moe_trace_record": (ctypes.c_int, [ctypes.c_int32, ctypes.POINTER(ctypes.c_char_p),
                                        ctypes.POINTER(ctypes.c_float)]),
    "moe_trace_dropped": (ctypes.c_int32, []),
}

_lib = None


def load():
    """Load libmoe.so once and declare the signatures. Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m token_routing_gb300.build` "
                               "(there is no non-CUDA fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_str(status):
    try:
        return load().moe_status_str(status).decode()
    except Exception:  # the library may be the thing that is missing
        return "unknown"


def check(fn_name, status):
    if status != MOE_OK:
        raise MoeError(fn_name, status)


def header_symbols(path=HEADER_PATH):
    """Names of the functions include/moe.h declares with MOE_API."""
    text = open(path).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)
