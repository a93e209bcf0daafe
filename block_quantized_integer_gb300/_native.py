"""ctypes loader of libqgemm.so (the C ABI declared in include/qgemm.h).

Loading fails loudly: there is no CPU fallback anywhere in this package.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqgemm.so")

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int32
SZ = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/qgemm.h
SIGNATURES = {
    "qg_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "qg_device_sm_count": (ctypes.c_int, []),
    "qg_device_error": (ctypes.c_uint, []),
    "qg_debug_set_wait_limit": (ctypes.c_int, [ctypes.c_longlong]),
    "qgemm_workspace_size": (SZ, [ctypes.c_int, I64, I64, I64, I64, I32, I32]),
    "quantize_act_q8": (ctypes.c_int, [P, I64, I64, I64, P, P, P]),
    "quantize_weight_q8_0": (ctypes.c_int, [P, I64, I64, P, P, P]),
    "quantize_weight_q4_0": (ctypes.c_int, [P, I64, I64, P, P, P]),
    "qgemm_q8_0": (ctypes.c_int, [P, P, I64, I64, I64, P, P, P, I64, P, SZ, P]),
    "qgemm_q4_0": (ctypes.c_int, [P, P, I64, I64, I64, P, P, P, I64, P, SZ, P]),
    "qgemv_q8_0_f32": (ctypes.c_int, [P, I64, I64, I64, P, P, I64, P, I64, P]),
    "qgemm_q8_0_ex": (ctypes.c_int, [P, P, I64, I64, I64, P, P, P, I64, P, SZ, ctypes.c_int, P]),
    "qgemm_q4_0_ex": (ctypes.c_int, [P, P, I64, I64, I64, P, P, P, I64, P, SZ, ctypes.c_int, P]),
    "moe_route": (ctypes.c_int, [P, I64, I32, I32, P, P, P, P, P]),
    "grouped_qgemm_moe": (ctypes.c_int, [P, P, I64, I64, P, I64, I32, I32, P, P, I32, I64, P,
                                         P, P, SZ, P]),
    "grouped_qgemm_moe_noalloc": (ctypes.c_int, [P, P, I64, I64, P, I64, I32, I32, P, P, I32,
                                                 I64, P, P, P]),
    "qgemm_debug_group_dots": (ctypes.c_int, [P, I64, I64, I64, P, ctypes.c_int, ctypes.c_int, P,
                                              P, SZ, P]),
    "import_gguf_q8_0": (ctypes.c_int, [P, I64, I64, P, P, P]),
    "import_gguf_q4_0": (ctypes.c_int, [P, I64, I64, P, P, P]),
    "attn_splitk_merge": (ctypes.c_int, [P, P, P, I32, I64, I64, P, P, P]),
    "kv3_encode": (ctypes.c_int, [P, I64, I32, I64, P, P, P]),
    "kv3_decode": (ctypes.c_int, [P, P, I64, I32, P, I64, P]),
    "qg_kv3_codebook": (None, [P, P]),
    "moe_swiglu_quant": (ctypes.c_int, [P, I64, I64, I64, P, P, P]),
    "moe_combine": (ctypes.c_int, [P, P, I64, I32, I64, P, P]),
}


class QGError(RuntimeError):
    def __init__(self, fn: str, status: int, name: str):
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status
        self.name = name


def load(path: str = LIB_PATH):
    """Load the library (building it first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path) or os.environ.get("QG_NO_AUTOBUILD") is None:
                from . import build as _build
                path = _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def call(name: str, *args) -> None:
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        raise QGError(name, st, lib.qg_status_string(st).decode())
