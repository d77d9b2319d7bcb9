"""ctypes view of the C ABI in include/mla_dcp.h (same names, same order).

Loading fails loudly if the library has not been built: there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_LOCK = threading.Lock()
_LIB = None

P = ctypes.c_void_p
I = ctypes.c_int
F = ctypes.c_float

# name -> (restype, argtypes), mirroring include/mla_dcp.h
SIGNATURES = {
    "mla_dcp_decode_partial": (I, [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, P, P, P,
                                   ctypes.c_uint64, P]),
    "mla_dcp_decode_partial_sliced": (I, [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, P, P,
                                          P, ctypes.c_uint64, I, P]),
    "mla_dcp_decode_partial_fp8": (I, [P, P, P, P, P, P, I, I, I, I, I, I, I, F, F, I, I, P, P,
                                       P, P, ctypes.c_uint64, I, P]),
    "mla_dcp_decode_partial_workspace_size": (ctypes.c_uint64, [I, I, I, I]),
    "mla_dcp_combine_exchanged": (I, [P, P, I, I, I, I, I, I, I, I, P, P, P]),
    "mla_dcp_decode_partial_noalloc": (I, [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, P, P,
                                           P]),
    "mla_lse_combine": (I, [P, P, I, P, P, I, I, I, I, P, P, P]),
    "mla_vup": (I, [P, P, I, I, I, P, P, P]),
    "mla_lse_combine_vup": (I, [P, P, I, P, P, P, I, I, I, I, P, P, P, P, P]),
    "mla_gather_kv": (I, [P, P, P, I, I, I, I, I, P, P, P]),
    "mla_get_error_string": (ctypes.c_char_p, [I]),
    "mla_device_error_string": (ctypes.c_char_p, [I]),
    "mla_version": (I, []),
    "mla_debug_set_spin_limit": (None, [ctypes.c_uint32]),
}

STATUS = {0: "MLA_OK", 1: "MLA_ERR_NULL_POINTER", 2: "MLA_ERR_BAD_SHAPE",
          3: "MLA_ERR_BAD_DTYPE", 4: "MLA_ERR_MISALIGNED", 5: "MLA_ERR_BAD_SHARDS",
          6: "MLA_ERR_BAD_BLOCK", 7: "MLA_ERR_CUDA"}
DTYPE = {"bf16": 0, "fp16": 1, "fp32": 2}


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        text = lib().mla_get_error_string(status).decode()
        super().__init__(f"{fn} -> {STATUS.get(status, status)}: {text}")
        self.status = status


def lib(path: str | None = None):
    """Load libmla_dcp.so (built in-tree by ``build.build()``)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = path or _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build the CUDA library first "
                    "(mla_decode_attention_kv_gb300.build.build())")
            so = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(so, name)
                fn.restype = res
                fn.argtypes = args
            _LIB = so
    return _LIB


def check(fn: str, status: int) -> None:
    if status != 0:
        raise MlaError(fn, status)
