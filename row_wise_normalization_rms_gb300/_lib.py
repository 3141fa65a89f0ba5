"""ctypes declarations of librmsnorm.so's C ABI (include/rmsnorm.h)."""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librmsnorm.so")

_lock = threading.Lock()
_lib = None

c_i64 = ctypes.c_int64
c_vp = ctypes.c_void_p
c_int = ctypes.c_int
c_float = ctypes.c_float
c_size = ctypes.c_size_t

# name -> (restype, argtypes), in header order.
SIGNATURES = {
    "rms_fwd": (c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_float, c_int, c_int, c_vp]),
    "rms_fwd_ex": (c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_float, c_int, c_int, c_int, c_vp]),
    "rms_bwd": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_int, c_int, c_int,
                        c_vp]),
    "rms_bwd_ex": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_i64, c_i64, c_int,
                           c_int, c_int, c_int, c_vp]),
    "rms_bwd_reduction": (c_int, [c_i64, c_i64, c_int, c_int, c_int, c_int, c_vp, c_vp]),
    "rms_dgamma_combine": (c_int, [c_vp, c_i64, c_i64, c_vp, c_vp]),
    "rms_dgamma_cast": (c_int, [c_vp, c_vp, c_i64, c_int, c_vp]),
    "rms_bwd_noalloc": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_int, c_int,
                                c_int, c_vp]),
    "rms_fwd_add": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_float, c_int, c_int,
                            c_vp]),
    "rms_fwd_add_ex": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_float, c_int,
                               c_int, c_int, c_vp]),
    "rms_fwd_quant": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_float, c_int, c_int,
                              c_vp]),
    "rms_fwd_quant_ex": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_float, c_int,
                                 c_int, c_int, c_vp]),
    "rms_bwd_add": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_int,
                            c_int, c_int, c_vp]),
    "rms_bwd_add_ex": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_i64,
                               c_i64, c_int, c_int, c_int, c_int, c_vp]),
    "ln_fwd": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_float, c_int, c_vp]),
    "ln_fwd_ex": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_float, c_int, c_int,
                          c_vp]),
    "ln_bwd": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_int,
                       c_int, c_vp]),
    "ln_bwd_ex": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_i64,
                          c_i64, c_int, c_int, c_int, c_vp]),
    "ln_bwd_reduction": (c_int, [c_i64, c_i64, c_int, c_int, c_vp, c_vp]),
    "ln_bwd_workspace_size": (c_size, [c_i64, c_i64]),
    "rms_bwd_workspace_size": (c_size, [c_i64, c_i64]),
    "rms_status_string": (ctypes.c_char_p, [c_int]),
    "rms_last_device_status": (c_int, [c_vp]),
    "rms_set_wait_limit": (c_i64, [c_i64]),
    "rms_launch_count": (ctypes.c_uint64, []),
}


def load() -> ctypes.CDLL:
    """The loaded library.  Raises RuntimeError when it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()' or python -m row_wise_normalization_rms_gb300.build); "
                "there is no fallback implementation")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib
