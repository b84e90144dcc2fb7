"""ctypes declarations of the C ABI in include/attn.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn_gb300.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5
ATTN_ERR_SCRATCH_LIMIT = 6

DTYPE_F16 = 0
DTYPE_BF16 = 1
DTYPE_F32 = 2

PATH_AUTO = 0
PATH_WARP_MMA = 1
PATH_TCGEN05 = 2
PATH_SHORT = 3
PATH_DECODE = 4
PATHS = {"auto": PATH_AUTO, "warp_mma": PATH_WARP_MMA, "tcgen05": PATH_TCGEN05,
         "short": PATH_SHORT, "decode": PATH_DECODE}
DECODE_MAX_ROWS = 16     # query rows per head (after query-group packing) the decoding kernel takes
DECODE_MIN_KEYS = 256    # ATTN_DECODE_MIN_KEYS

_vp, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float


class DebugOpts(ctypes.Structure):
    """attn_debug_opts_t of include/attn.h."""
    _fields_ = [("wait_limit_ns", ctypes.c_uint64), ("inject_missing_arrive", ctypes.c_int)]


# name -> (restype, argtypes); every function include/attn.h declares.
SIGNATURES = {
    "attn_fwd": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp]),
    "attn_fwd_lse": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp]),
    "attn_fwd_path": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "attn_fwd_debug": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i,
                            ctypes.POINTER(DebugOpts), _vp]),
    "attn_auto_path": (_i, [_i, _i]),
    "attn_auto_path_ex": (_i, [_i, _i, _i, _i, _i, _i, _i]),
    "attn_debug_schedule": (_i, [_i, _i, _i, _i, _i, _i, _i, _vp, _i, _vp, _vp, _vp]),
    "attn_status_str": (ctypes.c_char_p, [_i]),
    "attn_read_device_status": (_i, [_vp]),
    "attn_fwd_splitkv": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp,
                              ctypes.c_size_t, _vp]),
    "attn_splitkv_workspace_bytes": (ctypes.c_size_t, [_i, _i, _i, _i, _i]),
    "attn_splitkv_auto_splits": (_i, [_i, _i, _i, _i, _i]),
    "attn_fwd_splitkv_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "attn_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "attn_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "attn_fwd_splitkv_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _i,
                                 _vp, ctypes.c_size_t, _vp]),
    "attn_splitkv_auto_splits_ex": (_i, [_i, _i, _i, _i, _i, _i, _i]),
    "attn_fwd_naive": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp,
                            ctypes.c_size_t, _vp]),
    "attn_naive_workspace_bytes": (ctypes.c_size_t, [_i, _i, _i]),
}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = status_str(status) if _lib is not None else f"status {status}"
        super().__init__(f"{what}: {msg} (status {status})" if what else f"{msg} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded CUDA library. Raises when it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -m exact_scaled_dot_attn_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().attn_status_str(int(status)).decode()
