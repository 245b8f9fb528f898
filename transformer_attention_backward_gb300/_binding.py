"""ctypes declarations of the C ABI in ``include/attn_bwd.h``.

Loading never falls back to anything: if the library is missing it is built
(nvcc for sm_103a), and if that fails the import error propagates.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

OK, EINVAL, ENOTSUP, ECUDA, ETIMEOUT, EWORKSPACE = range(6)
F32, BF16 = 0, 1
STATUS_NAMES = {OK: "ABW_OK", EINVAL: "ABW_EINVAL", ENOTSUP: "ABW_ENOTSUP", ECUDA: "ABW_ECUDA",
                ETIMEOUT: "ABW_ETIMEOUT", EWORKSPACE: "ABW_EWORKSPACE"}

# Every function the header declares, with (restype, argtypes).
_vp, _i, _f, _sz, _ull = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_ulonglong
SIGNATURES = {
    "abw_last_error": (ctypes.c_char_p, []),
    "abw_version": (_i, []),
    "abw_device_check": (_i, [_vp]),
    "abw_set_wait_limit_ns": (None, [_ull]),
    "abw_selftest_wait_timeout": (_i, [_ull, _vp]),
    "softmax_bwd": (_i, [_vp, _vp, _vp, _i, _i, _vp]),
    "rope_bwd": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _i, _f, _i, _vp]),
    "rmsnorm_bwd": (_i, [_vp, _i, _vp, _vp, _vp, _i, _i, _i, _f, _vp]),
    "attn_bwd_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _f, _i, _vp]),
    "rmsnorm_bwd_dgamma": (_i, [_vp, _i, _vp, _vp, _vp, _i, _vp, _i, _i, _f, _vp]),
    "relu2_mul_bwd": (_i, [_vp, _vp, _i, _vp, _vp, _vp, ctypes.c_longlong, _vp]),
    "lora_bwd_workspace_bytes": (_sz, [_i, _i]),
    "lora_bwd": (_i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "attn_fwd_causal": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "attn_bwd_causal_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "attn_bwd_causal": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _f, _i,
                             _vp, _sz, _vp]),
    "attn_bwd_causal_saved_p": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _f, _i,
                                     _vp, _sz, _vp]),
    "attn_bwd_causal_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _f, _i,
                                     _vp]),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_missing else _build.LIB
        if not os.path.exists(path):
            raise ImportError(f"libattnbwd.so not found at {path}")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def last_error() -> str:
    return load().abw_last_error().decode(errors="replace")


class AbwError(RuntimeError):
    def __init__(self, status: int, op: str):
        self.status = status
        super().__init__(f"{op}: {STATUS_NAMES.get(status, status)}: {last_error()}")


def check(status: int, op: str) -> None:
    if status != OK:
        raise AbwError(status, op)
