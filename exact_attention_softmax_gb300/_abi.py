"""ctypes view of the C ABI in ``include/sdpa.h`` (``libsdpa_gb300.so``).

Argument marshalling only: every step of the attention computation runs in
the library's CUDA kernels. If the library is missing this module raises;
there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

SDPA_F32, SDPA_F16, SDPA_BF16 = 0, 1, 2
SDPA_OK = 0
SDPA_ERR_ARG = -1
SDPA_ERR_UNSUPPORTED = -2
SDPA_ERR_CUDA = -3
SDPA_ERR_TIMEOUT = -4
SDPA_ERR_WORKSPACE = -5
SDPA_ERR_BOUNDS = -6
SDPA_STATUS_TIMEOUT = 1
SDPA_STATUS_SEQLEN = 2
SDPA_STATUS_BOUNDS = 4

# Another build of the library (e.g. the debug build,
# ``lib/libsdpa_gb300_debug.so``) is loaded instead when this names it.
LIB_ENV = "SDPA_GB300_LIB"

# Every entry point the header declares, with its ctypes signature.
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "sdpa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "sdpa_fwd_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _vp, _i, _vp]),
    "sdpa_fwd_strided": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "sdpa_bwd_strided": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                              _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _sz, _vp]),
    "sdpa_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "sdpa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                      _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _sz, _vp]),
    "sdpa_bwd_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                             _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _vp, _i, _vp, _sz, _vp]),
    "sdpa_fwd_blocksparse": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i,
                                  _vp, ctypes.c_longlong, ctypes.c_longlong, _i, _i, _vp]),
    "sdpa_bwd_blocksparse": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i,
                                  _vp, ctypes.c_longlong, ctypes.c_longlong, _i, _i, _vp, _sz, _vp]),
    "sdpa_fwd_masked": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i,
                             _vp, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong, _i, _vp]),
    "sdpa_bwd_masked": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i,
                             _vp, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong, _i, _vp, _sz, _vp]),
    "sdpa_fwd_dropout": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _f, ctypes.c_ulonglong, _i, _vp]),
    "sdpa_bwd_dropout": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i,
                              _f, ctypes.c_ulonglong, _i, _vp, _sz, _vp]),
    "sdpa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                              _i, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "sdpa_device_status": (_i, [_vp, ctypes.POINTER(ctypes.c_uint)]),
    "sdpa_trace_events": (_i, [_i, _vp, _vp]),
    "sdpa_debug_set": (_i, [_i]),
    "sdpa_last_error": (ctypes.c_char_p, []),
    "sdpa_version": (_i, []),
    "sdpa_debug_build": (_i, []),
}

_lib = None


def load(path: str | None = None):
    """Load the library once (raises RuntimeError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get(LIB_ENV) or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m exact_attention_softmax_gb300.build` "
            "(the attention ops have no non-CUDA implementation)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class SdpaError(RuntimeError):
    """A nonzero return from the C ABI (message from sdpa_last_error)."""

    def __init__(self, code: int, msg: str):
        super().__init__(f"sdpa error {code}: {msg}")
        self.code = code


def check(rc: int):
    if rc != SDPA_OK:
        raise SdpaError(rc, load().sdpa_last_error().decode())
    return rc
