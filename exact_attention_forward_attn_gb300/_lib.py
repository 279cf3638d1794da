"""ctypes loader for the C ABI in ``include/attn.h`` (``_build/libgb300attn.so``).

There is no fallback: if the library has not been built (``build.build()``), loading raises.
With ``ATTN_DEBUG_LIB=1`` in the environment the index-checking debug build
(``_build/libgb300attn_debug.so``, ``build.build(debug=True)``) is loaded instead, for running
the whole test suite under its checks.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import DEBUG_LIB_PATH, LIB_PATH

# Every symbol include/attn.h declares, with its ctypes signature.
_c_int, _c_float, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
SIGNATURES = {
    "attn_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                          _c_float, _vp]),
    "attn_status_string": (ctypes.c_char_p, [_c_int]),
    "attn_last_cuda_error": (_c_int, []),
    "attn_debug_status": (_c_int, [_vp]),
    "attn_fwd_splitkv": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                  _c_int, _c_float, _c_int, _vp, ctypes.c_size_t, _vp]),
    "attn_fwd_splitkv_workspace_bytes": (ctypes.c_size_t, [_c_int, _c_int, _c_int, _c_int,
                                                            _c_int]),
    "attn_fwd_splitkv_num_splits": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "attn_fwd_num_splits": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "attn_fwd_test_split_choice": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                            ctypes.POINTER(_c_int), _c_int, ctypes.c_longlong]),
    "attn_fwd_splitkv_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                          _c_int, _c_int, _c_int, _c_float, _c_int, _vp]),
    "attn_fwd_splitkv_noalloc_max_bytes": (ctypes.c_size_t, []),
    "attn_fwd_test_stall": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                     _c_int, _c_int, _c_float, _c_int, _vp]),
    "attn_fwd_test_kernel": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                      _c_int, _c_int, _c_float, _c_int, _c_int, _vp]),
    "attn_bwd": (_c_int, [_vp] * 9 + [_c_int] * 6 + [_c_float, _vp, ctypes.c_size_t, _vp]),
    "attn_bwd_workspace_bytes": (ctypes.c_size_t, [_c_int, _c_int, _c_int]),
    "attn_fwd_strided": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                  _c_int, _c_float, _vp, _vp, _vp, _vp, _vp]),
    "attn_mla_decode": (_c_int, [_vp, _vp, _vp, _vp] + [_c_int] * 5 + [_c_float, _c_int, _vp,
                                                                      ctypes.c_size_t, _vp]),
    "attn_mla_decode_test_stall": (_c_int, [_vp, _vp, _vp, _vp] + [_c_int] * 5
                                   + [_c_float, _c_int, _vp, ctypes.c_size_t, _c_int, _vp]),
    "attn_mla_decode_num_splits": (_c_int, [_c_int, _c_int, _c_int]),
    "attn_mla_decode_workspace_bytes": (ctypes.c_size_t, [_c_int, _c_int, _c_int, _c_int]),
}

_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Load the built library once and attach the signatures of every exported function."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or (DEBUG_LIB_PATH if os.environ.get("ATTN_DEBUG_LIB") == "1" else LIB_PATH)
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library not found at {p}; build it first "
                "(python -m exact_attention_forward_attn_gb300.build or __graft_entry__.build())")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib
