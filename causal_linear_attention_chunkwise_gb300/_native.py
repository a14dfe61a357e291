"""ctypes loader for ``_lib/libla_gb300.so`` (the C ABI in ``include/la_gb300.h``).

There is no fallback: if the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libla_gb300.so")

# Symbols the header declares, with (restype, argtypes).
_vp, _i, _u, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
SIGNATURES = {
    "la_set_feature_map": (_i, [_i]),
    "la_get_feature_map": (_i, []),
    "la_chunk_fwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "la_chunk_fwd_kernel_count": (_i, [_i, _i, _i, _i, _i, _i, _i]),
    "la_chunk_fwd": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp,
                          _vp, _sz, _vp]),
    "la_decode_step": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "la_chunk_fwd_noalloc": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp,
                                  _vp, _vp]),
    "la_chunk_fwd_noalloc_prepare": (_i, []),
    "la_chunk_fwd_noalloc_scratch_bytes": (_sz, []),
    "la_noncausal_fwd": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "la_noncausal_fwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "la_normalised_fwd": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp,
                               _vp, _vp, _vp, _vp, _sz, _vp]),
    "la_normalised_fwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "la_channel_gate_fwd": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp,
                                 _vp, _sz, _vp]),
    "la_channel_gate_fwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "la_delta_fwd": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp]),
    "la_device_status": (_i, [_vp]),
    "la_selftest_wait_timeout": (_i, [_u, _vp]),
    "la_last_error": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


class LibraryNotBuilt(RuntimeError):
    pass


def load():
    """Load the library once; raise LibraryNotBuilt if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise LibraryNotBuilt(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m causal_linear_attention_chunkwise_gb300.build` "
                    "(there is no fallback implementation)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
