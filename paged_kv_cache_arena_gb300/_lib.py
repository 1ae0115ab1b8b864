"""ctypes loader for libkshipra.so (the C ABI in include/kshipra.h).

There is no fallback: if the library is missing or fails to load, every call
raises.  Build it with ``paged_kv_cache_arena_gb300.build.build()`` (or the
repository's ``__graft_entry__.build()``).
"""

from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkshipra.so")

# exported symbols, in the order include/kshipra.h declares them
EXPORTS = (
    "kshipra_kv_bytes_per_token",
    "kshipra_rope_table_build",
    "kshipra_kv_append_rope",
    "kshipra_paged_attention_workspace_size",
    "kshipra_paged_attention",
    "kshipra_decode_step",
    "kshipra_paged_attention_noalloc",
    "kshipra_device_status",
    "kshipra_set_option",
    "kshipra_status_string",
    "kshipra_last_error",
)

_lock = threading.Lock()
_lib = None

P, I, D, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_float, ctypes.c_size_t


def load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libkshipra.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        lib.kshipra_kv_bytes_per_token.argtypes = [I, I, I, I]
        lib.kshipra_kv_bytes_per_token.restype = SZ
        lib.kshipra_rope_table_build.argtypes = [P, I, I, D]
        lib.kshipra_kv_append_rope.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, P]
        lib.kshipra_paged_attention_workspace_size.argtypes = [I, I, I, I, I, I, I, ctypes.POINTER(SZ)]
        lib.kshipra_paged_attention.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, I, P, SZ, P]
        lib.kshipra_decode_step.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, I, F, I,
                                            P, SZ, P]
        lib.kshipra_paged_attention_noalloc.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, I,
                                                        P]
        lib.kshipra_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32), P]
        lib.kshipra_set_option.argtypes = [I, I]
        lib.kshipra_status_string.argtypes = [I]
        lib.kshipra_status_string.restype = ctypes.c_char_p
        lib.kshipra_last_error.argtypes = []
        lib.kshipra_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib
