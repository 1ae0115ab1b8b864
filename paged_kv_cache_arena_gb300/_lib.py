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
    "kshipra_block_pool_create",
    "kshipra_block_pool_destroy",
    "kshipra_block_pool_num_free",
    "kshipra_block_alloc",
    "kshipra_block_share",
    "kshipra_block_release",
    "kshipra_block_refcount",
    "kshipra_block_make_private",
    "kshipra_blocks_copy",
    "kshipra_blocks_swap_out",
    "kshipra_blocks_swap_in",
    "kshipra_prefix_cache_create",
    "kshipra_prefix_cache_destroy",
    "kshipra_prefix_cache_match",
    "kshipra_prefix_cache_insert",
    "kshipra_prefix_cache_evict",
    "kshipra_prefix_cache_evictable",
    "kshipra_prefix_cache_num_nodes",
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
        PI32 = ctypes.POINTER(ctypes.c_int32)
        lib.kshipra_block_pool_create.argtypes = [I, ctypes.POINTER(P)]
        lib.kshipra_block_pool_destroy.argtypes = [P]
        lib.kshipra_block_pool_destroy.restype = None
        lib.kshipra_block_pool_num_free.argtypes = [P]
        lib.kshipra_block_alloc.argtypes = [P, I, PI32]
        lib.kshipra_block_share.argtypes = [P, PI32, I]
        lib.kshipra_block_release.argtypes = [P, PI32, I]
        lib.kshipra_block_refcount.argtypes = [P, I]
        lib.kshipra_block_make_private.argtypes = [P, PI32, PI32]
        lib.kshipra_blocks_copy.argtypes = [P, P, P, P, I, I, I, I, I, I, P]
        lib.kshipra_blocks_swap_out.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P]
        lib.kshipra_blocks_swap_in.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P]
        PI = ctypes.POINTER(I)
        lib.kshipra_prefix_cache_create.argtypes = [P, I, ctypes.POINTER(P)]
        lib.kshipra_prefix_cache_destroy.argtypes = [P]
        lib.kshipra_prefix_cache_destroy.restype = None
        lib.kshipra_prefix_cache_match.argtypes = [P, PI32, I, PI32, I, PI, PI]
        lib.kshipra_prefix_cache_insert.argtypes = [P, PI32, I, PI32, I, PI]
        lib.kshipra_prefix_cache_evict.argtypes = [P, I, PI]
        lib.kshipra_prefix_cache_evictable.argtypes = [P]
        lib.kshipra_prefix_cache_num_nodes.argtypes = [P]
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
