"""Paged GQA attention over a block-arena KV cache, for GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/kshipra.h``: each function has
the C entry point's name, takes torch tensors for the device buffers, reads
sizes off their shapes and passes raw pointers through ctypes.  All
arithmetic runs in the library's CUDA kernels; nothing here computes.

Pages "Building Kshipra" part 3 (kshipra-3): section 1 (block arena, KV bytes
per token), section 4 (RoPE at absolute positions, online-softmax attention
over in-place arena blocks, causal mask over the chunk), section 5 (mixed
prefill/decode batches).
"""

from __future__ import annotations

import ctypes

import numpy as np

from . import _lib

KSHIPRA_OK = 0
KSHIPRA_ERR_INVALID_ARG = 1
KSHIPRA_ERR_UNSUPPORTED = 2
KSHIPRA_ERR_WORKSPACE_TOO_SMALL = 3
KSHIPRA_ERR_CUDA = 4
KSHIPRA_ERR_OUT_OF_BLOCKS = 5

KSHIPRA_DEV_BAD_BLOCK_ID = 0x1
KSHIPRA_DEV_BAD_POSITION = 0x2
KSHIPRA_DEV_BAD_LENGTHS = 0x4
KSHIPRA_DEV_TIMEOUT = 0x8

KSHIPRA_DTYPE_F16 = 0
KSHIPRA_DTYPE_BF16 = 1

KSHIPRA_OPT_SPLIT_TOKENS = 0
KSHIPRA_OPT_DECODE_MAX_ROWS = 1


class KshipraError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = _lib.load()
        msg = lib.kshipra_last_error().decode() or lib.kshipra_status_string(code).decode()
        super().__init__("%s: %s (status %d)" % (where, msg, code))
        self.code = code


def _check(code: int, where: str) -> None:
    if code != KSHIPRA_OK:
        raise KshipraError(code, where)


def _ptr(t) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return KSHIPRA_DTYPE_F16
    if t.dtype == torch.bfloat16:
        return KSHIPRA_DTYPE_BF16
    raise ValueError("unsupported tensor dtype %s" % t.dtype)


def kshipra_kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, dtype: int) -> int:
    return int(_lib.load().kshipra_kv_bytes_per_token(num_layers, num_kv_heads, head_dim, dtype))


def kshipra_rope_table_build(max_pos: int, head_dim: int, theta: float) -> np.ndarray:
    """Host float32 table [max_pos, head_dim/2, 2] of (cos, sin)."""
    out = np.empty((max_pos, head_dim // 2, 2), dtype=np.float32)
    _check(_lib.load().kshipra_rope_table_build(ctypes.c_void_p(out.ctypes.data), max_pos, head_dim, float(theta)),
           "kshipra_rope_table_build")
    return out


def kshipra_kv_append_rope(q, k, v, q_rot, k_arena, v_arena, block_tables, query_start_loc, positions,
                           rope_table, stream=None) -> None:
    """q/q_rot may be None (prefix fill).  Shapes as in include/kshipra.h."""
    num_tokens, num_kv_heads, head_dim = k.shape
    num_q_heads = q.shape[1] if q is not None else num_kv_heads
    num_blocks, _, block_size, _ = k_arena.shape
    _check(_lib.load().kshipra_kv_append_rope(
        _ptr(q), _ptr(k), _ptr(v), _ptr(q_rot), _ptr(k_arena), _ptr(v_arena), _ptr(block_tables),
        _ptr(query_start_loc), _ptr(positions), _ptr(rope_table), rope_table.shape[0],
        query_start_loc.shape[0] - 1, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
        block_tables.shape[1], num_blocks, _dtype_code(k), _stream(stream)), "kshipra_kv_append_rope")


class BlockPool:
    """The library's LIFO block pool (host state; see include/kshipra.h)."""

    def __init__(self, num_blocks: int):
        lib = _lib.load()
        h = ctypes.c_void_p(0)
        _check(lib.kshipra_block_pool_create(num_blocks, ctypes.byref(h)), "kshipra_block_pool_create")
        self._h = h
        self.num_blocks = num_blocks

    def close(self) -> None:
        if self._h:
            _lib.load().kshipra_block_pool_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def num_free(self) -> int:
        return _lib.load().kshipra_block_pool_num_free(self._h)

    @staticmethod
    def _ids(ids):
        arr = (ctypes.c_int32 * len(ids))(*[int(i) for i in ids])
        return arr, len(ids)

    def alloc(self, n: int) -> list:
        arr = (ctypes.c_int32 * max(n, 1))()
        _check(_lib.load().kshipra_block_alloc(self._h, n, arr), "kshipra_block_alloc")
        return [int(arr[i]) for i in range(n)]

    def share(self, ids) -> None:
        arr, n = self._ids(ids)
        _check(_lib.load().kshipra_block_share(self._h, arr, n), "kshipra_block_share")

    def release(self, ids) -> None:
        arr, n = self._ids(ids)
        _check(_lib.load().kshipra_block_release(self._h, arr, n), "kshipra_block_release")

    def refcount(self, block_id: int) -> int:
        return _lib.load().kshipra_block_refcount(self._h, int(block_id))

    def make_private(self, block_id: int):
        """(id to write into, id to copy from or -1)."""
        bid, src = ctypes.c_int32(int(block_id)), ctypes.c_int32(0)
        _check(_lib.load().kshipra_block_make_private(self._h, ctypes.byref(bid), ctypes.byref(src)),
               "kshipra_block_make_private")
        return int(bid.value), int(src.value)


def _arena_shape(k_arena):
    num_blocks, num_kv_heads, block_size, head_dim = k_arena.shape
    return num_kv_heads, block_size, head_dim, num_blocks


def kshipra_blocks_copy(k_arena, v_arena, src_ids, dst_ids, stream=None) -> None:
    hk, bs, d, nb = _arena_shape(k_arena)
    _check(_lib.load().kshipra_blocks_copy(_ptr(k_arena), _ptr(v_arena), _ptr(src_ids), _ptr(dst_ids),
                                           src_ids.numel(), hk, bs, d, nb, _dtype_code(k_arena), _stream(stream)),
           "kshipra_blocks_copy")


def kshipra_blocks_swap_out(k_out, v_out, k_arena, v_arena, ids, stream=None) -> None:
    hk, bs, d, nb = _arena_shape(k_arena)
    _check(_lib.load().kshipra_blocks_swap_out(_ptr(k_out), _ptr(v_out), _ptr(k_arena), _ptr(v_arena), _ptr(ids),
                                               ids.numel(), hk, bs, d, nb, _dtype_code(k_arena), _stream(stream)),
           "kshipra_blocks_swap_out")


def kshipra_blocks_swap_in(k_arena, v_arena, k_in, v_in, ids, stream=None) -> None:
    hk, bs, d, nb = _arena_shape(k_arena)
    _check(_lib.load().kshipra_blocks_swap_in(_ptr(k_arena), _ptr(v_arena), _ptr(k_in), _ptr(v_in), _ptr(ids),
                                              ids.numel(), hk, bs, d, nb, _dtype_code(k_arena), _stream(stream)),
           "kshipra_blocks_swap_in")


class PrefixCache:
    """The library's radix-tree prefix cache over a BlockPool (host state; see
    include/kshipra.h).  Close it before the pool."""

    def __init__(self, pool: BlockPool, block_size: int):
        h = ctypes.c_void_p(0)
        _check(_lib.load().kshipra_prefix_cache_create(pool._h, block_size, ctypes.byref(h)),
               "kshipra_prefix_cache_create")
        self._h = h
        self.pool = pool  # keeps the pool alive
        self.block_size = block_size

    def close(self) -> None:
        if self._h:
            _lib.load().kshipra_prefix_cache_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _tokens(tokens):
        n = len(tokens)
        return (ctypes.c_int32 * max(n, 1))(*[int(t) for t in tokens]), n

    def match(self, tokens):
        """(blocks, matched token count); the caller holds one reference to
        each returned block."""
        arr, n = self._tokens(tokens)
        cap = -(-n // self.block_size)
        out = (ctypes.c_int32 * max(cap, 1))()
        nb, nt = ctypes.c_int(0), ctypes.c_int(0)
        _check(_lib.load().kshipra_prefix_cache_match(self._h, arr, n, out, cap, ctypes.byref(nb), ctypes.byref(nt)),
               "kshipra_prefix_cache_match")
        return [int(out[i]) for i in range(nb.value)], int(nt.value)

    def insert(self, tokens, blocks) -> int:
        """Caches the full blocks of tokens; returns how many were added."""
        arr, n = self._tokens(tokens)
        ids = (ctypes.c_int32 * max(len(blocks), 1))(*[int(b) for b in blocks])
        added = ctypes.c_int(0)
        _check(_lib.load().kshipra_prefix_cache_insert(self._h, arr, n, ids, len(blocks), ctypes.byref(added)),
               "kshipra_prefix_cache_insert")
        return int(added.value)

    def evict(self, num_blocks: int) -> int:
        freed = ctypes.c_int(0)
        _check(_lib.load().kshipra_prefix_cache_evict(self._h, num_blocks, ctypes.byref(freed)),
               "kshipra_prefix_cache_evict")
        return int(freed.value)

    @property
    def evictable(self) -> int:
        return _lib.load().kshipra_prefix_cache_evictable(self._h)

    @property
    def num_nodes(self) -> int:
        return _lib.load().kshipra_prefix_cache_num_nodes(self._h)


def kshipra_paged_attention_workspace_size(num_seqs: int, num_tokens: int, max_context_len: int,
                                           num_q_heads: int, num_kv_heads: int, head_dim: int,
                                           sm_count: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.load().kshipra_paged_attention_workspace_size(num_seqs, num_tokens, max_context_len, num_q_heads,
                                                              num_kv_heads, head_dim, sm_count, ctypes.byref(out)),
           "kshipra_paged_attention_workspace_size")
    return int(out.value)


def kshipra_paged_attention(out, q_rot, k_arena, v_arena, block_tables, context_lens, query_start_loc, positions,
                            max_query_len: int, max_context_len: int, scale: float, workspace=None,
                            stream=None) -> None:
    num_tokens, num_q_heads, head_dim = q_rot.shape
    num_blocks, num_kv_heads, block_size, _ = k_arena.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.load().kshipra_paged_attention(
        _ptr(out), _ptr(q_rot), _ptr(k_arena), _ptr(v_arena), _ptr(block_tables), _ptr(context_lens),
        _ptr(query_start_loc), _ptr(positions), query_start_loc.shape[0] - 1, num_tokens, max_query_len,
        max_context_len, num_q_heads, num_kv_heads, head_dim, block_size, block_tables.shape[1], num_blocks,
        float(scale), _dtype_code(q_rot), _ptr(workspace), ws_bytes, _stream(stream)), "kshipra_paged_attention")


def kshipra_decode_step(out, q, k, v, q_rot, k_arena, v_arena, block_tables, context_lens, query_start_loc,
                        positions, rope_table, max_query_len: int, max_context_len: int, scale: float,
                        workspace=None, stream=None) -> None:
    """RoPE-and-append then attention: one launch for decode-class batches,
    otherwise a K/V append and attention kernels that rotate q themselves;
    q_rot may be None.  Shapes as in include/kshipra.h."""
    num_tokens, num_q_heads, head_dim = q.shape
    num_blocks, num_kv_heads, block_size, _ = k_arena.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.load().kshipra_decode_step(
        _ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(q_rot), _ptr(k_arena), _ptr(v_arena), _ptr(block_tables),
        _ptr(context_lens), _ptr(query_start_loc), _ptr(positions), _ptr(rope_table), rope_table.shape[0],
        query_start_loc.shape[0] - 1, num_tokens, max_query_len, max_context_len, num_q_heads, num_kv_heads,
        head_dim, block_size, block_tables.shape[1], num_blocks, float(scale), _dtype_code(q), _ptr(workspace),
        ws_bytes, _stream(stream)), "kshipra_decode_step")


def kshipra_paged_attention_noalloc(out, q_rot, k_arena, v_arena, block_tables, context_lens, query_start_loc,
                                    positions, max_query_len: int, max_context_len: int, scale: float,
                                    stream=None) -> None:
    """kshipra_paged_attention without a workspace, for callers that can't
    allocate device memory; uses the library's fixed scratch array (calls
    that overlap on the GPU race)."""
    num_tokens, num_q_heads, head_dim = q_rot.shape
    num_blocks, num_kv_heads, block_size, _ = k_arena.shape
    _check(_lib.load().kshipra_paged_attention_noalloc(
        _ptr(out), _ptr(q_rot), _ptr(k_arena), _ptr(v_arena), _ptr(block_tables), _ptr(context_lens),
        _ptr(query_start_loc), _ptr(positions), query_start_loc.shape[0] - 1, num_tokens, max_query_len,
        max_context_len, num_q_heads, num_kv_heads, head_dim, block_size, block_tables.shape[1], num_blocks,
        float(scale), _dtype_code(q_rot), _stream(stream)), "kshipra_paged_attention_noalloc")


def kshipra_device_status(stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(_lib.load().kshipra_device_status(ctypes.byref(code), _stream(stream)), "kshipra_device_status")
    return int(code.value)


def kshipra_set_option(option: int, value: int) -> None:
    _check(_lib.load().kshipra_set_option(option, value), "kshipra_set_option")
