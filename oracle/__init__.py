"""Float64 CPU oracle for paged GQA attention over a block arena.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.
The CUDA library never calls it and shares no code with it.

``oracle.c`` holds the arithmetic (IEEE conversions, RoPE, arena placement,
dense masked softmax attention); this module compiles it with gcc on first
use and wraps it with ctypes.  ``brute.py`` is an independent pure-Python
restatement for tiny inputs that pins the C code.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1
DTYPE = {"f16": F16, "bf16": BF16, F16: F16, BF16: BF16}


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def open_library(path: str):
    """ctypes handle of a compiled oracle (``liboracle.so``, or a copy built
    from a modified source by the tests that plant mistakes in it)."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I, L, D = ctypes.c_int, ctypes.c_long, ctypes.c_double
    lib.oracle_rope_table.argtypes = [P, I, I, D]
    lib.oracle_rope_rows.argtypes = [P, P, P, L, I, I, D, I]
    lib.oracle_arena_image.argtypes = [P, P, P, P, P, P, I, P, I, I, I, I, I, D, I]
    lib.oracle_attention.argtypes = [P, P, I, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, D, D, I, I]
    lib.oracle_decode_bits.argtypes = [P, P, L, I]
    lib.oracle_encode_bits.argtypes = [P, P, L, I]
    lib.oracle_default_threads.restype = I
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None and a.size else ctypes.c_void_p(0)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def bits_to_f64(bits, dtype) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode_bits(_p(b), _p(out), b.size, DTYPE[dtype])
    return out


def f64_to_bits(x, dtype) -> np.ndarray:
    a = _c(x, np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_encode_bits(_p(a), _p(out), a.size, DTYPE[dtype])
    return out


def rope_table(max_pos: int, head_dim: int, theta: float) -> np.ndarray:
    """(cos, sin) of position * theta^(-2i/d), shape [max_pos, d/2, 2]."""
    out = np.empty((max_pos, head_dim // 2, 2), dtype=np.float64)
    rc = _load().oracle_rope_table(_p(out), max_pos, head_dim, float(theta))
    if rc:
        raise ValueError("oracle_rope_table failed (%d)" % rc)
    return out


def rope_rows(rows, positions, theta: float, dtype) -> np.ndarray:
    """Rotated rows [n, H, d] at ``positions``, rounded once to ``dtype`` bits."""
    r = _c(rows, np.uint16)
    pos = _c(positions, np.int32)
    n, H, d = r.shape
    out = np.empty_like(r)
    rc = _load().oracle_rope_rows(_p(r), _p(out), _p(pos), n, H, d, float(theta), DTYPE[dtype])
    if rc:
        raise ValueError("oracle_rope_rows failed (%d)" % rc)
    return out


def arena_image(k_arena, v_arena, k_rows, v_rows, query_start_loc, positions, block_tables,
                num_blocks: int, block_size: int, theta: float, dtype) -> None:
    """Write the expected arena contents (in place) after appending the rows.

    Arenas are ``[num_blocks, Hkv, bs, d]`` uint16 arrays pre-filled by the
    caller; slots no row maps to are left untouched.
    """
    kr, vr = _c(k_rows, np.uint16), _c(v_rows, np.uint16)
    qsl, pos = _c(query_start_loc, np.int32), _c(positions, np.int32)
    bt = _c(block_tables, np.int32)
    assert k_arena.flags.c_contiguous and v_arena.flags.c_contiguous
    Hkv, d = k_arena.shape[1], k_arena.shape[3]
    rc = _load().oracle_arena_image(_p(k_arena), _p(v_arena), _p(kr), _p(vr), _p(qsl), _p(pos), len(qsl) - 1,
                                    _p(bt), bt.shape[1], num_blocks, Hkv, block_size, d, float(theta),
                                    DTYPE[dtype])
    if rc:
        raise ValueError("oracle_arena_image failed (%d)" % rc)


def attention(q, k_all, v_all, kv_start, query_start_loc, positions, context_lens, num_kv_heads: int,
              theta: float, scale: float, dtype, tokens=None, nthreads: int = 0, block_tables=None,
              block_size: int = 0, num_blocks: int = 0) -> np.ndarray:
    """Dense masked softmax attention in float64.

    With ``block_tables`` the keys and values are written into the oracle's
    own arena of ``num_blocks`` blocks of ``block_size`` slots through the
    tables and gathered back through them (a gathered NaN, an aliased slot or
    a block id outside the arena raises); without, they are read in logical
    order.  Returns ``[len(tokens), Hq, d]`` (all tokens when ``tokens`` is
    None).
    """
    qq = _c(q, np.uint16)
    T, Hq, d = qq.shape
    ka, va = _c(k_all, np.uint16), _c(v_all, np.uint16)
    ks = _c(kv_start, np.int64)
    qsl, pos, ctx = _c(query_start_loc, np.int32), _c(positions, np.int32), _c(context_lens, np.int32)
    toks = None if tokens is None else _c(tokens, np.int32)
    bt = None if block_tables is None else _c(block_tables, np.int32)
    n_out = T if toks is None else len(toks)
    out = np.zeros((n_out, Hq, d), dtype=np.float64)
    rc = _load().oracle_attention(_p(out), _p(toks) if toks is not None else ctypes.c_void_p(0), n_out, _p(qq),
                                  _p(ka), _p(va), _p(ks), _p(qsl), _p(pos), _p(ctx),
                                  _p(bt) if bt is not None else ctypes.c_void_p(0),
                                  bt.shape[1] if bt is not None else 0, int(block_size), int(num_blocks),
                                  len(qsl) - 1, T, Hq, num_kv_heads, d, float(theta), float(scale), DTYPE[dtype],
                                  int(nthreads))
    if rc:
        raise ValueError("oracle_attention failed (%d: %s)" % (rc, _ATTN_ERRORS.get(rc, "?")))
    return out


_ATTN_ERRORS = {1: "bad shape", 2: "block id outside the arena", 3: "out of memory",
                4: "position outside the context", 5: "two different rows written to one arena slot",
                6: "a NaN was gathered"}


# ---- conveniences over a generated workload (duck-typed) -----------------

def workload_attention(w, tokens=None, nthreads: int = 0, gather: bool = True) -> np.ndarray:
    """Attention of a workload's query tokens, keys and values through the
    oracle's own block arena (``gather=False``: in logical order)."""
    bt = dict(block_tables=w.block_tables, block_size=w.block_size, num_blocks=w.num_blocks) if gather else {}
    return attention(w.q, w.k_all, w.v_all, w.kv_start, w.query_start_loc, w.positions, w.context_lens,
                     w.num_kv_heads, w.theta, w.scale, w.dtype, tokens=tokens, nthreads=nthreads, **bt)


def workload_arena(w, sentinel: int, include_prefix: bool = True, include_step: bool = True):
    """Expected (k_arena, v_arena) after the prefix append and the step append."""
    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    ka = np.full(shape, sentinel, dtype=np.uint16)
    va = np.full(shape, sentinel, dtype=np.uint16)
    if include_prefix:
        kp, vp, qsl_p, pos_p = w.prefix_batch()
        arena_image(ka, va, kp, vp, qsl_p, pos_p, w.block_tables, w.num_blocks, w.block_size, w.theta, w.dtype)
    if include_step:
        kn, vn = w.step_kv()
        arena_image(ka, va, kn, vn, w.query_start_loc, w.positions, w.block_tables, w.num_blocks,
                    w.block_size, w.theta, w.dtype)
    return ka, va


def workload_q_rot(w) -> np.ndarray:
    return rope_rows(w.q, w.positions, w.theta, w.dtype)
