"""C-ABI checks that need no GPU: exports, host-only entry points, and the
argument validation that must reject bad calls before any CUDA work."""

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kshipra.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_arena_gb300 import _lib
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(kshipra_\w+)\s*\(", text, re.M)))


def test_header_declares_the_binding_exports():
    from paged_kv_cache_arena_gb300 import _lib
    assert declared_symbols() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    from paged_kv_cache_arena_gb300 import _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (kshipra_\w+)", out))
    for name in declared_symbols():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_kv_bytes_per_token_matches_the_pages(lib):
    # kshipra-3 section 1: 128 KiB / 512 KiB per token, 512 MiB vs 2 GiB at 4096 tokens
    rows = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "kv_bytes.txt"))
            if l.strip() and not l.startswith("#")]
    for layers, heads, hd, be, tokens, expected in (map(int, r) for r in rows):
        assert be == 2
        assert lib.kshipra_kv_bytes_per_token(layers, heads, hd, 0) * tokens == expected
        assert lib.kshipra_kv_bytes_per_token(layers, heads, hd, 1) * tokens == expected
    assert lib.kshipra_kv_bytes_per_token(0, 8, 128, 0) == 0
    assert lib.kshipra_kv_bytes_per_token(32, 8, 128, 7) == 0


def test_rope_table_equals_oracle_table(lib, oracle_mod):
    import paged_kv_cache_arena_gb300 as K
    for max_pos, d, theta in [(100, 64, 1.0e4), (5000, 128, 5.0e5), (1, 128, 5.0e5)]:
        got = K.kshipra_rope_table_build(max_pos, d, theta)
        ref = oracle_mod.rope_table(max_pos, d, theta).astype(np.float32)
        assert np.array_equal(got, ref)  # same float64 definition, each entry rounded once to float32


def test_rope_table_rejects_bad_arguments(lib):
    buf = np.zeros(16, dtype=np.float32)
    p = ctypes.c_void_p(buf.ctypes.data)
    assert lib.kshipra_rope_table_build(None, 4, 4, 1e4) == 1
    assert lib.kshipra_rope_table_build(p, -1, 4, 1e4) == 1
    assert lib.kshipra_rope_table_build(p, 4, 3, 1e4) == 1
    assert lib.kshipra_rope_table_build(p, 4, 4, 0.0) == 1
    assert lib.kshipra_rope_table_build(p, 0, 4, 1e4) == 0


class Mem:
    """Real, zero-filled, 256-byte aligned memory for every pointer argument
    of the validation tests: device memory when a GPU is present, so that a
    host check that stopped rejecting would launch on valid buffers (zero
    lengths, block ids and positions) rather than on invented addresses;
    host memory otherwise (without a device no kernel can launch).  Each
    name gets its own buffer of ``SIZE`` bytes, kept for the module."""

    SIZE = 1 << 20

    def __init__(self):
        try:
            import torch
            self.torch = torch if torch.cuda.is_available() else None
        except ImportError:
            self.torch = None
        self.bufs = {}

    def __call__(self, name, offset=0):
        if name not in self.bufs:
            if self.torch is not None:
                t = self.torch.zeros(self.SIZE, dtype=self.torch.uint8, device="cuda")
                base = t.data_ptr()
            else:
                t = np.zeros(self.SIZE + 256, dtype=np.uint8)
                base = (t.ctypes.data + 255) // 256 * 256
            self.bufs[name] = (t, base)
        return ctypes.c_void_p(self.bufs[name][1] + offset)


@pytest.fixture(scope="module")
def mem():
    return Mem()


class Ptr:
    """A pointer argument resolved against ``mem`` when the call is made:
    buffer ``name`` plus ``offset`` bytes."""

    def __init__(self, name, offset=0):
        self.name, self.offset = name, offset


def _resolve(mem, values):
    return [mem(v.name, v.offset) if isinstance(v, Ptr) else v for v in values]


def append_args(mem, **over):
    a = dict(q=Ptr("q"), k=Ptr("k"), v=Ptr("v"), q_rot=Ptr("q_rot"), k_arena=Ptr("k_arena"),
             v_arena=Ptr("v_arena"), bt=Ptr("bt"), qsl=Ptr("qsl"), pos=Ptr("pos"), table=Ptr("table"),
             rope_max_pos=64, num_seqs=1, num_tokens=1, hq=4, hkv=2, d=64, bs=16, maxb=4, nb=16, dtype=0,
             stream=None)
    a.update(over)
    return _resolve(mem, a.values())


@pytest.mark.parametrize("over,code", [
    (dict(num_seqs=-1), 1), (dict(num_tokens=-1), 1), (dict(num_seqs=0), 1), (dict(hq=5), 1), (dict(hkv=0), 1),
    (dict(hq=48, hkv=2), 2), (dict(d=96), 2), (dict(bs=8), 2), (dict(dtype=2), 2), (dict(nb=0), 1),
    (dict(maxb=0), 1), (dict(q=None), 1), (dict(k=None), 1), (dict(bt=None), 1), (dict(table=None), 1),
    (dict(rope_max_pos=0), 1), (dict(k_arena=Ptr("k_arena", 8)), 1),
    (dict(nb=1 << 26, hkv=8, hq=8), 2),
])
def test_append_validation(lib, mem, over, code):
    assert lib.kshipra_kv_append_rope(*append_args(mem, **over)) == code
    assert lib.kshipra_last_error()


def test_append_with_no_tokens_is_a_noop(lib, mem):
    assert lib.kshipra_kv_append_rope(*append_args(mem, num_tokens=0, num_seqs=0)) == 0


def attn_args(mem, **over):
    a = dict(out=Ptr("out"), q_rot=Ptr("q_rot"), k_arena=Ptr("k_arena"), v_arena=Ptr("v_arena"), bt=Ptr("bt"),
             ctx=Ptr("ctx"), qsl=Ptr("qsl"), pos=Ptr("pos"), num_seqs=1, num_tokens=1, max_q=1, max_ctx=10, hq=4,
             hkv=2, d=64, bs=16, maxb=4, nb=16, scale=0.125, dtype=0, ws=Ptr("ws"), ws_bytes=Mem.SIZE,
             stream=None)
    a.update(over)
    return _resolve(mem, a.values())


@pytest.mark.parametrize("over,code", [
    (dict(num_seqs=-1), 1), (dict(num_seqs=0), 1), (dict(max_ctx=0), 1), (dict(max_q=0), 1),
    (dict(max_ctx=65), 1), (dict(hq=6, hkv=4), 1), (dict(hq=24, hkv=1), 2), (dict(d=256), 2), (dict(bs=64), 2),
    (dict(dtype=-1), 2), (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(out=None), 1),
    (dict(ctx=None), 1), (dict(q_rot=Ptr("out")), 1), (dict(v_arena=Ptr("v_arena", 4)), 1),
])
def test_attention_validation(lib, mem, over, code):
    assert lib.kshipra_paged_attention(*attn_args(mem, **over)) == code


def test_attention_with_no_tokens_is_a_noop(lib, mem):
    assert lib.kshipra_paged_attention(*attn_args(mem, num_tokens=0, num_seqs=0)) == 0


def test_workspace_size_host_only(lib):
    import paged_kv_cache_arena_gb300 as K
    r256 = lambda x: -(-x // 256) * 256
    # a short context needs one split: no partials, only the prefill work list
    # (one 8-byte entry per pair of 128-row query tiles per sequence, plus its length)
    items = -(-4 // 64) + 4
    assert K.kshipra_paged_attention_workspace_size(4, 4, 100, 32, 8, 128, sm_count=152) == r256(items * 8 + 4)
    big = K.kshipra_paged_attention_workspace_size(16, 16, 32768, 32, 8, 128, sm_count=152)
    assert big > 0 and big % 256 == 0
    K.kshipra_set_option(K.KSHIPRA_OPT_SPLIT_TOKENS, 1024)
    try:
        ws = K.kshipra_paged_attention_workspace_size(16, 16, 32768, 32, 8, 128, sm_count=152)
        splits = 32
        counters = r256(16 * 8 * 4)  # one finished-split counter per (sequence, kv head)
        items = -(-16 // 64) + 16
        assert ws == (r256(splits * 16 * 32 * 128 * 4) + r256(splits * 16 * 32 * 2 * 4) + counters
                      + r256(items * 8 + 4))
    finally:
        K.kshipra_set_option(K.KSHIPRA_OPT_SPLIT_TOKENS, 0)
    out = ctypes.c_size_t(0)
    assert lib.kshipra_paged_attention_workspace_size(1, 1, 10, 0, 1, 64, 152, ctypes.byref(out)) == 1
    assert lib.kshipra_paged_attention_workspace_size(1, 1, 10, 4, 1, 64, 152, None) == 1


def test_options_validation(lib):
    assert lib.kshipra_set_option(0, 100) == 1
    assert lib.kshipra_set_option(0, -64) == 1
    assert lib.kshipra_set_option(1, 17) == 1
    assert lib.kshipra_set_option(9, 0) == 1
    assert lib.kshipra_set_option(0, 0) == 0
    assert lib.kshipra_set_option(1, 16) == 0


def test_options_belong_to_the_calling_thread(lib):
    # two host threads with different split sizes, querying workspace sizes
    # at the same time, each see only their own setting (ctypes drops the
    # interpreter lock during the calls)
    import threading
    import paged_kv_cache_arena_gb300 as K
    want = {}
    for split in (256, 1024):
        K.kshipra_set_option(K.KSHIPRA_OPT_SPLIT_TOKENS, split)
        want[split] = K.kshipra_paged_attention_workspace_size(16, 16, 32768, 32, 8, 128, sm_count=152)
    K.kshipra_set_option(K.KSHIPRA_OPT_SPLIT_TOKENS, 0)
    auto = K.kshipra_paged_attention_workspace_size(16, 16, 32768, 32, 8, 128, sm_count=152)
    assert len({want[256], want[1024], auto}) == 3
    seen, start = {}, threading.Barrier(2)

    def worker(split):
        K.kshipra_set_option(K.KSHIPRA_OPT_SPLIT_TOKENS, split)
        start.wait()
        seen[split] = {K.kshipra_paged_attention_workspace_size(16, 16, 32768, 32, 8, 128, sm_count=152)
                       for _ in range(2000)}

    threads = [threading.Thread(target=worker, args=(s_,)) for s_ in (256, 1024)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert seen == {256: {want[256]}, 1024: {want[1024]}}
    # this thread's setting was never touched by the workers
    assert K.kshipra_paged_attention_workspace_size(16, 16, 32768, 32, 8, 128, sm_count=152) == auto


def test_status_strings(lib):
    for code in range(5):
        assert lib.kshipra_status_string(code)
    assert lib.kshipra_status_string(99) == b"unknown status"


def step_args(mem, **over):
    a = dict(out=Ptr("out"), q=Ptr("q"), k=Ptr("k"), v=Ptr("v"), q_rot=Ptr("q_rot"), k_arena=Ptr("k_arena"),
             v_arena=Ptr("v_arena"), bt=Ptr("bt"), ctx=Ptr("ctx"), qsl=Ptr("qsl"), pos=Ptr("pos"),
             table=Ptr("table"), rope_max_pos=64, num_seqs=1, num_tokens=1, max_q=1, max_ctx=10, hq=4, hkv=2, d=64,
             bs=16, maxb=4, nb=16, scale=0.125, dtype=0, ws=Ptr("ws"), ws_bytes=Mem.SIZE, stream=None)
    a.update(over)
    return _resolve(mem, a.values())


@pytest.mark.parametrize("over,code", [
    (dict(rope_max_pos=0), 1), (dict(q=None), 1), (dict(table=None), 1), (dict(k=Ptr("k", 8)), 1),
    (dict(dtype=2), 2), (dict(d=96), 2), (dict(hq=6, hkv=4), 1), (dict(q_rot=Ptr("out")), 1),
    # a 40-token chunk (prefill kernel path) with q_rot aliasing q
    (dict(max_q=40, num_tokens=40, q_rot=Ptr("q")), 1),
])
def test_decode_step_validation(lib, mem, over, code):
    assert lib.kshipra_decode_step(*step_args(mem, **over)) == code
    assert lib.kshipra_last_error()


# block moves (copy-on-write copy, swap-out, swap-in): host checks before any launch

def _move_calls(lib, mem, n=1, heads=8, bs=16, d=128, nblocks=64, dtype=0, ids=Ptr("ids"), ka=Ptr("k_arena"),
                va=Ptr("v_arena"), kb=Ptr("k_dense"), vb=Ptr("v_dense"), dst=Ptr("dst_ids")):
    ids, ka, va, kb, vb, dst = _resolve(mem, [ids, ka, va, kb, vb, dst])
    return {
        "copy": lambda: lib.kshipra_blocks_copy(ka, va, ids, dst, n, heads, bs, d, nblocks, dtype, None),
        "swap_out": lambda: lib.kshipra_blocks_swap_out(kb, vb, ka, va, ids, n, heads, bs, d, nblocks, dtype, None),
        "swap_in": lambda: lib.kshipra_blocks_swap_in(ka, va, kb, vb, ids, n, heads, bs, d, nblocks, dtype, None),
    }


@pytest.mark.parametrize("call", ["copy", "swap_out", "swap_in"])
@pytest.mark.parametrize("over, code, why", [
    (dict(n=-1), 1, "negative block count"),
    (dict(heads=0), 1, "bad arena shape"),
    (dict(nblocks=0), 1, "bad arena shape"),
    (dict(d=96), 2, "head_dim 96"),
    (dict(bs=8), 2, "block_size 8"),
    (dict(dtype=7), 2, "dtype 7"),
    (dict(ids=None), 1, "NULL"),                              # id list missing for n > 0
    (dict(ka=None), 1, "a required pointer is NULL"),         # an arena missing
    (dict(va=Ptr("v_arena", 8)), 1, "16-byte aligned"),
])
def test_block_move_validation(lib, mem, call, over, code, why):
    assert _move_calls(lib, mem, **over)[call]() == code
    assert why in lib.kshipra_last_error().decode()  # rejected by that check, before any CUDA call


@pytest.mark.parametrize("call", ["copy", "swap_out", "swap_in"])
def test_block_move_of_nothing_is_a_noop(lib, mem, call):
    assert _move_calls(lib, mem, n=0, ids=None, ka=None, va=None, kb=None, vb=None, dst=None)[call]() == 0
