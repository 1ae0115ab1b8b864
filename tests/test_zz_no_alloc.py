"""kshipra_paged_attention_noalloc: the entry point for callers that can't
allocate device memory (for example a server whose KV arena already holds all
free device memory, or a framework whose allocator owns every device byte).

It must give the same results as kshipra_paged_attention with a caller
workspace, call after call, although all calls share one fixed scratch array
inside the library.  Named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from helpers import assert_close, random_decode
from workloads.device import DeviceWorkload, bits_of

pytestmark = pytest.mark.gpu


def _args(dw, out):
    w = dw.w
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return [p(out), p(dw.q_rot), p(dw.k_arena), p(dw.v_arena), p(dw.block_tables), p(dw.context_lens),
            p(dw.query_start_loc), p(dw.positions), w.num_seqs, w.num_tokens, w.max_query_len, w.max_context_len,
            w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.max_blocks_per_seq, w.num_blocks,
            ctypes.c_float(w.scale), w.dtype_code]


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(clean_status):
    K = clean_status
    lib = K._lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # small splits so that every sequence spreads its keys over several
    # partials in the scratch array
    K.kshipra_set_option(K.KSHIPRA_OPT_SPLIT_TOKENS, 128)
    cases = [random_decode(31, 6, 300, 2000), random_decode(32, 5, 500, 3000, bs=32, dtype="bf16")]
    dws, refs = [], []
    for w in cases:
        dw = DeviceWorkload(w)
        dw.append_step()
        ws = torch.empty(max(dw.ws_bytes, 256), dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(dw.q)
        assert dw.ws_bytes > 0
        rc = lib.kshipra_paged_attention(*_args(dw, ref), ctypes.c_void_p(ws.data_ptr()), ws.numel(), stream)
        assert rc == 0, lib.kshipra_last_error()
        dws.append(dw)
        refs.append(ref)
    outs = [torch.full_like(r, float("nan")) for r in refs]
    for dw, out in zip(dws, outs):  # two calls in a row, sharing the scratch
        rc = lib.kshipra_paged_attention_noalloc(*_args(dw, out), stream)
        assert rc == 0, lib.kshipra_last_error()
    torch.cuda.synchronize()
    for w, ref, out in zip(cases, refs, outs):
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        assert_close(got, want, w.dtype, "noalloc vs workspace entry point")
        assert np.array_equal(bits_of(out), bits_of(ref))


def test_noalloc_rejects_sizes_beyond_its_scratch(clean_status):
    K = clean_status
    lib = K._lib.load()
    K.kshipra_set_option(K.KSHIPRA_OPT_SPLIT_TOKENS, 64)
    S, ctx, hq, hkv, d, bs = 64, 4096, 32, 8, 128, 16
    need = K.kshipra_paged_attention_workspace_size(S, S, ctx, hq, hkv, d)
    assert need > 16 << 20
    # real, zero-filled buffers of the sizes the call names: were the size
    # check ever to let this call through, its kernels would read and write
    # valid memory only (zero lengths, block 0)
    nb, maxb = 256, ctx // bs
    dev = lambda shape, dt: torch.zeros(shape, dtype=dt, device="cuda")
    out, q_rot = dev((S, hq, d), torch.float16), dev((S, hq, d), torch.float16)
    ka, va = dev((nb, hkv, bs, d), torch.float16), dev((nb, hkv, bs, d), torch.float16)
    bt, ctx_lens = dev((S, maxb), torch.int32), dev((S,), torch.int32)
    qsl, pos = dev((S + 1,), torch.int32), dev((S,), torch.int32)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.kshipra_paged_attention_noalloc(p(out), p(q_rot), p(ka), p(va), p(bt), p(ctx_lens), p(qsl), p(pos), S, S,
                                             1, ctx, hq, hkv, d, bs, maxb, nb, ctypes.c_float(d ** -0.5), 0, None)
    assert rc == K.KSHIPRA_ERR_WORKSPACE_TOO_SMALL
    assert b"workspace" in lib.kshipra_last_error()
