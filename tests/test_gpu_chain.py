"""Calls that follow each other on one stream, each reading what the one
before wrote (the way one layer's attention output feeds the next layer):
every kernel of the library starts as a programmatic dependent of the grid
before it and must still see that grid's writes.  Each chain runs once with
nothing between the calls and once with a device synchronisation between
them; the outputs must be bit-identical."""

import numpy as np
import pytest
import torch

from helpers import custom, random_decode
from workloads.device import DeviceWorkload, bits_of

pytestmark = pytest.mark.gpu


def _attention(K, dw, out, q_rot):
    w = dw.w
    K.kshipra_paged_attention(out, q_rot, dw.k_arena, dw.v_arena, dw.block_tables, dw.context_lens,
                              dw.query_start_loc, dw.positions, w.max_query_len, w.max_context_len, w.scale,
                              dw.workspace)


def _step(K, dw, out, q):
    w = dw.w
    K.kshipra_decode_step(out, q, dw.k_new, dw.v_new, None, dw.k_arena, dw.v_arena, dw.block_tables,
                          dw.context_lens, dw.query_start_loc, dw.positions, dw.rope_table, w.max_query_len,
                          w.max_context_len, w.scale, dw.workspace)


def _chain(K, dw, call, sync, links=4):
    outs = [torch.empty_like(dw.q) for _ in range(links)]
    src = dw.q_rot
    for o in outs:
        call(K, dw, o, src)
        if sync:
            torch.cuda.synchronize()
        src = o
    torch.cuda.synchronize()
    return [bits_of(o) for o in outs]


CASES = {
    "decode": lambda: random_decode(71, 12, 300, 3000),
    "prefill": lambda: custom(72, prefix=[100, 300, 0], qlen=[130, 70, 256]),
    "mixed": lambda: custom(73, prefix=[100, 600, 2000, 40], qlen=[200, 1, 1, 64]),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("call", ["attention", "step"])
def test_each_call_sees_the_previous_output(clean_status, name, call):
    K = clean_status
    fn = _attention if call == "attention" else _step
    dw = DeviceWorkload(CASES[name]())
    dw.append_step()
    torch.cuda.synchronize()
    free = _chain(K, dw, fn, sync=False)
    synced = _chain(K, dw, fn, sync=True)
    for a, b in zip(free, synced):
        assert np.array_equal(a, b)
    # the chain is not trivial: each link changes the values
    assert not np.array_equal(free[0], free[1])


def test_mixed_batches_from_two_host_threads(clean_status):
    # a mixed batch runs its prefill kernel on a side stream of the calling
    # thread; two threads issuing mixed batches on their own streams at once
    # must each get the bits they get alone
    import threading
    ws = [custom(81, prefix=[100, 600, 2000, 40], qlen=[200, 1, 1, 64]),
          custom(82, Hq=16, Hkv=4, prefix=[300, 5, 900, 1500], qlen=[1, 150, 1, 1])]
    dws = [DeviceWorkload(w) for w in ws]
    refs = []
    for dw in dws:
        dw.append_step()
        dw.attention()
        torch.cuda.synchronize()
        refs.append(bits_of(dw.out))
    results = [None, None]
    errors = []

    def run(i):
        try:
            s = torch.cuda.Stream()
            outs = []
            for _ in range(6):
                o = torch.empty_like(dws[i].out)
                dws[i].attention(out=o, stream=s)
                outs.append(o)
            s.synchronize()
            results[i] = [bits_of(o) for o in outs]
        except Exception as exc:  # reported below, on the test's thread
            errors.append(exc)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        for got in results[i]:
            assert np.array_equal(got, refs[i])


@pytest.mark.parametrize("name", ["mixed-config", "custom", "custom-d64"])
def test_mixed_batch_side_by_side_equals_one_after_the_other(clean_status, name):
    # kshipra_paged_attention runs a mixed batch's prefill kernel beside the
    # decode kernel, on a side stream and on part of the SMs; the no-alloc
    # entry point runs the same kernels one after the other on the caller's
    # stream: the outputs must be bit-identical
    from workloads import make_config
    K = clean_status
    # (sizes whose split partials fit the no-alloc scratch)
    if name == "mixed-config":
        w = make_config("mixed")
    else:
        w = custom(83, d=64 if name == "custom-d64" else 128,
                   prefix=[0, 2500] + [(211 * k) % 3000 + 64 for k in range(20)], qlen=[150, 60] + [1, 2] * 10)
    dw = DeviceWorkload(w)
    dw.append_step()
    dw.attention()
    torch.cuda.synchronize()
    side = bits_of(dw.out)
    out = torch.empty_like(dw.out)
    K.kshipra_paged_attention_noalloc(out, dw.q_rot, dw.k_arena, dw.v_arena, dw.block_tables, dw.context_lens,
                                      dw.query_start_loc, dw.positions, w.max_query_len, w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert np.array_equal(side, bits_of(out))
