"""Chunked-prefill attention (tcgen05 kernel) and mixed batches on the GPU
against the float64 oracle (pages "Building Kshipra" part 3, section 4:
chunks at absolute positions after the cached prefix, causal mask over the
chunk, online softmax over in-place arena blocks; section 5: mixed steps;
section 3: shared prefix blocks)."""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, custom, random_decode
from workloads import make_config
from workloads.device import DeviceWorkload, bits_of

pytestmark = pytest.mark.gpu


def run(w, max_rows=None, split=None):
    import paged_kv_cache_arena_gb300 as K
    if max_rows is not None:
        K.kshipra_set_option(K.KSHIPRA_OPT_DECODE_MAX_ROWS, max_rows)
    if split is not None:
        K.kshipra_set_option(K.KSHIPRA_OPT_SPLIT_TOKENS, split)
    dw = DeviceWorkload(w)
    dw.step()
    torch.cuda.synchronize()
    return dw


CASES = {
    # one 17-token chunk starting mid-block plus one decode (both kernels)
    "tiny": lambda: make_config("tiny"),
    # chunks spanning several key tiles, ragged query and key tiles
    "g4-multi-tile": lambda: custom(21, prefix=[0, 130, 300], qlen=[200, 77, 129]),
    "g1": lambda: custom(22, Hq=4, Hkv=4, prefix=[5, 250], qlen=[130, 40]),
    "g2-d64": lambda: custom(23, Hq=8, Hkv=4, d=64, prefix=[17, 0], qlen=[100, 65]),
    "g8": lambda: custom(24, Hq=16, Hkv=2, prefix=[33, 400], qlen=[20, 3]),
    "g16-bs32": lambda: custom(25, Hq=32, Hkv=2, bs=32, prefix=[64, 7], qlen=[9, 30]),
    "bf16-bs32": lambda: custom(26, bs=32, dtype="bf16", prefix=[100, 500], qlen=[90, 33]),
    "d64-bf16": lambda: custom(27, Hq=16, Hkv=4, d=64, dtype="bf16", prefix=[129], qlen=[255]),
    "shared-prefix": lambda: custom(28, Hq=8, Hkv=2, prefix=[64, 96, 200], qlen=[40, 1, 70], shared_len=64,
                                    shared=(0, 1, 2)),
    # head_dim 128 with two q heads per kv head: quads of 256 tokens on CTA pairs
    "g2-d128": lambda: custom(35, Hq=8, Hkv=4, prefix=[300, 0, 77], qlen=[260, 513, 31]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(clean_status, name):
    w = CASES[name]()
    dw = run(w)
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype, name)


@pytest.mark.parametrize("name", ["g4-multi-tile", "bf16-bs32", "tiny"])
def test_everything_through_the_prefill_kernel(clean_status, name):
    w = CASES[name]()
    dw = run(w, max_rows=0)  # even single-token sequences on the tensor-core kernel
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype, name)


def test_decode_sequences_on_prefill_kernel(clean_status):
    w = random_decode(29, 6, 1, 700)
    dw = run(w, max_rows=0)
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype)


def test_decode_equals_last_row_of_prefill_across_kernels(clean_status):
    chunk = custom(30, prefix=[100, 37], qlen=[60, 90])
    full = run(chunk).out_f64()
    dec = custom(30, prefix=[100, 37], qlen=[60, 90])
    dec.prefix_lens = chunk.prefix_lens + chunk.query_lens - 1
    dec.query_lens = np.ones_like(chunk.query_lens)
    last = chunk.query_start_loc[1:] - 1
    dec.q = chunk.q[last]
    got = run(dec).out_f64()  # decode kernel
    assert_close(got, full[last], "f16", "decode vs last prefill row")


def test_prefill_block_permutation_gives_identical_bits(clean_status):
    w = custom(31, prefix=[70, 300], qlen=[100, 64], spare=30)
    a = bits_of(run(w).out)
    perm = np.random.default_rng(4).permutation(w.num_blocks).astype(np.int32)
    w.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    assert np.array_equal(a, bits_of(run(w).out))


def test_prefill_shared_prefix_gives_identical_bits(clean_status):
    shared = custom(32, Hq=8, Hkv=2, prefix=[64, 80], qlen=[50, 70], shared_len=64, shared=(0, 1))
    private = custom(32, Hq=8, Hkv=2, prefix=[64, 80], qlen=[50, 70])
    private.q, private.k_all, private.v_all = shared.q, shared.k_all, shared.v_all
    assert np.array_equal(bits_of(run(shared).out), bits_of(run(private).out))


def test_first_chunk_token_sees_only_itself(clean_status):
    w = custom(33, Hq=8, Hkv=2, prefix=[0], qlen=[70])
    dw = run(w)
    got = bits_of(dw.out)[0].reshape(2, 4, -1)
    v0 = bits_of(dw.v_new)[0]
    for g in range(4):
        assert np.array_equal(got[:, g], v0)


@pytest.mark.parametrize("name", ["tiny", "chunked-prefill", "mixed"])
def test_full_config_every_row(clean_status, name):
    # every output row of the full-size workloads against the oracle (the
    # chunks, the decodes of the mixed step, the shared prefix blocks)
    w = make_config(name)
    dw = run(w)
    got = dw.out_f64()
    assert np.all(np.isfinite(got))
    assert_close(got, oracle.workload_attention(w), w.dtype, "full %s (attention)" % name)


def test_long_work_list_planned_on_its_own(clean_status):
    # 1030 short chunks: more work-list entries than the attention kernel
    # plans for itself, so the planning kernel lists them (past its sort
    # capacity in plan order); every row must still be computed once
    S = 1030
    prefix = [(7 * k) % 23 for k in range(S)]
    w = custom(36, Hq=8, Hkv=2, prefix=prefix, qlen=[5] * S)
    dw = run(w)
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype, "1030 chunks")


def test_batched_equals_sequential(clean_status):
    # kshipra-2 section 2's batching check ("batched output equals
    # sequential"): every (sequence, kv head) is computed the same way whatever
    # else is in the batch, so at a fixed split size each sequence's output is
    # bit-identical run alone or batched -- prefill chunks and decode rows
    # mixed, several splits per decode sequence
    from helpers import one_sequence
    w = custom(50, prefix=[0, 130, 300, 700, 45, 2000], qlen=[200, 1, 77, 1, 3, 1])
    batched = bits_of(run(w, split=64).out)
    qsl = w.query_start_loc
    for s in range(w.num_seqs):
        alone = bits_of(run(one_sequence(w, s), split=64).out)
        assert np.array_equal(batched[qsl[s]:qsl[s + 1]], alone), "sequence %d" % s
