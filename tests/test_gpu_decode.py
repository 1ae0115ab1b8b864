"""Split-KV decode attention on the GPU against the float64 oracle (pages
"Building Kshipra" part 3, section 4: online softmax over in-place arena
blocks; section 1: blocks reached through block tables)."""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, custom, random_decode
from workloads import make_config
from workloads.device import DeviceWorkload, bits_of

pytestmark = pytest.mark.gpu


def run(w, K=None, split=None, max_rows=None):
    import paged_kv_cache_arena_gb300 as KK
    if split is not None:
        KK.kshipra_set_option(KK.KSHIPRA_OPT_SPLIT_TOKENS, split)
    if max_rows is not None:
        KK.kshipra_set_option(KK.KSHIPRA_OPT_DECODE_MAX_ROWS, max_rows)
    dw = DeviceWorkload(w)
    dw.step()
    torch.cuda.synchronize()
    return dw


CASES = {
    # several 16-key chunks per warp, ragged tails, several splits
    "llama-shape": lambda: random_decode(1, 8, 17, 700),
    "bs32-bf16": lambda: random_decode(2, 6, 1, 900, bs=32, dtype="bf16"),
    "d64": lambda: random_decode(3, 5, 30, 500, Hq=16, Hkv=4, d=64),
    "g1": lambda: random_decode(4, 4, 100, 400, Hq=8, Hkv=8),
    "g2": lambda: random_decode(5, 4, 100, 400, Hq=8, Hkv=4),
    "g8": lambda: random_decode(6, 4, 100, 400, Hq=16, Hkv=2),
    "g16": lambda: random_decode(7, 3, 100, 400, Hq=32, Hkv=2, bs=32),
    # several query tokens per sequence that still fit the decode kernel
    "qlen2-g4": lambda: custom(8, prefix=[50, 300, 0], qlen=[2, 4, 3]),
    "qlen2-g8-bf16": lambda: custom(9, Hq=16, Hkv=2, dtype="bf16", prefix=[77, 5], qlen=[2, 2]),
    "ctx1": lambda: custom(10, prefix=[0, 0, 1], qlen=[1, 1, 1]),
}


@pytest.mark.parametrize("split", [None, 64, 192])
@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_matches_oracle(clean_status, name, split):
    w = CASES[name]()
    dw = run(w, split=split)
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype, name)


def test_single_key_returns_its_value_exactly(clean_status):
    w = custom(11, Hq=8, Hkv=2, prefix=[0, 0], qlen=[1, 1])
    dw = run(w)
    v0 = bits_of(dw.v_new)  # the only key of each sequence is the new token
    got = bits_of(dw.out).reshape(2, 2, 4, -1)
    for s in range(2):
        for g in range(4):
            assert np.array_equal(got[s, :, g], v0[s])


def test_block_permutation_gives_identical_bits(clean_status):
    w = random_decode(12, 6, 40, 600, spare=20)
    a = bits_of(run(w).out)
    perm = np.random.default_rng(3).permutation(w.num_blocks).astype(np.int32)
    w.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    b = bits_of(run(w).out)
    assert np.array_equal(a, b)


def test_shared_prefix_blocks_give_identical_bits(clean_status):
    shared = custom(13, prefix=[128, 200, 300], qlen=[1, 1, 1], shared_len=128, shared=(0, 1, 2))
    private = custom(13, prefix=[128, 200, 300], qlen=[1, 1, 1])
    private.q, private.k_all, private.v_all = shared.q, shared.k_all, shared.v_all
    assert np.array_equal(bits_of(run(shared).out), bits_of(run(private).out))


def test_nan_in_unused_slots_never_reaches_the_output(clean_status):
    # contexts ending mid-block leave NaN-filled slots in their last block
    w = random_decode(14, 8, 1, 64)
    dw = run(w)
    assert np.all(np.isfinite(dw.out_f64()))
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype)


@pytest.mark.parametrize("name", ["llama-decode", "long-decode"])
def test_full_decode_config_every_row(clean_status, name):
    # every output row of the full-size decode workloads against the oracle
    w = make_config(name)
    dw = run(w)
    got = dw.out_f64()
    assert np.all(np.isfinite(got))
    assert_close(got, oracle.workload_attention(w), w.dtype, "full %s (attention)" % name)


def test_decode_is_deterministic(clean_status):
    w = random_decode(15, 4, 200, 900)
    dw = run(w, split=64)
    a = bits_of(dw.out).copy()
    dw.attention()
    torch.cuda.synchronize()
    assert np.array_equal(a, bits_of(dw.out))


@pytest.mark.parametrize("copies", [14, 110])
@pytest.mark.parametrize("split", [None, 64])
def test_full_and_last_splits_in_one_batch(clean_status, split, copies):
    # the decode CTAs take every full split first, then the shorter last splits
    # by decreasing length: contexts that are whole multiples of the split
    # (no last split), contexts one key past a multiple (a one-key last split),
    # equal contexts (equal last splits, kept in sequence order) and a
    # one-key context; 140 sequences take that order, 1100 (more than the
    # ordered lookup holds) the grid's index order
    ctx = [64, 128, 192, 65, 129, 1, 100, 100, 63, 256] * copies
    w = custom(37, Hq=8, Hkv=2, prefix=[c - 1 for c in ctx], qlen=[1] * len(ctx))
    dw = run(w, split=split)
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype, "split order (%d sequences)" % len(ctx))
