"""RoPE-and-append on the GPU against the oracle's arena image, bit for bit
(pages "Building Kshipra" part 3: section 1 block arena, section 4 RoPE at
absolute positions)."""

import numpy as np
import pytest
import torch

import oracle
from helpers import custom
from workloads import make_config
from workloads.device import NAN_SENTINEL, DeviceWorkload, bits_of

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": lambda: make_config("tiny"),
    "chunked-prefill": lambda: make_config("chunked-prefill"),
    "decode-bs32-bf16": lambda: custom(3, d=128, bs=32, dtype="bf16", prefix=[70, 31, 0, 200], qlen=[1, 1, 5, 40]),
    "d64-g1": lambda: custom(4, Hq=4, Hkv=4, d=64, prefix=[15, 16, 17], qlen=[1, 33, 2]),
    "shared-prefix": lambda: custom(5, Hq=8, Hkv=2, prefix=[64, 70, 90, 10], qlen=[3, 1, 20, 2], shared_len=64,
                                    shared=(0, 1, 2)),
}


def _many_sequences():
    # more sequences than an append CTA has threads, with runs of empty ones:
    # a run of tokens whose sequences lie more than 256 entries apart
    # (sequence 0 ends at token 350, sequences 1-300 have no new token,
    # sequence 301 starts at token 351), and 400 more short sequences
    qlen = [351] + [0] * 300 + [349] + [1, 0] * 200
    prefix = [3] + [5] * 300 + [20] + [7, 2] * 200
    return custom(7, Hq=8, Hkv=2, prefix=prefix, qlen=qlen, spare=4)


CASES["many-sequences"] = _many_sequences


@pytest.mark.parametrize("name", sorted(CASES))
def test_arena_and_q_rot_bit_exact(clean_status, name):
    w = CASES[name]()
    dw = DeviceWorkload(w)
    dw.append_step()
    torch.cuda.synchronize()
    ka, va = oracle.workload_arena(w, NAN_SENTINEL)
    assert np.array_equal(bits_of(dw.k_arena), ka)
    assert np.array_equal(bits_of(dw.v_arena), va)
    assert np.array_equal(bits_of(dw.q_rot), oracle.workload_q_rot(w))


def test_q_rot_may_alias_q(clean_status):
    w = make_config("tiny")
    dw = DeviceWorkload(w)
    K = clean_status
    K.kshipra_kv_append_rope(dw.q, dw.k_new, dw.v_new, dw.q, dw.k_arena, dw.v_arena, dw.block_tables,
                             dw.query_start_loc, dw.positions, dw.rope_table)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(dw.q), oracle.workload_q_rot(w))


def test_bad_block_id_and_position_are_reported_and_skipped(gpu):
    K = gpu
    w = custom(6, Hq=4, Hkv=2, d=64, prefix=[20, 5], qlen=[2, 1], spare=0)
    dw = DeviceWorkload(w)
    before_k = bits_of(dw.k_arena).copy()
    bt = dw.block_tables.clone()
    bt[0, 1] = w.num_blocks  # positions 20, 21 of sequence 0 live in logical block 1
    K.kshipra_kv_append_rope(dw.q, dw.k_new, dw.v_new, dw.q_rot, dw.k_arena, dw.v_arena, bt, dw.query_start_loc,
                             dw.positions, dw.rope_table)
    assert K.kshipra_device_status() & K.KSHIPRA_DEV_BAD_BLOCK_ID
    after_k = bits_of(dw.k_arena)
    # only sequence 1's token was written
    ka, _ = oracle.workload_arena(w, NAN_SENTINEL)
    changed = np.argwhere(np.any(after_k != before_k, axis=-1))
    assert len(changed) == w.num_kv_heads
    assert np.array_equal(after_k[tuple(changed.T)], ka[tuple(changed.T)])
    pos = dw.positions.clone()
    pos[0] = dw.rope_max_pos + 5
    K.kshipra_kv_append_rope(dw.q, dw.k_new, dw.v_new, dw.q_rot, dw.k_arena, dw.v_arena, dw.block_tables,
                             dw.query_start_loc, pos, dw.rope_table)
    assert K.kshipra_device_status() & K.KSHIPRA_DEV_BAD_POSITION
    assert K.kshipra_device_status() == 0  # reading clears the word


def test_full_llama_decode_arena_sampled(clean_status):
    w = make_config("llama-decode")
    dw = DeviceWorkload(w)
    dw.append_step()
    torch.cuda.synchronize()
    # compare the blocks of a sample of sequences: every row they hold
    rng = np.random.default_rng(0)
    seqs = rng.choice(w.num_seqs, 6, replace=False)
    kg, vg = bits_of(dw.k_arena), bits_of(dw.v_arena)
    ks = w.kv_start
    for s in seqs:
        ctx = int(w.context_lens[s])
        rows = np.arange(ks[s], ks[s] + ctx)
        pos = np.arange(ctx, dtype=np.int32)
        kref = oracle.rope_rows(w.k_all[rows], pos, w.theta, w.dtype)
        blk = w.block_tables[s, pos // w.block_size]
        slot = pos % w.block_size
        assert np.array_equal(kg[blk, :, slot], kref)
        assert np.array_equal(vg[blk, :, slot], w.v_all[rows])
