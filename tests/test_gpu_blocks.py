"""Block moves on the GPU against the oracle's numpy restatement, bit for bit:
the copy-on-write copy and swapping blocks out to pinned host memory and
back in (pages "Building Kshipra" part 3, sections 1, 3 and 5)."""

import numpy as np
import pytest
import torch

import oracle
from oracle.blocks import copy_blocks, gather_blocks, scatter_blocks
from workloads.device import bits_of, to_device_bits

pytestmark = pytest.mark.gpu


def random_arena(seed, nb=64, hkv=8, bs=16, d=128, dtype=torch.float16):
    rng = np.random.default_rng(seed)
    kb = rng.integers(0, 1 << 16, size=(nb, hkv, bs, d), dtype=np.uint16)
    vb = rng.integers(0, 1 << 16, size=(nb, hkv, bs, d), dtype=np.uint16)
    return kb, vb, to_device_bits(kb, dtype, "cuda"), to_device_bits(vb, dtype, "cuda")


def ids_dev(ids):
    return torch.tensor(ids, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("shape", [(64, 8, 16, 128), (40, 2, 32, 64), (20, 4, 16, 64)])
def test_blocks_copy(clean_status, shape):
    K = clean_status
    nb, hkv, bs, d = shape
    kb, vb, k, v = random_arena(1, nb, hkv, bs, d)
    src, dst = [3, 17, 5, nb - 1], [9, 0, 12, 6]
    K.kshipra_blocks_copy(k, v, ids_dev(src), ids_dev(dst))
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(k), copy_blocks(kb, src, dst))
    assert np.array_equal(bits_of(v), copy_blocks(vb, src, dst))


@pytest.mark.parametrize("pinned", [True, False])
def test_swap_out_and_in(clean_status, pinned):
    K = clean_status
    kb, vb, k, v = random_arena(2, dtype=torch.bfloat16)
    out_ids = [50, 3, 22, 7, 63]
    shape = (len(out_ids),) + tuple(k.shape[1:])
    if pinned:  # host side over the CPU-GPU link
        k_buf = torch.empty(shape, dtype=k.dtype, pin_memory=True)
        v_buf = torch.empty(shape, dtype=k.dtype, pin_memory=True)
    else:
        k_buf = torch.empty(shape, dtype=k.dtype, device="cuda")
        v_buf = torch.empty(shape, dtype=k.dtype, device="cuda")
    K.kshipra_blocks_swap_out(k_buf, v_buf, k, v, ids_dev(out_ids))
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(k_buf), gather_blocks(kb, out_ids))
    assert np.array_equal(bits_of(v_buf), gather_blocks(vb, out_ids))
    # restored into other physical blocks
    in_ids = [1, 2, 60, 30, 31]
    K.kshipra_blocks_swap_in(k, v, k_buf, v_buf, ids_dev(in_ids))
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(k), scatter_blocks(kb, in_ids, gather_blocks(kb, out_ids)))
    assert np.array_equal(bits_of(v), scatter_blocks(vb, in_ids, gather_blocks(vb, out_ids)))


def test_pageable_host_memory_is_rejected(gpu):
    K = gpu
    _, _, k, v = random_arena(3)
    k_buf = torch.empty((1,) + tuple(k.shape[1:]), dtype=k.dtype)  # pageable
    with pytest.raises(K.KshipraError) as e:
        K.kshipra_blocks_swap_out(k_buf, k_buf.clone(), k, v, ids_dev([0]))
    assert e.value.code == K.KSHIPRA_ERR_INVALID_ARG


def test_bad_block_id_is_reported_and_skipped(gpu):
    K = gpu
    kb, vb, k, v = random_arena(4)
    src, dst = [1, 2], [10, 64]  # 64 is past the arena
    K.kshipra_blocks_copy(k, v, ids_dev(src), ids_dev(dst))
    assert K.kshipra_device_status() & K.KSHIPRA_DEV_BAD_BLOCK_ID
    assert np.array_equal(bits_of(k), copy_blocks(kb, [1], [10]))


def test_copy_on_write_of_a_partly_filled_shared_block(clean_status):
    # sequences A and B share a 40-token prefix: blocks p0, p1 full and p2
    # holding positions 32..39.  Each then appends its own token at position
    # 40, which lands in p2: the first writer gets a private copy, the second
    # (now the only holder) writes in place.  Each sequence must then read its
    # prefix plus its own token.
    K = clean_status
    hkv, bs, d, theta = 2, 16, 64, 1e4
    pool = K.BlockPool(16)
    rng = np.random.default_rng(5)
    bits = lambda *s: oracle.f64_to_bits(rng.standard_normal(s), "f16")
    prefix_k, prefix_v = bits(40, hkv, d), bits(40, hkv, d)
    shared = pool.alloc(3)
    pool.share(shared)  # A and B both hold p0, p1, p2
    k = torch.zeros((16, hkv, bs, d), dtype=torch.float16, device="cuda")
    v = torch.zeros_like(k)
    table = torch.full((2, 4), -1, dtype=torch.int32, device="cuda")
    table[0, :3] = ids_dev(shared)
    table[1, :3] = ids_dev(shared)
    rope = torch.from_numpy(K.kshipra_rope_table_build(64, d, theta)).cuda()

    def append(seq_rows_k, seq_rows_v, positions, tab):
        qsl = torch.tensor([0, len(positions)], dtype=torch.int32, device="cuda")
        K.kshipra_kv_append_rope(None, to_device_bits(seq_rows_k, torch.float16, "cuda"),
                                 to_device_bits(seq_rows_v, torch.float16, "cuda"), None, k, v, tab, qsl,
                                 ids_dev(positions), rope)

    append(prefix_k, prefix_v, list(range(40)), table[:1])
    torch.cuda.synchronize()
    toks = {s: (bits(1, hkv, d), bits(1, hkv, d)) for s in (0, 1)}
    for s in (0, 1):  # A first, then B
        blk = int(table[s, 2])
        new, src = pool.make_private(blk)
        if src >= 0:
            K.kshipra_blocks_copy(k, v, ids_dev([src]), ids_dev([new]))
            table[s, 2] = new
        append(toks[s][0], toks[s][1], [40], table[s:s + 1])
    torch.cuda.synchronize()
    assert int(table[0, 2]) != shared[2] and int(table[1, 2]) == shared[2]
    assert pool.refcount(shared[2]) == 1 and pool.refcount(int(table[0, 2])) == 1
    kh, vh = bits_of(k), bits_of(v)
    rot = lambda rows, pos: oracle.rope_rows(rows, np.asarray(pos, dtype=np.int32), theta, "f16")
    for s in (0, 1):
        tab = table[s].cpu().numpy()
        got_k = np.stack([kh[tab[p // bs], :, p % bs] for p in range(41)])
        got_v = np.stack([vh[tab[p // bs], :, p % bs] for p in range(41)])
        want_k = np.concatenate([rot(prefix_k, range(40)), rot(toks[s][0], [40])])
        want_v = np.concatenate([prefix_v, toks[s][1]])
        assert np.array_equal(got_k, want_k), s
        assert np.array_equal(got_v, want_v), s
