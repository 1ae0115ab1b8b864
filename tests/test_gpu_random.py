"""Seeded random batches on the GPU against the float64 oracle: group sizes,
head_dim, block size, dtype, cached prefixes, chunk lengths and decode rows
drawn at random, some with shared prefix blocks, through the two calls and
through the fused step (pages "Building Kshipra" part 3: section 1 block
arena, section 3 shared prefix blocks, section 4 chunked prefill, section 5
mixed batches)."""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, custom
from workloads.device import NAN_SENTINEL, DeviceWorkload, bits_of

pytestmark = pytest.mark.gpu


def random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    G = int(rng.choice([1, 2, 4, 8, 16]))
    Hkv = int(rng.choice([1, 2, 4])) if G < 16 else int(rng.choice([1, 2]))
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32]))
    dtype = str(rng.choice(["f16", "bf16"]))
    S = int(rng.integers(1, 7))
    prefix, qlen = [], []
    for _ in range(S):
        kind = rng.random()
        if kind < 0.4:      # a decode row
            prefix.append(int(rng.integers(0, 1500)))
            qlen.append(1)
        elif kind < 0.6:    # a few tokens
            prefix.append(int(rng.integers(0, 600)))
            qlen.append(int(rng.integers(2, 5)))
        else:               # a prefill chunk
            prefix.append(int(rng.integers(0, 1200)))
            qlen.append(int(rng.integers(5, 300)))
    shared_len, shared = 0, ()
    if S >= 2 and rng.random() < 0.4:
        shared_len = bs * int(rng.integers(1, 4))
        members = [s for s in range(S) if prefix[s] >= shared_len]
        if len(members) >= 2:
            shared = tuple(members)
        else:
            shared_len = 0
    return custom(seed, Hq=G * Hkv, Hkv=Hkv, d=d, bs=bs, dtype=dtype, prefix=prefix, qlen=qlen, spare=3,
                  shared_len=shared_len, shared=shared)


@pytest.mark.parametrize("seed", range(64))
def test_random_batch_two_calls_and_fused_step(clean_status, seed):
    w = random_case(seed)
    ref = oracle.workload_attention(w)
    ka, va = oracle.workload_arena(w, NAN_SENTINEL)
    two = DeviceWorkload(w)
    two.step()
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(two.k_arena), ka) and np.array_equal(bits_of(two.v_arena), va)
    assert np.array_equal(bits_of(two.q_rot), oracle.workload_q_rot(w))
    assert_close(two.out_f64(), ref, w.dtype, "random %d (two calls)" % seed)
    fused = DeviceWorkload(w)
    fused.decode_step()
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(fused.k_arena), ka) and np.array_equal(bits_of(fused.v_arena), va)
    assert np.array_equal(bits_of(fused.q_rot), oracle.workload_q_rot(w))
    assert np.array_equal(bits_of(fused.out), bits_of(two.out))
