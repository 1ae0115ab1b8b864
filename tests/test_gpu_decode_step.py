"""kshipra_decode_step (RoPE-and-append fused into the decode kernel) on the
GPU: the same arena image and rotated q, bit for bit, as the append kernel
and the oracle (pages "Building Kshipra" part 3: section 1 block arena,
section 4 RoPE at absolute positions), and attention within tolerance of the
float64 oracle and bit-identical to the two-call path."""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, custom, random_decode
from workloads import make_config
from workloads.device import NAN_SENTINEL, DeviceWorkload, bits_of

pytestmark = pytest.mark.gpu

CASES = {
    "llama-decode": lambda: make_config("llama-decode"),
    "long-decode": lambda: make_config("long-decode"),
    "tiny-decode": lambda: random_decode(41, 3, 1, 60, Hq=4, Hkv=2, d=64),
    "g1-d64": lambda: random_decode(42, 5, 2, 300, Hq=4, Hkv=4, d=64),
    "g8-bs32-bf16": lambda: random_decode(43, 6, 40, 900, Hq=16, Hkv=2, bs=32, dtype="bf16"),
    # several new tokens per sequence (query_len x group <= 16)
    "multi-token": lambda: custom(44, prefix=[0, 17, 250, 1023], qlen=[4, 3, 2, 4]),
    "shared-prefix": lambda: custom(45, Hq=8, Hkv=2, prefix=[64, 70, 100], qlen=[1, 2, 1], shared_len=64,
                                    shared=(0, 1, 2)),
}


def fused(w, q_rot=True, split=None):
    import paged_kv_cache_arena_gb300 as K
    if split is not None:
        K.kshipra_set_option(K.KSHIPRA_OPT_SPLIT_TOKENS, split)
    dw = DeviceWorkload(w)
    dw.decode_step(q_rot=q_rot)
    torch.cuda.synchronize()
    return dw


def two_calls(w, split=None):
    import paged_kv_cache_arena_gb300 as K
    if split is not None:
        K.kshipra_set_option(K.KSHIPRA_OPT_SPLIT_TOKENS, split)
    dw = DeviceWorkload(w)
    dw.step()
    torch.cuda.synchronize()
    return dw


@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_step_matches_oracle_and_two_calls(clean_status, name):
    w = CASES[name]()
    dw = fused(w)
    ka, va = oracle.workload_arena(w, NAN_SENTINEL)
    assert np.array_equal(bits_of(dw.k_arena), ka)
    assert np.array_equal(bits_of(dw.v_arena), va)
    assert np.array_equal(bits_of(dw.q_rot), oracle.workload_q_rot(w))
    got = dw.out_f64()
    what = ("full %s (fused step)" % name) if name in ("llama-decode", "long-decode") else name
    assert_close(got, oracle.workload_attention(w), w.dtype, what)  # every row
    ref = two_calls(w)
    assert np.array_equal(bits_of(dw.out), bits_of(ref.out))


def test_new_tokens_across_a_split_boundary(clean_status):
    # 64-key splits; sequence 0's four new tokens sit at positions 62..65,
    # written by two different split CTAs
    w = custom(46, prefix=[62, 60, 1], qlen=[4, 4, 1])
    dw = fused(w, split=64)
    ka, va = oracle.workload_arena(w, NAN_SENTINEL)
    assert np.array_equal(bits_of(dw.k_arena), ka)
    assert np.array_equal(bits_of(dw.v_arena), va)
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype, "split boundary")
    ref = two_calls(w, split=64)
    assert np.array_equal(bits_of(dw.out), bits_of(ref.out))


def test_without_q_rot_buffer(clean_status):
    w = random_decode(47, 4, 5, 400)
    dw = fused(w, q_rot=False)
    ka, _ = oracle.workload_arena(w, NAN_SENTINEL)
    assert np.array_equal(bits_of(dw.k_arena), ka)
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype, "no q_rot")


def test_prefill_rows_take_the_two_calls(clean_status):
    # a chunk of 40 tokens is beyond the decode kernel: append + attention
    w = custom(48, Hq=8, Hkv=2, prefix=[10, 300], qlen=[40, 1])
    dw = fused(w)
    ka, va = oracle.workload_arena(w, NAN_SENTINEL)
    assert np.array_equal(bits_of(dw.k_arena), ka)
    assert np.array_equal(bits_of(dw.q_rot), oracle.workload_q_rot(w))
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype, "two calls")
