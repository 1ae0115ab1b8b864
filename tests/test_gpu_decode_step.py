"""kshipra_decode_step on the GPU: for decode batches RoPE-and-append fused
into the decode kernel, for batches with prefill rows a K/V append followed by
attention kernels that rotate q themselves.  The same arena image and rotated
q, bit for bit, as the append kernel and the oracle (pages "Building Kshipra"
part 3: section 1 block arena, section 4 RoPE at absolute positions), and
attention within tolerance of the float64 oracle and bit-identical to the
two-call path."""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, custom, random_decode
from workloads import make_config
from workloads.device import NAN_SENTINEL, DeviceWorkload, bits_of, to_device_bits

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


PREFILL_CASES = {
    # batches with prefill-class rows: a K/V-only append, then attention
    # kernels that rotate q themselves (head_dim 128), decode rows included
    "chunked-prefill": lambda: make_config("chunked-prefill"),
    "mixed": lambda: make_config("mixed"),
    "g1": lambda: custom(61, Hq=4, Hkv=4, prefix=[5, 250], qlen=[130, 40]),
    "g2": lambda: custom(62, Hq=8, Hkv=4, prefix=[300, 0, 77], qlen=[260, 513, 31]),
    "g8-bs32-bf16": lambda: custom(63, Hq=16, Hkv=2, bs=32, dtype="bf16", prefix=[33, 400], qlen=[20, 3]),
    "g16-bs32": lambda: custom(64, Hq=32, Hkv=2, bs=32, prefix=[64, 7], qlen=[9, 30]),
    "shared-prefix": lambda: custom(65, Hq=8, Hkv=2, prefix=[64, 96, 200], qlen=[40, 1, 70], shared_len=64,
                                    shared=(0, 1, 2)),
    # more work-list entries than the attention kernel plans itself: the
    # planning kernel runs first
    "1030-chunks": lambda: custom(36, Hq=8, Hkv=2, prefix=[(7 * k) % 23 for k in range(1030)], qlen=[5] * 1030),
}


@pytest.mark.parametrize("name", sorted(PREFILL_CASES))
def test_fused_prefill_step(clean_status, name):
    w = PREFILL_CASES[name]()
    dw = fused(w)
    ka, va = oracle.workload_arena(w, NAN_SENTINEL)
    assert np.array_equal(bits_of(dw.k_arena), ka)
    assert np.array_equal(bits_of(dw.v_arena), va)
    assert np.array_equal(bits_of(dw.q_rot), oracle.workload_q_rot(w))
    what = ("full %s (fused step)" % name) if name in ("chunked-prefill", "mixed") else name
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype, what)
    ref = two_calls(w)
    assert np.array_equal(bits_of(dw.out), bits_of(ref.out))


def test_fused_prefill_step_without_q_rot(clean_status):
    w = custom(66, prefix=[10, 300, 0], qlen=[140, 1, 64])
    dw = fused(w, q_rot=False)
    ka, va = oracle.workload_arena(w, NAN_SENTINEL)
    assert np.array_equal(bits_of(dw.k_arena), ka) and np.array_equal(bits_of(dw.v_arena), va)
    assert np.array_equal(bits_of(dw.out), bits_of(two_calls(w).out))


def test_fused_prefill_steps_in_a_row(clean_status):
    # consecutive steps on one stream: each step's attention starts while its
    # own append finishes, never before the previous step is done
    w = custom(67, prefix=[0, 700], qlen=[300, 129])
    dw = DeviceWorkload(w)
    outs = []
    for _ in range(4):
        dw.decode_step()
        outs.append(dw.out.clone())
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert np.array_equal(bits_of(o), bits_of(outs[0]))
    assert_close(outs[0].float().cpu().numpy().astype(np.float64), oracle.workload_attention(w), w.dtype, "in a row")


def test_fused_prefill_step_sees_inputs_written_just_before(clean_status):
    # the step's attention kernels read q, positions and tables before they
    # wait for the K/V append: those inputs must still be the ones that the
    # kernels queued before the step wrote -- here q is overwritten by a copy
    # on the same stream right before each step
    w = custom(68, prefix=[0, 900, 2000], qlen=[256, 384, 128])
    w2 = custom(69, prefix=[0, 900, 2000], qlen=[256, 384, 128])
    dw = DeviceWorkload(w)
    q_a = dw.q.clone()
    q_b = to_device_bits(w2.q, dw.q.dtype, "cuda")
    for _ in range(3):
        dw.q.copy_(q_b)
        dw.decode_step()
        out_b = dw.out.clone()
        dw.q.copy_(q_a)
        dw.decode_step()
        out_a = dw.out.clone()
    torch.cuda.synchronize()
    ref = two_calls(w)
    assert np.array_equal(bits_of(out_a), bits_of(ref.out))
    w.q = w2.q
    assert_close(out_b.float().cpu().numpy().astype(np.float64), oracle.workload_attention(w), w.dtype, "q from b")


HD64_CASES = {
    "g4": lambda: custom(48, Hq=8, Hkv=2, d=64, prefix=[10, 300], qlen=[40, 1]),
    "g1-bf16-bs32": lambda: custom(49, Hq=4, Hkv=4, d=64, bs=32, dtype="bf16", prefix=[0, 500, 77],
                                   qlen=[130, 200, 3]),
    "g16-many-tiles": lambda: custom(50, Hq=16, Hkv=1, d=64, prefix=[1200, 0], qlen=[33, 260]),
}


@pytest.mark.parametrize("name", sorted(HD64_CASES))
def test_fused_prefill_step_head_dim_64(clean_status, name):
    # head_dim 64 (one-CTA prefill kernel): K/V append, then the prefill
    # kernel rotating q in shared memory; the arena and q_rot bit for bit, the
    # output as the two calls give it
    w = HD64_CASES[name]()
    dw = fused(w)
    ka, va = oracle.workload_arena(w, NAN_SENTINEL)
    assert np.array_equal(bits_of(dw.k_arena), ka) and np.array_equal(bits_of(dw.v_arena), va)
    assert np.array_equal(bits_of(dw.q_rot), oracle.workload_q_rot(w))
    assert_close(dw.out_f64(), oracle.workload_attention(w), w.dtype, "fused step, head_dim 64")
    assert np.array_equal(bits_of(dw.out), bits_of(two_calls(w).out))


def test_fused_prefill_step_head_dim_64_without_q_rot(clean_status):
    w = custom(51, Hq=8, Hkv=2, d=64, prefix=[10, 300, 0], qlen=[140, 1, 64])
    dw = fused(w, q_rot=False)
    ka, va = oracle.workload_arena(w, NAN_SENTINEL)
    assert np.array_equal(bits_of(dw.k_arena), ka) and np.array_equal(bits_of(dw.v_arena), va)
    assert np.array_equal(bits_of(dw.out), bits_of(two_calls(w).out))
