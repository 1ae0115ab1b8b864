"""Requests served through the radix-tree prefix cache (pages "Building
Kshipra" part 3, section 3): a request reuses the cached blocks of its
longest cached prefix in place, copies a shared block before writing into it,
computes only the rest, and its attention over the mixed cached and fresh
blocks equals the float64 oracle over its whole sequence."""

import numpy as np
import pytest
import torch

import oracle
from workloads.device import to_device_bits

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS, THETA, NB = 8, 2, 128, 16, 1.0e4, 32


class Rows:
    """Synthetic q, k, v rows for each token, drawn once per token prefix:
    two sequences that agree up to position p have the same rows up to p, as
    a causal model's would."""

    def __init__(self, seed):
        self.rng = np.random.default_rng(seed)
        self.memo = {}

    def __call__(self, tokens):
        out = []
        for p in range(len(tokens)):
            key = tuple(tokens[:p + 1])
            if key not in self.memo:
                draw = lambda h: oracle.f64_to_bits(self.rng.standard_normal((h, D)), "f16")
                self.memo[key] = (draw(HQ), draw(HKV), draw(HKV))
            out.append(self.memo[key])
        return [np.stack([r[i] for r in out]) for i in range(3)]


def serve(K, pool, cache, rows, tokens, k_arena, v_arena, rope):
    """One request: reuse, copy-on-write, append the rest, attention over its
    new tokens; checked against the oracle; then cached and finished."""
    n = len(tokens)
    blocks, m = cache.match(tokens[:n - 1])  # at least the last token is computed
    if m % BS:
        new, src = pool.make_private(blocks[-1])
        if src >= 0:
            K.kshipra_blocks_copy(k_arena, v_arena, torch.tensor([src], dtype=torch.int32, device="cuda"),
                                  torch.tensor([new], dtype=torch.int32, device="cuda"))
            blocks[-1] = new
    blocks += pool.alloc(-(-n // BS) - len(blocks))
    q, k, v = rows(tokens)
    dev = lambda a: to_device_bits(a, torch.float16, "cuda")
    i32 = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    table = i32([blocks])
    qsl, pos, ctx = [0, n - m], list(range(m, n)), [n]
    q_rot = torch.empty((n - m, HQ, D), dtype=torch.float16, device="cuda")
    K.kshipra_kv_append_rope(dev(q[m:]), dev(k[m:]), dev(v[m:]), q_rot, k_arena, v_arena, table, i32(qsl), i32(pos),
                             rope)
    out = torch.empty_like(q_rot)
    ws = torch.empty(max(K.kshipra_paged_attention_workspace_size(1, n - m, n, HQ, HKV, D), 1), dtype=torch.uint8,
                     device="cuda")
    K.kshipra_paged_attention(out, q_rot, k_arena, v_arena, table, i32(ctx), i32(qsl), i32(pos), n - m, n,
                              D ** -0.5, ws)
    torch.cuda.synchronize()
    ref = oracle.attention(q[m:], k, v, np.array([0]), np.array(qsl), np.array(pos), np.array(ctx), HKV, THETA,
                           D ** -0.5, "f16", block_tables=np.array([blocks]), block_size=BS, num_blocks=NB)
    err = np.abs(out.float().cpu().numpy().astype(np.float64) - ref).max()
    assert err <= 2e-3, (m, err)
    cache.insert(tokens, blocks)
    pool.release(blocks)
    return m, blocks


def test_requests_share_cached_blocks_in_place(clean_status):
    K = clean_status
    pool = K.BlockPool(NB)
    cache = K.PrefixCache(pool, BS)
    k_arena = torch.full((NB, HKV, BS, D), float("nan"), dtype=torch.float16, device="cuda")
    v_arena = torch.full_like(k_arena, float("nan"))
    rope = torch.from_numpy(K.kshipra_rope_table_build(128, D, THETA)).cuda()
    rows = Rows(11)
    rng = np.random.default_rng(12)
    a = [int(t) for t in rng.integers(0, 50, 57)]
    b = a[:40] + [int(t) + 50 for t in rng.integers(0, 50, 15)]  # diverges at slot 8 of block 2
    a2 = a + [7, 8]

    m, a_blocks = serve(K, pool, cache, rows, a, k_arena, v_arena, rope)
    assert m == 0 and cache.num_nodes == 3                   # A's three full blocks
    m, b_blocks = serve(K, pool, cache, rows, b, k_arena, v_arena, rope)
    assert m == 40 and b_blocks[:2] == a_blocks[:2] and b_blocks[2] != a_blocks[2]
    assert cache.num_nodes == 4                               # B's own block 2 joins the tree
    m, a2_blocks = serve(K, pool, cache, rows, a2, k_arena, v_arena, rope)
    assert m == 48 and a2_blocks[:3] == a_blocks[:3]          # A's block 2 kept A's rows
    assert cache.evictable == 4
    assert cache.evict(NB) == 4 and pool.num_free == NB
    cache.close()
    pool.close()
