"""The radix-tree prefix cache: the oracle pinned to what kshipra-3 section 3
states (brute force, the eviction cascade, LRU order, reference counts), then
the library (host C++ behind the C ABI) against the oracle.  No GPU needed."""

import itertools
import random

import pytest

from oracle.blocks import OK, LifoPool
from oracle.prefix_cache import PrefixCache

BS = 4


@pytest.fixture(scope="module")
def K():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_arena_gb300 as K
    return K


def cached_request(cache, pool, tokens):
    """A request that computed all its tokens into fresh blocks, cached them
    and finished (its own references dropped)."""
    nblk = -(-len(tokens) // cache.bs)
    st, blocks = pool.alloc(nblk)
    assert st == OK
    assert cache.insert(tokens, blocks)[0] == OK
    assert pool.release(blocks) == OK
    return blocks


def lcp(a, b):
    n = 0
    while n < min(len(a), len(b)) and a[n] == b[n]:
        n += 1
    return n


# ---- pins

def test_oracle_match_is_the_longest_cached_prefix():
    # brute force: every full-block prefix any insert cached, in a flat dict
    # (first insert wins); the match is the longest common prefix with any of
    # them, and its blocks are the cached prefixes of the request
    for seed in range(40):
        rnd = random.Random(seed)
        pool = LifoPool(400)
        cache = PrefixCache(pool, BS)
        flat = {}
        for _ in range(12):
            toks = [rnd.randrange(3) for _ in range(rnd.randrange(0, 20))]
            blocks = cached_request(cache, pool, toks)
            for j in range(len(toks) // BS):
                flat.setdefault(tuple(toks[:(j + 1) * BS]), blocks[j])
        for _ in range(30):
            q = [rnd.randrange(3) for _ in range(rnd.randrange(0, 20))]
            want_n = max([lcp(p, q) for p in flat] + [0])
            k, c = divmod(want_n, BS)
            want = [flat[tuple(q[:(j + 1) * BS])] for j in range(k)]
            if c:
                want.append(min(b for p, b in flat.items() if len(p) == (k + 1) * BS and lcp(p, q) == want_n))
            blocks, n = cache.match(q)
            assert (blocks, n) == (want, want_n), (seed, q)
            assert pool.release(blocks) == OK


def test_oracle_eviction_cascades_to_the_parent():
    # the section's failing case: a chain of two cached blocks; evicting the
    # leaf makes its parent a leaf, so evict(2) frees both
    pool = LifoPool(8)
    cache = PrefixCache(pool, BS)
    cached_request(cache, pool, list(range(2 * BS)))
    assert cache.evictable() == 2
    assert cache.evict(2) == 2
    assert cache.num_nodes() == 0 and len(pool.free) == 8


def test_the_cascade_pin_catches_a_leaf_snapshot():
    # plant the bug the section describes (leaves listed once) in the oracle:
    # the same case then frees only one block
    class Snapshot(PrefixCache):
        def evict(self, target):
            leaves = sorted((n for n in self.nodes() if not n.children and self.pool.refcount(n.block) == 1),
                            key=lambda n: (n.stamp, n.block))
            freed = 0
            for leaf in leaves[:target]:
                del leaf.parent.children[leaf.tokens]
                self.pool.release([leaf.block])
                freed += 1
            return freed

    pool = LifoPool(8)
    cache = Snapshot(pool, BS)
    cached_request(cache, pool, list(range(2 * BS)))
    assert cache.evict(2) == 1


def test_oracle_evicts_the_least_recently_used_leaf_first():
    pool = LifoPool(16)
    cache = PrefixCache(pool, BS)
    a = cached_request(cache, pool, [1] * BS)          # stamp 1
    b = cached_request(cache, pool, [2] * BS)          # stamp 2
    c = cached_request(cache, pool, [3] * BS)          # stamp 3
    got, _ = cache.match([1] * BS)                     # a used again: stamp 4
    pool.release(got)
    assert cache.evict(1) == 1 and pool.free[-1] == b[0]
    assert cache.evict(1) == 1 and pool.free[-1] == c[0]
    assert cache.evict(1) == 1 and pool.free[-1] == a[0]


def test_oracle_keeps_blocks_a_request_still_holds():
    pool = LifoPool(16)
    cache = PrefixCache(pool, BS)
    cached_request(cache, pool, list(range(3 * BS)))
    held, n = cache.match(list(range(2 * BS)) + [99])  # holds the first two blocks
    assert n == 2 * BS and len(held) == 2
    assert cache.evictable() == 1
    assert cache.evict(3) == 1                          # only the unheld leaf
    assert all(pool.refcount(b) == 2 for b in held)
    pool.release(held)
    assert cache.evict(3) == 2 and cache.num_nodes() == 0


def test_oracle_reference_counts():
    pool = LifoPool(16)
    cache = PrefixCache(pool, BS)
    st, blocks = pool.alloc(3)
    toks = list(range(2 * BS + 1))                      # two full blocks and one token
    assert cache.insert(toks, blocks) == (OK, 2)        # the partial block is not cached
    assert [pool.refcount(b) for b in blocks] == [2, 2, 1]
    again, _ = cache.match(toks)
    assert again == blocks[:2] and [pool.refcount(b) for b in blocks] == [3, 3, 1]
    assert cache.insert(toks, blocks) == (OK, 0)        # already cached: no new reference
    pool.release(again)
    pool.release(blocks)
    cache.clear()
    assert len(pool.free) == 16


def test_oracle_duplicate_block_keeps_the_cached_one():
    pool = LifoPool(16)
    cache = PrefixCache(pool, BS)
    first = cached_request(cache, pool, list(range(BS)))
    st, mine = pool.alloc(2)                            # computed the same block again, and one more
    assert cache.insert(list(range(2 * BS)), mine) == (OK, 1)
    got, n = cache.match(list(range(2 * BS)))
    assert got == [first[0], mine[1]] and n == 2 * BS


def test_oracle_divergence_inside_a_cached_block_needs_copy_on_write():
    pool = LifoPool(16)
    cache = PrefixCache(pool, BS)
    cached = cached_request(cache, pool, [5, 6, 7, 8, 9, 10, 11, 12])
    got, n = cache.match([5, 6, 7, 8, 9, 10, 42])       # diverges at slot 2 of block 1
    assert got == cached and n == 6
    st, fresh, src = pool.make_private(got[1])          # before writing slot 2
    assert st == OK and src == cached[1] and fresh != cached[1]
    assert pool.refcount(cached[1]) == 1                # the tree's reference


def test_oracle_evictable_is_what_evict_frees():
    for seed in range(20):
        rnd = random.Random(seed)
        pool = LifoPool(300)
        cache = PrefixCache(pool, BS)
        held = []
        for _ in range(15):
            cached_request(cache, pool, [rnd.randrange(2) for _ in range(rnd.randrange(BS, 24))])
            if rnd.random() < 0.3:
                held.append(cache.match([rnd.randrange(2) for _ in range(rnd.randrange(0, 24))])[0])
        want = cache.evictable()
        assert cache.evict(10 ** 6) == want
        assert cache.evictable() == 0


# ---- the library against the oracle

def run_ops(K, seed, num_blocks=160, steps=500):
    rnd = random.Random(seed)
    pool_o, pool_l = LifoPool(num_blocks), K.BlockPool(num_blocks)
    cache_o, cache_l = PrefixCache(pool_o, BS), K.PrefixCache(pool_l, BS)
    held = []  # references the test holds (same ids on both sides)
    prompts = [[rnd.randrange(3) for _ in range(rnd.randrange(0, 28))] for _ in range(6)]

    def request_tokens():
        base = rnd.choice(prompts)
        return base[:rnd.randrange(len(base) + 1)] + [rnd.randrange(3) for _ in range(rnd.randrange(0, 10))]

    for _ in range(steps):
        op = rnd.choice(["match", "insert", "insert", "release", "evict", "private"])
        if op == "match":
            q = request_tokens()
            got = cache_o.match(q)
            assert cache_l.match(q) == got
            held += got[0]
        elif op == "insert":
            toks = request_tokens()
            nblk = -(-len(toks) // BS)
            st, blocks = pool_o.alloc(nblk)
            if st != OK:
                with pytest.raises(K.KshipraError):
                    pool_l.alloc(nblk)
                continue
            assert pool_l.alloc(nblk) == blocks
            assert cache_l.insert(toks, blocks) == cache_o.insert(toks, blocks)[1]
            pool_o.release(blocks)
            pool_l.release(blocks)
        elif op == "release" and held:
            ids = [held.pop(rnd.randrange(len(held))) for _ in range(min(len(held), rnd.randint(1, 6)))]
            pool_o.release(ids)
            pool_l.release(ids)
        elif op == "evict":
            n = rnd.randint(0, 12)
            assert cache_l.evict(n) == cache_o.evict(n)
        elif op == "private" and held:
            j = rnd.randrange(len(held))
            st, new, src = pool_o.make_private(held[j])
            if st == OK:
                assert pool_l.make_private(held[j]) == (new, src)
                held[j] = new
            else:
                with pytest.raises(K.KshipraError):
                    pool_l.make_private(held[j])
        assert cache_l.num_nodes == cache_o.num_nodes()
        assert cache_l.evictable == cache_o.evictable()
        assert pool_l.num_free == len(pool_o.free)
    assert all(pool_l.refcount(i) == pool_o.refcount(i) for i in range(num_blocks))
    cache_l.close()
    cache_o.clear()
    pool_l.release(held)
    assert pool_l.num_free == num_blocks
    pool_l.close()


@pytest.mark.parametrize("seed", range(6))
def test_library_cache_matches_oracle(K, seed):
    run_ops(K, seed)


def test_library_insert_checks_before_it_changes_anything(K):
    pool = K.BlockPool(8)
    cache = K.PrefixCache(pool, BS)
    blocks = pool.alloc(2)
    with pytest.raises(K.KshipraError):
        cache.insert(list(range(2 * BS)), [blocks[0], 7])   # block 7 is free
    assert cache.num_nodes == 0 and pool.refcount(blocks[0]) == 1
    with pytest.raises(K.KshipraError):
        cache.insert(list(range(2 * BS)), [blocks[0], blocks[0]])  # one block twice
    with pytest.raises(K.KshipraError):
        cache.insert(list(range(2 * BS)), blocks[:1])         # too few blocks
    assert cache.insert(list(range(2 * BS)), blocks) == 2
    cache.close()


def test_library_long_chain_cascade(K):
    # one 4096-block sequence evicted leaf by leaf, each parent in turn
    pool = K.BlockPool(4096)
    cache = K.PrefixCache(pool, 16)
    blocks = pool.alloc(4096)
    toks = list(itertools.islice(itertools.cycle(range(7)), 4096 * 16))
    assert cache.insert(toks, blocks) == 4096
    pool.release(blocks)
    assert cache.evictable == 4096
    assert cache.evict(5000) == 4096
    assert pool.num_free == 4096 and cache.num_nodes == 0
