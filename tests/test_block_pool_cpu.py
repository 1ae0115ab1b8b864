"""The block pool (host C++ behind the C ABI) against the oracle's restatement
of kshipra-3 sections 1 and 3, and the oracle against the pages' own
statements.  No GPU needed."""

import random
import threading

import pytest

from oracle.blocks import INVALID_ARG, OK, OUT_OF_BLOCKS, LifoPool


@pytest.fixture(scope="module")
def K():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_arena_gb300 as K
    return K


# ---- pins: the pages' rules, stated directly

def test_oracle_first_allocation_is_the_highest_id():
    # "free = list(range(num_blocks)) # pop() returns the highest block ID first" (section 1)
    pool = LifoPool(10)
    assert pool.alloc(3) == (OK, [9, 8, 7])


def test_oracle_reuses_the_most_recently_freed_block():
    # freeing appends; the next allocation reuses that block (section 1)
    pool = LifoPool(10)
    _, ids = pool.alloc(4)                # 9 8 7 6
    assert pool.release([8]) == OK
    assert pool.release([6]) == OK
    assert pool.alloc(2) == (OK, [6, 8])  # last freed first
    assert pool.alloc(1) == (OK, [5])


def test_oracle_shared_blocks_stay_alive_until_the_last_reference():
    # reference counts keep shared prefix blocks alive (section 3)
    pool = LifoPool(4)
    _, (a,) = pool.alloc(1)
    pool.share([a])
    pool.release([a])
    assert pool.refcount(a) == 1 and a not in pool.free
    pool.release([a])
    assert pool.refcount(a) == 0 and pool.free[-1] == a


def test_oracle_copy_on_write():
    # a shared block is copied before a request that diverges inside it writes it (section 3)
    pool = LifoPool(6)
    _, (a,) = pool.alloc(1)
    assert pool.make_private(a) == (OK, a, -1)      # private: write in place
    pool.share([a])
    st, fresh, src = pool.make_private(a)
    assert st == OK and src == a and fresh != a
    assert pool.refcount(a) == 1 and pool.refcount(fresh) == 1


# ---- the library against the oracle

def run_ops(K, seed, num_blocks=48, steps=600):
    rnd = random.Random(seed)
    ref, lib = LifoPool(num_blocks), K.BlockPool(num_blocks)
    held = []  # ids with one reference owned by the test
    for _ in range(steps):
        op = rnd.choice(["alloc", "alloc", "share", "release", "release", "private", "bad"])
        if op == "alloc":
            n = rnd.randint(0, 6)
            st, ids = ref.alloc(n)
            if st == OK:
                assert lib.alloc(n) == ids
                held += ids
            else:
                with pytest.raises(K.KshipraError) as e:
                    lib.alloc(n)
                assert e.value.code == OUT_OF_BLOCKS
        elif op == "share" and held:
            ids = rnd.sample(held, min(len(held), rnd.randint(1, 3)))
            assert ref.share(ids) == OK
            lib.share(ids)
            held += ids
        elif op == "release" and held:
            ids = [held.pop(rnd.randrange(len(held))) for _ in range(min(len(held), rnd.randint(1, 4)))]
            assert ref.release(ids) == OK
            lib.release(ids)
        elif op == "private" and held:
            j = rnd.randrange(len(held))
            st, new, src = ref.make_private(held[j])
            if st == OK:
                assert lib.make_private(held[j]) == (new, src)
                held[j] = new
            else:
                with pytest.raises(K.KshipraError) as e:
                    lib.make_private(held[j])
                assert e.value.code == st
        elif op == "bad":
            # releasing a free block, or one too many references, changes nothing
            free_id = ref.free[0] if ref.free else None
            if free_id is not None:
                assert ref.release([free_id]) == INVALID_ARG
                with pytest.raises(K.KshipraError):
                    lib.release([free_id])
        assert lib.num_free == len(ref.free)
        for i in range(num_blocks):
            assert lib.refcount(i) == ref.refcount(i)
    lib.close()


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_library_pool_matches_oracle(K, seed):
    run_ops(K, seed)


def test_alloc_is_all_or_nothing(K):
    pool = K.BlockPool(4)
    pool.alloc(3)
    with pytest.raises(K.KshipraError) as e:
        pool.alloc(2)
    assert e.value.code == OUT_OF_BLOCKS and pool.num_free == 1
    assert pool.alloc(1) == [0]


def test_release_with_a_bad_entry_changes_nothing(K):
    pool = K.BlockPool(4)
    ids = pool.alloc(2)  # 3, 2
    with pytest.raises(K.KshipraError):
        pool.release([ids[0], ids[0]])  # the second drop would go below zero
    assert pool.refcount(ids[0]) == 1 and pool.num_free == 2
    with pytest.raises(K.KshipraError):
        pool.release([7])


def test_concurrent_callers_keep_the_pool_consistent(K):
    pool = K.BlockPool(4096)

    def worker(seed):
        rnd = random.Random(seed)
        mine = []
        for _ in range(400):
            if mine and rnd.random() < 0.5:
                pool.release([mine.pop()])
            else:
                mine += pool.alloc(rnd.randint(1, 4))
        pool.release(mine)

    threads = [threading.Thread(target=worker, args=(s,)) for s in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert pool.num_free == 4096
    assert all(pool.refcount(i) == 0 for i in range(4096))
