"""Test infrastructure: the oracle of the block pool and of block moves.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg use this
module; the library never does.

Pages "Building Kshipra" part 3 (kshipra-3):
  section 1 -- the arena's blocks sit on a free list that starts as
    list(range(num_blocks)); allocation is list.pop() (the highest id first),
    freeing is list.append(block) (the next allocation reuses it: LIFO);
  section 3 -- reference counts keep shared prefix blocks alive; a block is
    copied before a request that diverges inside it writes it;
  section 5 -- a preempted sequence's blocks are swapped out of the arena and
    restored later.
This restates those rules with a Python list and dict, and the moves as numpy
indexing, with no shortcuts.
"""

from __future__ import annotations

import numpy as np

OK, INVALID_ARG, OUT_OF_BLOCKS = 0, 1, 5


class LifoPool:
    def __init__(self, num_blocks: int):
        self.free = list(range(num_blocks))  # pop() returns the highest id first
        self.refs = {}                         # allocated id -> reference count

    def alloc(self, n: int):
        if n > len(self.free):
            return OUT_OF_BLOCKS, []
        ids = [self.free.pop() for _ in range(n)]
        for i in ids:
            self.refs[i] = 1
        return OK, ids

    def share(self, ids):
        if any(i not in self.refs for i in ids):
            return INVALID_ARG
        for i in ids:
            self.refs[i] += 1
        return OK

    def release(self, ids):
        left = dict(self.refs)
        for i in ids:  # all or nothing
            if left.get(i, 0) <= 0:
                return INVALID_ARG
            left[i] -= 1
        for i in ids:
            self.refs[i] -= 1
            if self.refs[i] == 0:
                del self.refs[i]
                self.free.append(i)  # the next allocation reuses it
        return OK

    def refcount(self, i: int) -> int:
        return self.refs.get(i, 0)

    def make_private(self, i: int):
        """(status, id to write into, id to copy from or -1)."""
        if i not in self.refs:
            return INVALID_ARG, i, -1
        if self.refs[i] == 1:
            return OK, i, -1
        if not self.free:
            return OUT_OF_BLOCKS, i, -1
        fresh = self.free.pop()
        self.refs[fresh] = 1
        self.refs[i] -= 1
        return OK, fresh, i


def copy_blocks(arena: np.ndarray, src_ids, dst_ids) -> np.ndarray:
    """arena [num_blocks][...] with block dst_ids[i] replaced by src_ids[i]."""
    out = arena.copy()
    out[np.asarray(dst_ids)] = arena[np.asarray(src_ids)]
    return out


def gather_blocks(arena: np.ndarray, ids) -> np.ndarray:
    return arena[np.asarray(ids)].copy()


def scatter_blocks(arena: np.ndarray, ids, rows: np.ndarray) -> np.ndarray:
    out = arena.copy()
    out[np.asarray(ids)] = rows
    return out
