"""Test infrastructure: the oracle of the radix-tree prefix cache.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg use this
module; the library never does.

Pages "Building Kshipra" part 3 (kshipra-3), section 3 "Radix-Tree Prefix
Cache and the Eviction Bug":
  - the cached KV blocks form a tree whose edges are blocks of tokens; a new
    request walks down from the root, reuses every block that matches and
    computes only what is left;
  - reference counts (the block pool of section 1) keep shared blocks alive;
    a request that diverges inside a shared block copies it before writing;
  - under memory pressure the least recently used leaf is evicted; eviction
    looks for that leaf again on every iteration, because removing a leaf
    can make its parent a leaf (the bug the section describes came from
    listing the leaves once).

Readings where the section leaves a step open (plainest reading):
  - a node holds one full block: block_size tokens and the physical block
    with their K/V; children of a node are keyed by their whole token block;
  - the walk takes full blocks while one matches, then, if no full block
    matches, the child sharing the longest run of leading tokens with the
    rest of the request (ties: the smaller block id); that block is reused
    for those tokens only, and the request copies it before writing the
    next slot (the copy-on-write case);
  - the tree holds one reference to each block it caches; match() takes one
    more for the caller; a leaf is evictable when the tree's reference is the
    only one left; recency is a logical clock that advances once per
    match()/insert() and stamps every node the call walks; the least
    recently used evictable leaf is the one with the smallest stamp (ties:
    the smaller block id);
  - insert() registers the full blocks of a request's tokens; where a block
    with the same tokens is already cached under the same parent, the cached
    one stays and the request's own block is not added.
This restates those rules with plain Python objects, dicts and a full tree
re-scan for every evicted leaf, with no index structures.
"""

from __future__ import annotations

from oracle.blocks import INVALID_ARG, OK, LifoPool


class _Node:
    __slots__ = ("tokens", "block", "parent", "children", "stamp")

    def __init__(self, tokens, block, parent):
        self.tokens = tokens      # tuple of block_size token ids (root: ())
        self.block = block        # physical block id (root: -1)
        self.parent = parent
        self.children = {}        # tokens tuple -> _Node
        self.stamp = 0


class PrefixCache:
    def __init__(self, pool: LifoPool, block_size: int):
        self.pool = pool
        self.bs = block_size
        self.root = _Node((), -1, None)
        self.clock = 0

    # -- walking
    def nodes(self):
        out, stack = [], list(self.root.children.values())
        while stack:
            n = stack.pop()
            out.append(n)
            stack.extend(n.children.values())
        return out

    def match(self, tokens):
        """Longest cached prefix of tokens: (blocks, matched token count).
        The caller gets one reference to each returned block."""
        self.clock += 1
        bs, node, i, path = self.bs, self.root, 0, []
        while len(tokens) - i >= bs:
            child = node.children.get(tuple(tokens[i:i + bs]))
            if child is None:
                break
            path.append(child)
            node, i = child, i + bs
        rest = tokens[i:i + bs]
        best, best_c = None, 0
        for child in node.children.values():
            c = 0
            while c < len(rest) and child.tokens[c] == rest[c]:
                c += 1
            if c > best_c or (c == best_c and c > 0 and child.block < best.block):
                best, best_c = child, c
        if best is not None:
            path.append(best)
            i += best_c
        for n in path:
            n.stamp = self.clock
        blocks = [n.block for n in path]
        assert self.pool.share(blocks) == OK
        return blocks, i

    def insert(self, tokens, blocks):
        """Caches the full blocks of tokens (block j holds tokens
        [j*bs, (j+1)*bs)).  Returns (status, number of blocks added)."""
        bs = self.bs
        full = len(tokens) // bs
        if len(blocks) < full:
            return INVALID_ARG, 0
        cached = {n.block for n in self.nodes()}
        # check everything before changing anything
        node, new = self.root, []
        for j in range(full):
            key = tuple(tokens[j * bs:(j + 1) * bs])
            child = node.children.get(key) if node is not None else None
            if child is None:
                b = blocks[j]
                if self.pool.refcount(b) <= 0 or b in cached or b in new:
                    return INVALID_ARG, 0
                new.append(b)
            node = child
        self.clock += 1
        node, added = self.root, 0
        for j in range(full):
            key = tuple(tokens[j * bs:(j + 1) * bs])
            child = node.children.get(key)
            if child is None:
                child = _Node(key, blocks[j], node)
                node.children[key] = child
                assert self.pool.share([blocks[j]]) == OK  # the tree's reference
                added += 1
            child.stamp = self.clock
            node = child
        return OK, added

    # -- eviction
    def _lru_leaf(self):
        best = None
        for n in self.nodes():  # the whole tree, every time
            if n.children or self.pool.refcount(n.block) != 1:
                continue
            if best is None or (n.stamp, n.block) < (best.stamp, best.block):
                best = n
        return best

    def evict(self, target: int) -> int:
        freed = 0
        while freed < target:
            leaf = self._lru_leaf()
            if leaf is None:
                break  # nothing evictable left
            del leaf.parent.children[leaf.tokens]
            assert self.pool.release([leaf.block]) == OK
            freed += 1
        return freed

    def evictable(self) -> int:
        """Blocks that evict() could free now, counting leaves that appear as
        their children go (a node whose whole subtree is held by the tree
        alone)."""
        def count(n):
            total, whole = 0, True
            for c in n.children.values():
                t, w = count(c)
                total += t
                whole = whole and w
            if n is self.root:
                return total, whole
            if whole and self.pool.refcount(n.block) == 1:
                return total + 1, True
            return total, False
        return count(self.root)[0]

    def num_nodes(self) -> int:
        return len(self.nodes())

    def clear(self):
        for n in self.nodes():
            assert self.pool.release([n.block]) == OK
        self.root.children = {}
