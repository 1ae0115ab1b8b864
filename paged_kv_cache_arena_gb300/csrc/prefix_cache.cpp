// The radix-tree prefix cache over the block pool.
//
// Pages "Building Kshipra" part 3 (kshipra-3), section 3 "Radix-Tree Prefix
// Cache and the Eviction Bug": cached KV blocks form a tree whose edges are
// blocks of tokens; a request walks it from the root and reuses every
// matching block; reference counts keep shared blocks alive and a request
// that diverges inside a shared block copies it before writing; under memory
// pressure the least recently used leaf goes, and the evictable leaf is
// looked up again after every eviction, since removing a leaf can turn its
// parent into one.
//
// Layout: flat node records in one vector, the nodes' tokens in one token
// arena (node i's block of tokens at [i * block_size, (i + 1) * block_size)),
// a hash index from (parent, token block) to node for the full-block walk,
// intrusive child lists for the partial match, and the leaves kept in a set
// ordered by (last use, block id).  Eviction walks that set from its least
// recently used end to the first leaf whose block only the tree still holds:
// the same leaf a full re-scan of the tree finds, without visiting every node.
//
// Readings of the section (where it leaves a step open): a node holds one
// full block; when no full block matches, the child sharing the longest run of
// leading tokens with the rest of the request is reused for those tokens
// (ties: the smaller block id); recency is a logical clock that advances once
// per match or insert and stamps every node the call walks; a leaf is
// evictable when the tree's reference is the last one; ties in recency go to
// the smaller block id; insert keeps an already cached block for the same
// tokens under the same parent.
#include <algorithm>
#include <mutex>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "internal.h"
#include "../../include/kshipra.h"

namespace {

struct Node {
  int32_t parent = -1;
  int32_t block = -1;
  int32_t first_child = -1, next_sibling = -1, prev_sibling = -1;
  int32_t num_children = 0;
  uint64_t stamp = 0;  // last use (logical clock)
  uint64_t key = 0;    // hash of (parent, token block)
};

// SplitMix64's finaliser (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators", 2014) as the mixing step of the key hash.
uint64_t mix64(uint64_t x) {
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}

}  // namespace

struct kshipra_prefix_cache {
  std::mutex mu;
  kshipra_block_pool* pool = nullptr;
  int bs = 0;
  uint64_t clock = 0;
  std::vector<Node> nodes;          // nodes[0] is the root (no block, no tokens)
  std::vector<int32_t> tokens;      // token arena
  std::vector<int32_t> free_nodes;  // node slots to reuse
  int32_t live = 0;                 // nodes other than the root
  std::unordered_multimap<uint64_t, int32_t> index;
  std::unordered_map<int32_t, int32_t> node_of_block;
  std::set<std::pair<uint64_t, int32_t>> leaves;  // (stamp, block), least recently used first

  uint64_t key_of(int32_t parent, const int32_t* toks) const {
    uint64_t h = mix64(static_cast<uint64_t>(static_cast<uint32_t>(parent)));
    for (int i = 0; i < bs; ++i) h = mix64(h ^ static_cast<uint32_t>(toks[i]));
    return h;
  }
  const int32_t* toks_of(int32_t n) const { return tokens.data() + static_cast<size_t>(n) * bs; }
  bool is_leaf(int32_t n) const { return n != 0 && nodes[n].num_children == 0; }

  // the child of `parent` whose token block is toks, or -1
  int32_t find_full(int32_t parent, const int32_t* toks) const {
    auto range = index.equal_range(key_of(parent, toks));
    for (auto it = range.first; it != range.second; ++it) {
      const int32_t c = it->second;
      if (nodes[c].parent != parent) continue;
      const int32_t* ct = toks_of(c);
      bool same = true;
      for (int i = 0; i < bs && same; ++i) same = ct[i] == toks[i];
      if (same) return c;
    }
    return -1;
  }

  void set_stamp(int32_t n, uint64_t s) {
    if (is_leaf(n)) {
      leaves.erase({nodes[n].stamp, nodes[n].block});
      leaves.insert({s, nodes[n].block});
    }
    nodes[n].stamp = s;
  }

  int32_t add_child(int32_t parent, const int32_t* toks, int32_t block) {
    int32_t c;
    if (!free_nodes.empty()) {
      c = free_nodes.back();
      free_nodes.pop_back();
    } else {
      c = static_cast<int32_t>(nodes.size());
      nodes.emplace_back();
      tokens.resize(tokens.size() + bs);
    }
    std::copy(toks, toks + bs, tokens.begin() + static_cast<size_t>(c) * bs);
    Node& n = nodes[c];
    n = Node{};
    n.parent = parent;
    n.block = block;
    n.key = key_of(parent, toks);
    Node& p = nodes[parent];
    if (parent != 0 && p.num_children == 0) leaves.erase({p.stamp, p.block});
    n.next_sibling = p.first_child;
    if (p.first_child >= 0) nodes[p.first_child].prev_sibling = c;
    p.first_child = c;
    ++p.num_children;
    index.emplace(n.key, c);
    node_of_block[block] = c;
    leaves.insert({n.stamp, block});
    ++live;
    return c;
  }

  // removes leaf n (its block reference is the caller's to drop)
  void remove_leaf(int32_t c) {
    Node& n = nodes[c];
    leaves.erase({n.stamp, n.block});
    auto range = index.equal_range(n.key);
    for (auto it = range.first; it != range.second; ++it)
      if (it->second == c) {
        index.erase(it);
        break;
      }
    node_of_block.erase(n.block);
    Node& p = nodes[n.parent];
    if (n.prev_sibling >= 0) nodes[n.prev_sibling].next_sibling = n.next_sibling;
    else p.first_child = n.next_sibling;
    if (n.next_sibling >= 0) nodes[n.next_sibling].prev_sibling = n.prev_sibling;
    if (--p.num_children == 0 && n.parent != 0) leaves.insert({p.stamp, p.block});
    n = Node{};
    free_nodes.push_back(c);
    --live;
  }
};

using kshipra::api_clear_error;
using kshipra::api_fail;

extern "C" {

int kshipra_prefix_cache_create(kshipra_block_pool* pool, int block_size, kshipra_prefix_cache** cache_out) {
  api_clear_error();
  if (!cache_out) return api_fail(KSHIPRA_ERR_INVALID_ARG, "cache_out is NULL");
  *cache_out = nullptr;
  if (!pool) return api_fail(KSHIPRA_ERR_INVALID_ARG, "pool is NULL");
  if (block_size <= 0) return api_fail(KSHIPRA_ERR_INVALID_ARG, "block_size %d must be positive", block_size);
  auto* c = new (std::nothrow) kshipra_prefix_cache;
  if (!c) return api_fail(KSHIPRA_ERR_INVALID_ARG, "out of host memory");
  c->pool = pool;
  c->bs = block_size;
  c->nodes.emplace_back();  // the root
  c->tokens.resize(block_size);
  *cache_out = c;
  return KSHIPRA_OK;
}

void kshipra_prefix_cache_destroy(kshipra_prefix_cache* cache) {
  if (!cache) return;
  {
    std::lock_guard<std::mutex> g(cache->mu);
    std::vector<int32_t> held;
    for (size_t i = 1; i < cache->nodes.size(); ++i)
      if (cache->nodes[i].block >= 0) held.push_back(cache->nodes[i].block);
    kshipra_block_release(cache->pool, held.data(), static_cast<int>(held.size()));
  }
  delete cache;
}

int kshipra_prefix_cache_match(kshipra_prefix_cache* cache, const int32_t* tokens, int num_tokens,
                               int32_t* blocks_out, int max_blocks, int* num_blocks_out, int* num_matched_out) {
  api_clear_error();
  if (!cache || num_tokens < 0 || (num_tokens > 0 && !tokens) || !num_blocks_out || !num_matched_out)
    return api_fail(KSHIPRA_ERR_INVALID_ARG, "bad prefix_cache_match arguments");
  std::lock_guard<std::mutex> g(cache->mu);
  const int bs = cache->bs;
  const int need = (num_tokens + bs - 1) / bs;
  if (max_blocks < need || (need > 0 && !blocks_out))
    return api_fail(KSHIPRA_ERR_INVALID_ARG, "blocks_out holds %d ids, %d may be returned", max_blocks, need);
  const uint64_t now = ++cache->clock;
  int32_t node = 0;
  int i = 0, nb = 0;
  while (num_tokens - i >= bs) {
    const int32_t c = cache->find_full(node, tokens + i);
    if (c < 0) break;
    blocks_out[nb++] = cache->nodes[c].block;
    cache->set_stamp(c, now);
    node = c;
    i += bs;
  }
  const int rest = std::min(bs, num_tokens - i);
  int32_t best = -1;
  int best_len = 0;
  for (int32_t c = cache->nodes[node].first_child; c >= 0 && rest > 0; c = cache->nodes[c].next_sibling) {
    const int32_t* ct = cache->toks_of(c);
    int len = 0;
    while (len < rest && ct[len] == tokens[i + len]) ++len;
    if (len > best_len || (len == best_len && len > 0 && cache->nodes[c].block < cache->nodes[best].block)) {
      best = c;
      best_len = len;
    }
  }
  if (best >= 0) {
    blocks_out[nb++] = cache->nodes[best].block;
    cache->set_stamp(best, now);
    i += best_len;
  }
  // the caller's references; every id is held by the tree, so this cannot fail
  const int rc = kshipra_block_share(cache->pool, blocks_out, nb);
  if (rc != KSHIPRA_OK) return rc;
  *num_blocks_out = nb;
  *num_matched_out = i;
  return KSHIPRA_OK;
}

int kshipra_prefix_cache_insert(kshipra_prefix_cache* cache, const int32_t* tokens, int num_tokens,
                                const int32_t* blocks, int num_blocks, int* num_added_out) {
  api_clear_error();
  if (!cache || num_tokens < 0 || (num_tokens > 0 && !tokens) || num_blocks < 0 || (num_blocks > 0 && !blocks))
    return api_fail(KSHIPRA_ERR_INVALID_ARG, "bad prefix_cache_insert arguments");
  std::lock_guard<std::mutex> g(cache->mu);
  const int bs = cache->bs;
  const int full = num_tokens / bs;
  if (num_blocks < full) return api_fail(KSHIPRA_ERR_INVALID_ARG, "%d full blocks of tokens, %d block ids", full, num_blocks);
  // check everything before changing anything
  std::vector<int32_t> fresh;
  for (int32_t j = 0, node = 0; j < full; ++j) {
    const int32_t c = node >= 0 ? cache->find_full(node, tokens + static_cast<size_t>(j) * bs) : -1;
    if (c < 0) {
      const int32_t b = blocks[j];
      bool dup = cache->node_of_block.count(b) != 0;
      for (int32_t f : fresh) dup = dup || f == b;
      if (dup || kshipra_block_refcount(cache->pool, b) <= 0)
        return api_fail(KSHIPRA_ERR_INVALID_ARG, "block %d is not allocated, or is cached already", b);
      fresh.push_back(b);
    }
    node = c;
  }
  // the tree's references
  int rc = kshipra_block_share(cache->pool, fresh.data(), static_cast<int>(fresh.size()));
  if (rc != KSHIPRA_OK) return rc;
  const uint64_t now = ++cache->clock;
  int32_t node = 0;
  for (int j = 0; j < full; ++j) {
    const int32_t* toks = tokens + static_cast<size_t>(j) * bs;
    int32_t c = cache->find_full(node, toks);
    if (c < 0) c = cache->add_child(node, toks, blocks[j]);
    cache->set_stamp(c, now);
    node = c;
  }
  if (num_added_out) *num_added_out = static_cast<int>(fresh.size());
  return KSHIPRA_OK;
}

int kshipra_prefix_cache_evict(kshipra_prefix_cache* cache, int num_blocks, int* num_freed_out) {
  api_clear_error();
  if (!cache || num_blocks < 0) return api_fail(KSHIPRA_ERR_INVALID_ARG, "bad prefix_cache_evict arguments");
  std::lock_guard<std::mutex> g(cache->mu);
  int freed = 0;
  while (freed < num_blocks) {
    // the least recently used leaf that only the tree still holds, found
    // again after every eviction (a removed leaf may leave its parent a leaf)
    int32_t victim = -1;
    for (const auto& e : cache->leaves)
      if (kshipra_block_refcount(cache->pool, e.second) == 1) {
        victim = e.second;
        break;
      }
    if (victim < 0) break;  // nothing evictable left
    cache->remove_leaf(cache->node_of_block.at(victim));
    const int rc = kshipra_block_release(cache->pool, &victim, 1);
    if (rc != KSHIPRA_OK) return rc;
    ++freed;
  }
  if (num_freed_out) *num_freed_out = freed;
  return KSHIPRA_OK;
}

int kshipra_prefix_cache_evictable(kshipra_prefix_cache* cache) {
  if (!cache) return -1;
  std::lock_guard<std::mutex> g(cache->mu);
  // children before parents: reverse of a depth-first preorder
  std::vector<int32_t> order, stack{0};
  while (!stack.empty()) {
    const int32_t n = stack.back();
    stack.pop_back();
    order.push_back(n);
    for (int32_t c = cache->nodes[n].first_child; c >= 0; c = cache->nodes[c].next_sibling) stack.push_back(c);
  }
  std::vector<char> whole(cache->nodes.size(), 1);
  int count = 0;
  for (auto it = order.rbegin(); it != order.rend(); ++it) {
    const int32_t n = *it;
    if (n == 0) break;
    bool w = kshipra_block_refcount(cache->pool, cache->nodes[n].block) == 1;
    for (int32_t c = cache->nodes[n].first_child; c >= 0 && w; c = cache->nodes[c].next_sibling) w = whole[c];
    whole[n] = w;
    count += w;
  }
  return count;
}

int kshipra_prefix_cache_num_nodes(kshipra_prefix_cache* cache) {
  if (!cache) return -1;
  std::lock_guard<std::mutex> g(cache->mu);
  return cache->live;
}

}  // extern "C"
