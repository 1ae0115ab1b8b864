// Block management around the arena: the LIFO block pool with reference
// counts and copy-on-write, and the kernel that moves whole blocks (the
// copy-on-write copy, and swapping a preempted sequence's blocks out to
// pinned host memory and back in).
//
// Pages "Building Kshipra" part 3 (kshipra-3): section 1 (the arena is
// reserved once; a LIFO free list, initially 0 .. n-1, hands out the highest
// id first and reuses the most recently freed block first), section 3
// (reference counts keep shared prefix blocks alive; a block is copied before
// a request that diverges inside it writes it), section 5 (a preempted
// sequence's blocks are swapped out of the arena and restored later instead
// of recomputed).
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

// ---------------------------------------------------------------- host pool

struct kshipra_block_pool {
  std::mutex mu;
  std::vector<int32_t> free_list;  // back = next allocation
  std::vector<int32_t> refs;       // 0 = free
};

namespace kshipra {
namespace {

// ---------------------------------------------------------------- block move
//
// One CTA per (block i, group of kMoveHeads kv heads): moves the group's
// bs x d tiles of K and of V from src to dst.  The group's 16-byte vectors
// are walked kMoveInFlight per thread at a time, every load of a round issued
// before its stores, so that each thread keeps several loads in flight (the
// copy is bound by memory latency x bytes in flight, over HBM and even more
// over the CPU-GPU link).  Each side is either the arena (block id from its
// id list, layout [blocks][Hkv][bs][d]) or a dense buffer [n][Hkv][bs][d]
// indexed by i (ids == nullptr), which may be pinned host memory reached over
// the CPU-GPU link.  Ids outside the arena are reported and skipped.
// Launched as a programmatic dependent of the previous grid, it waits for it
// before touching memory.
constexpr int kMoveThreads = 256;
constexpr int kMoveHeads = 4;
constexpr int kMoveInFlight = 2;  // vectors of K (and of V) per thread per round

__global__ void __launch_bounds__(kMoveThreads) block_move_kernel(uint4* dst_k, uint4* dst_v, const int32_t* dst_ids,
                                                                  const uint4* src_k, const uint4* src_v,
                                                                  const int32_t* src_ids, int num_kv_heads,
                                                                  int tile_vec, int num_blocks, unsigned* status) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int i = blockIdx.x, h0 = blockIdx.y * kMoveHeads;
  const int sb = src_ids ? __ldg(src_ids + i) : i;
  const int db = dst_ids ? __ldg(dst_ids + i) : i;
  if ((src_ids && (sb < 0 || sb >= num_blocks)) || (dst_ids && (db < 0 || db >= num_blocks))) {
    if (blockIdx.y == 0 && threadIdx.x == 0) report(status, KSHIPRA_DEV_BAD_BLOCK_ID);
    return;
  }
  // the group's tiles are contiguous on both sides: heads h0 .. h0 + nh - 1
  const int nh = min(kMoveHeads, num_kv_heads - h0);
  const int total = nh * tile_vec;
  const size_t s0 = (static_cast<size_t>(sb) * num_kv_heads + h0) * tile_vec;
  const size_t d0 = (static_cast<size_t>(db) * num_kv_heads + h0) * tile_vec;
  for (int base = threadIdx.x; base < total; base += kMoveThreads * kMoveInFlight) {
    uint4 kv[kMoveInFlight], vv[kMoveInFlight];
#pragma unroll
    for (int u = 0; u < kMoveInFlight; ++u) {
      const int j = base + u * kMoveThreads;
      if (j < total) {
        kv[u] = src_k[s0 + j];
        vv[u] = src_v[s0 + j];
      }
    }
#pragma unroll
    for (int u = 0; u < kMoveInFlight; ++u) {
      const int j = base + u * kMoveThreads;
      if (j < total) {
        dst_k[d0 + j] = kv[u];
        dst_v[d0 + j] = vv[u];
      }
    }
  }
}

// The address a kernel uses for p: p itself for device (or managed) memory,
// the device alias of host memory the CUDA runtime has pinned; nullptr for
// anything else (pageable host memory).
const void* device_address(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return p;
  if (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr)
    return static_cast<const char*>(at.devicePointer) +
           (static_cast<const char*>(p) - static_cast<const char*>(at.hostPointer));
  return nullptr;
}

int move_blocks(void* dst_k, void* dst_v, const int32_t* dst_ids, const void* src_k, const void* src_v,
                const int32_t* src_ids, int n, int num_kv_heads, int block_size, int head_dim, int num_blocks,
                int dtype, void* stream, const char* what) {
  if (n < 0) return api_fail(KSHIPRA_ERR_INVALID_ARG, "%s: negative block count", what);
  if (num_kv_heads <= 0 || num_blocks <= 0) return api_fail(KSHIPRA_ERR_INVALID_ARG, "%s: bad arena shape", what);
  if (head_dim != 64 && head_dim != 128) return api_fail(KSHIPRA_ERR_UNSUPPORTED, "%s: head_dim %d", what, head_dim);
  if (block_size != 16 && block_size != 32)
    return api_fail(KSHIPRA_ERR_UNSUPPORTED, "%s: block_size %d", what, block_size);
  if (dtype != KSHIPRA_DTYPE_F16 && dtype != KSHIPRA_DTYPE_BF16)
    return api_fail(KSHIPRA_ERR_UNSUPPORTED, "%s: dtype %d", what, dtype);
  if (n == 0) return KSHIPRA_OK;
  const void* ptrs[] = {dst_k, dst_v, src_k, src_v};
  for (const void* p : ptrs) {
    if (!p) return api_fail(KSHIPRA_ERR_INVALID_ARG, "%s: a required pointer is NULL", what);
    if (reinterpret_cast<uintptr_t>(p) % 16) return api_fail(KSHIPRA_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", what);
  }
  const void* dev[4];
  for (int i = 0; i < 4; ++i)
    if (!(dev[i] = device_address(ptrs[i])))
      return api_fail(KSHIPRA_ERR_INVALID_ARG, "%s: buffers must be device memory or pinned host memory", what);
  unsigned* status = nullptr;
  cudaError_t e = api_status_ptr(&status);
  if (e != cudaSuccess) return api_cuda_fail(e, "status word");
  const int tile_vec = block_size * head_dim * 2 / 16;
  dim3 grid(n, (num_kv_heads + kMoveHeads - 1) / kMoveHeads);
  e = launch_kernel(block_move_kernel, grid, dim3(kMoveThreads), 0, static_cast<cudaStream_t>(stream), true,
                    static_cast<uint4*>(const_cast<void*>(dev[0])), static_cast<uint4*>(const_cast<void*>(dev[1])),
                    dst_ids, static_cast<const uint4*>(dev[2]), static_cast<const uint4*>(dev[3]), src_ids,
                    num_kv_heads, tile_vec, num_blocks, status);
  if (e != cudaSuccess) return api_cuda_fail(e, "block move kernel launch");
  return KSHIPRA_OK;
}

}  // namespace
}  // namespace kshipra

using namespace kshipra;

extern "C" {

int kshipra_block_pool_create(int num_blocks, kshipra_block_pool** pool_out) {
  api_clear_error();
  if (!pool_out) return api_fail(KSHIPRA_ERR_INVALID_ARG, "pool_out is NULL");
  *pool_out = nullptr;
  if (num_blocks <= 0) return api_fail(KSHIPRA_ERR_INVALID_ARG, "num_blocks %d must be positive", num_blocks);
  auto* p = new (std::nothrow) kshipra_block_pool;
  if (!p) return api_fail(KSHIPRA_ERR_INVALID_ARG, "out of host memory");
  p->free_list.resize(num_blocks);
  for (int i = 0; i < num_blocks; ++i) p->free_list[i] = i;  // pop() takes the highest id first
  p->refs.assign(num_blocks, 0);
  *pool_out = p;
  return KSHIPRA_OK;
}

void kshipra_block_pool_destroy(kshipra_block_pool* pool) { delete pool; }

int kshipra_block_pool_num_free(kshipra_block_pool* pool) {
  if (!pool) return -1;
  std::lock_guard<std::mutex> g(pool->mu);
  return static_cast<int>(pool->free_list.size());
}

int kshipra_block_alloc(kshipra_block_pool* pool, int n, int32_t* ids_out) {
  api_clear_error();
  if (!pool || (n > 0 && !ids_out) || n < 0) return api_fail(KSHIPRA_ERR_INVALID_ARG, "bad block_alloc arguments");
  std::lock_guard<std::mutex> g(pool->mu);
  if (static_cast<size_t>(n) > pool->free_list.size())
    return api_fail(KSHIPRA_ERR_OUT_OF_BLOCKS, "%d blocks requested, %zu free", n, pool->free_list.size());
  for (int i = 0; i < n; ++i) {
    const int32_t id = pool->free_list.back();
    pool->free_list.pop_back();
    pool->refs[id] = 1;
    ids_out[i] = id;
  }
  return KSHIPRA_OK;
}

int kshipra_block_share(kshipra_block_pool* pool, const int32_t* ids, int n) {
  api_clear_error();
  if (!pool || (n > 0 && !ids) || n < 0) return api_fail(KSHIPRA_ERR_INVALID_ARG, "bad block_share arguments");
  std::lock_guard<std::mutex> g(pool->mu);
  const int nb = static_cast<int>(pool->refs.size());
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= nb || pool->refs[ids[i]] == 0)
      return api_fail(KSHIPRA_ERR_INVALID_ARG, "block %d is not allocated", ids[i]);
  for (int i = 0; i < n; ++i) ++pool->refs[ids[i]];
  return KSHIPRA_OK;
}

int kshipra_block_release(kshipra_block_pool* pool, const int32_t* ids, int n) {
  api_clear_error();
  if (!pool || (n > 0 && !ids) || n < 0) return api_fail(KSHIPRA_ERR_INVALID_ARG, "bad block_release arguments");
  std::lock_guard<std::mutex> g(pool->mu);
  const int nb = static_cast<int>(pool->refs.size());
  // validate against the counts as they will be after the earlier entries
  std::vector<int32_t> pending;
  for (int i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= nb) return api_fail(KSHIPRA_ERR_INVALID_ARG, "block %d is outside the pool", ids[i]);
    int seen = 0;
    for (int32_t q : pending) seen += q == ids[i];
    if (pool->refs[ids[i]] - seen <= 0) return api_fail(KSHIPRA_ERR_INVALID_ARG, "block %d is not allocated", ids[i]);
    pending.push_back(ids[i]);
  }
  for (int i = 0; i < n; ++i)
    if (--pool->refs[ids[i]] == 0) pool->free_list.push_back(ids[i]);  // the next allocation reuses it
  return KSHIPRA_OK;
}

int kshipra_block_refcount(kshipra_block_pool* pool, int id) {
  if (!pool) return -1;
  std::lock_guard<std::mutex> g(pool->mu);
  if (id < 0 || id >= static_cast<int>(pool->refs.size())) return -1;
  return pool->refs[id];
}

int kshipra_block_make_private(kshipra_block_pool* pool, int32_t* id_inout, int32_t* copy_from_out) {
  api_clear_error();
  if (!pool || !id_inout || !copy_from_out) return api_fail(KSHIPRA_ERR_INVALID_ARG, "bad make_private arguments");
  std::lock_guard<std::mutex> g(pool->mu);
  const int32_t id = *id_inout;
  if (id < 0 || id >= static_cast<int>(pool->refs.size()) || pool->refs[id] == 0)
    return api_fail(KSHIPRA_ERR_INVALID_ARG, "block %d is not allocated", id);
  *copy_from_out = -1;
  if (pool->refs[id] == 1) return KSHIPRA_OK;  // already private: write in place
  if (pool->free_list.empty()) return api_fail(KSHIPRA_ERR_OUT_OF_BLOCKS, "no free block for the copy");
  const int32_t fresh = pool->free_list.back();
  pool->free_list.pop_back();
  pool->refs[fresh] = 1;
  --pool->refs[id];  // the other holders keep the shared block
  *id_inout = fresh;
  *copy_from_out = id;
  return KSHIPRA_OK;
}

int kshipra_blocks_copy(void* k_arena, void* v_arena, const int32_t* src_ids, const int32_t* dst_ids, int n,
                        int num_kv_heads, int block_size, int head_dim, int num_blocks, int dtype, void* stream) {
  api_clear_error();
  if (n > 0 && (!src_ids || !dst_ids)) return api_fail(KSHIPRA_ERR_INVALID_ARG, "blocks_copy: id lists are NULL");
  return move_blocks(k_arena, v_arena, dst_ids, k_arena, v_arena, src_ids, n, num_kv_heads, block_size, head_dim,
                     num_blocks, dtype, stream, "blocks_copy");
}

int kshipra_blocks_swap_out(void* k_out, void* v_out, const void* k_arena, const void* v_arena, const int32_t* ids,
                            int n, int num_kv_heads, int block_size, int head_dim, int num_blocks, int dtype,
                            void* stream) {
  api_clear_error();
  if (n > 0 && !ids) return api_fail(KSHIPRA_ERR_INVALID_ARG, "blocks_swap_out: ids is NULL");
  return move_blocks(k_out, v_out, nullptr, k_arena, v_arena, ids, n, num_kv_heads, block_size, head_dim, num_blocks,
                     dtype, stream, "blocks_swap_out");
}

int kshipra_blocks_swap_in(void* k_arena, void* v_arena, const void* k_in, const void* v_in, const int32_t* ids,
                           int n, int num_kv_heads, int block_size, int head_dim, int num_blocks, int dtype,
                           void* stream) {
  api_clear_error();
  if (n > 0 && !ids) return api_fail(KSHIPRA_ERR_INVALID_ARG, "blocks_swap_in: ids is NULL");
  return move_blocks(k_arena, v_arena, ids, k_in, v_in, nullptr, n, num_kv_heads, block_size, head_dim, num_blocks,
                     dtype, stream, "blocks_swap_in");
}

}  // extern "C"
