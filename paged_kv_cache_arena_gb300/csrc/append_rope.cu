// RoPE-and-append: rotates each new token's q and k at its absolute position
// and writes rotated K and raw V into the token's arena slot.
//
// Pages "Building Kshipra" part 3 (kshipra-3): section 1 (the block arena:
// the slot of position p is p % block_size in logical block p / block_size,
// reached through the sequence's block table; nothing is allocated per token)
// and section 4 (RoPE at absolute positions: a chunk after P cached tokens
// starts at position P).
//
// One warp per (token, head).  The rotation (rope.cuh) is done in float32 from
// the caller's (cos, sin) table with separately rounded products and one add,
// then rounded once to the storage type, so the arena image is reproducible
// bit for bit.  (float32 keeps the step off GB300's slow FP64 units.)  The
// volume is small (num_tokens x (Hq + Hkv) x head_dim elements per call); the
// kernel is memory-latency bound and far from the hot path's cost.
#include "common.cuh"
#include "internal.h"
#include "rope.cuh"

namespace kshipra {
namespace {

constexpr int kAppendWarps = 4;
constexpr int kAppendThreads = 32 * kAppendWarps;

// One warp per (token, head): warps of blockIdx.y cover q heads first, then
// kv heads (k rotated into the arena, v copied).  Lane i rotates pairs 2i and
// 2i + 1; with head_dim 64 the upper half of the warp idles.
template <bool kBf16>
__global__ void __launch_bounds__(kAppendThreads) append_rope_kernel(AppendArgs a) {
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = a.q != nullptr ? a.num_q_heads : 0;
  const int hh = blockIdx.y * kAppendWarps + warp;  // head slot: [0, nq) q heads, then kv heads
  if (t >= a.num_tokens || hh >= nq + a.num_kv_heads) return;
  // sequence of token t: the last s with query_start_loc[s] <= t
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.query_start_loc + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  const int s = lo;
  const bool first = blockIdx.y == 0 && threadIdx.x == 0;  // reports once per token
  if (t < __ldg(a.query_start_loc + s) || t >= __ldg(a.query_start_loc + s + 1)) {  // outside every sequence
    if (first) report(a.status, KSHIPRA_DEV_BAD_LENGTHS);
    return;
  }
  const int pos = __ldg(a.positions + t);
  if (pos < 0 || pos >= a.rope_max_pos || pos / a.block_size >= a.max_blocks_per_seq) {
    if (first) report(a.status, KSHIPRA_DEV_BAD_POSITION);
    return;
  }
  const int D = a.head_dim, half = D / 2;
  const float* cs = a.rope_table + static_cast<size_t>(pos) * D;  // [d/2][2] for this position
  const int i = 2 * lane;                                           // first pair of this lane
  if (hh < nq) {
    const size_t row = (static_cast<size_t>(t) * a.num_q_heads + hh) * D;
    if (i < half)
      rotate_two_pairs<kBf16>(static_cast<const uint16_t*>(a.q) + row, static_cast<uint16_t*>(a.q_rot) + row, i,
                              half, cs);
    return;
  }
  const int h = hh - nq;
  const int blk = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + pos / a.block_size);
  if (blk < 0 || blk >= a.num_blocks) {
    if (lane == 0) report(a.status, KSHIPRA_DEV_BAD_BLOCK_ID);
    return;
  }
  const size_t src = (static_cast<size_t>(t) * a.num_kv_heads + h) * D;
  const size_t dst = ((static_cast<size_t>(blk) * a.num_kv_heads + h) * a.block_size + pos % a.block_size) * D;
  if (i < half)
    rotate_two_pairs<kBf16>(static_cast<const uint16_t*>(a.k) + src, static_cast<uint16_t*>(a.k_arena) + dst, i,
                            half, cs);
  if (lane < D / 8)  // value row: bit copy in 16-byte pieces
    reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.v_arena) + dst)[lane] =
        reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.v) + src)[lane];
}

}  // namespace

cudaError_t launch_append_rope(const AppendArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  const int heads = (a.q != nullptr ? a.num_q_heads : 0) + a.num_kv_heads;
  dim3 grid(a.num_tokens, (heads + kAppendWarps - 1) / kAppendWarps), block(kAppendThreads);
  if (a.dtype == KSHIPRA_DTYPE_BF16)
    append_rope_kernel<true><<<grid, block, 0, stream>>>(a);
  else
    append_rope_kernel<false><<<grid, block, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kshipra
