// RoPE-and-append: rotates each new token's q and k at its absolute position
// and writes rotated K and raw V into the token's arena slot.
//
// Pages "Building Kshipra" part 3 (kshipra-3): section 1 (the block arena:
// the slot of position p is p % block_size in logical block p / block_size,
// reached through the sequence's block table; nothing is allocated per token)
// and section 4 (RoPE at absolute positions: a chunk after P cached tokens
// starts at position P).
//
// One CTA per token (or a few when a call has few tokens), so the token's
// sequence, position, table row and arena block are looked up once.  The
// token's work is cut into 16-byte units: a rotation unit rotates 8 pairs
// (i, i + d/2) of one q or k head row (rope.cuh: float32 from the caller's
// (cos, sin) table with separately rounded products and one add, then
// rounded once to the storage type, so the arena image is reproducible bit
// for bit; float32 keeps the step off GB300's slow FP64 units), a value unit
// copies 16 bytes of one V row.  Loads and stores are 16 bytes wide and a
// token's rows are contiguous, so the kernel streams q, k and v once.
#include "common.cuh"
#include "internal.h"
#include "rope.cuh"

namespace kshipra {
namespace {

constexpr int kAppendThreads = 128;

constexpr int kUnitsInFlight = 2;  // units a thread loads before any is stored

// Units of token blockIdx.x: rotation units of the q heads, then of the kv
// heads (k into the arena), then the value units; CTA blockIdx.y of
// gridDim.y takes every gridDim.y-th group of kAppendThreads units.  A
// thread first loads the sources of its first kUnitsInFlight units (they
// depend only on the token), then finds the token's sequence, position and
// arena block, then rotates and stores: the memory round trips overlap
// instead of following one another.
template <bool kBf16>
__global__ void __launch_bounds__(kAppendThreads, 16) append_rope_kernel(AppendArgs a) {
  // launched as a programmatic dependent of the previous grid on the stream:
  // wait for it before touching memory, then let the next grid (the step's
  // attention) start its own preparation.  In that order, the next grid
  // launches only once the previous one has completed, so it may read
  // anything but what this grid writes (the arena) before it waits
  grid_dependency_wait();
  grid_launch_dependents();
  const int t = blockIdx.x;
  if (t >= a.num_tokens) return;
  const int pos = __ldg(a.positions + t);
  const int D = a.head_dim, half = D / 2, groups = half / 8;
  const int nq = a.q != nullptr ? a.num_q_heads : 0;
  const int rot_units = (nq + a.num_kv_heads) * groups;
  const int units = rot_units + a.num_kv_heads * (D / 8);
  const int u0 = blockIdx.y * kAppendThreads + threadIdx.x, stride = gridDim.y * kAppendThreads;
  // source rows of unit u: q row, k row, or a 16-byte piece of a v row
  auto src_of = [&](int u, const uint16_t*& p) -> bool {  // true: rotation unit
    if (u < rot_units) {
      const int hh = u / groups;
      p = hh < nq ? static_cast<const uint16_t*>(a.q) + (static_cast<size_t>(t) * a.num_q_heads + hh) * D
                  : static_cast<const uint16_t*>(a.k) + (static_cast<size_t>(t) * a.num_kv_heads + hh - nq) * D;
      return true;
    }
    const int v = u - rot_units;
    p = static_cast<const uint16_t*>(a.v) + (static_cast<size_t>(t) * a.num_kv_heads + v / (D / 8)) * D +
        8 * (v % (D / 8));
    return false;
  };
  uint4 lo[kUnitsInFlight], hi[kUnitsInFlight];
#pragma unroll
  for (int j = 0; j < kUnitsInFlight; ++j) {
    const int u = u0 + j * stride;
    if (u < units) {
      const uint16_t* p;
      if (src_of(u, p)) {
        const int e = 8 * (u % groups);
        lo[j] = __ldg(reinterpret_cast<const uint4*>(p + e));
        hi[j] = __ldg(reinterpret_cast<const uint4*>(p + e + half));
      } else {
        lo[j] = __ldg(reinterpret_cast<const uint4*>(p));
      }
    }
  }
  const bool pos_ok = pos >= 0 && pos < a.rope_max_pos && pos / a.block_size < a.max_blocks_per_seq;
  const float* cs = a.rope_table + static_cast<size_t>(pos_ok ? pos : 0) * D;  // [d/2][2] for this position
  if (pos_ok && static_cast<int>(threadIdx.x) * 32 < D)  // the row's 128-byte lines into L1 for the units below
    asm volatile("prefetch.global.L1 [%0];" ::"l"(cs + threadIdx.x * 32));
  // sequence of token t: the last index s of query_start_loc[0..num_seqs]
  // with an entry <= t.  The entries do not decrease, so each round the CTA
  // loads up to kAppendThreads of them evenly spaced over the remaining
  // range and counts those <= t; two rounds cover 16 K sequences.  t lies in
  // sequence s unless no entry or the last one (the token count) is <= t.
  int lo_s = 0, width = a.num_seqs + 1;
  bool inside = true;
  while (width > 1) {
    const int step = (width + kAppendThreads - 1) / kAppendThreads;
    const int k = static_cast<int>(threadIdx.x);
    const bool le = k * step < width && __ldg(a.query_start_loc + lo_s + k * step) <= t;
    const int n = __syncthreads_count(le);
    if (n == 0) {  // before the first sequence
      inside = false;
      break;
    }
    lo_s += (n - 1) * step;
    width = min(step, width - (n - 1) * step);
  }
  const int s = lo_s;
  const bool first = blockIdx.y == 0 && threadIdx.x == 0;  // reports once per token
  if (!inside || s >= a.num_seqs) {  // outside every sequence
    if (first) report(a.status, KSHIPRA_DEV_BAD_LENGTHS);
    return;
  }
  if (!pos_ok) {
    if (first) report(a.status, KSHIPRA_DEV_BAD_POSITION);
    return;
  }
  const int blk = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + pos / a.block_size);
  const bool blk_ok = blk >= 0 && blk < a.num_blocks;
  if (!blk_ok && first) report(a.status, KSHIPRA_DEV_BAD_BLOCK_ID);
  const size_t slot = (static_cast<size_t>(blk) * a.num_kv_heads * a.block_size + pos % a.block_size) * D;
  // destination of unit u (nullptr: a kv unit with an invalid block)
  auto dst_of = [&](int u) -> uint16_t* {
    if (u < rot_units) {
      const int hh = u / groups;
      if (hh < nq) return static_cast<uint16_t*>(a.q_rot) + (static_cast<size_t>(t) * a.num_q_heads + hh) * D;
      return blk_ok ? static_cast<uint16_t*>(a.k_arena) + slot + static_cast<size_t>(hh - nq) * a.block_size * D
                    : nullptr;
    }
    const int v = u - rot_units;
    return blk_ok ? static_cast<uint16_t*>(a.v_arena) + slot + static_cast<size_t>(v / (D / 8)) * a.block_size * D +
                        8 * (v % (D / 8))
                  : nullptr;
  };
#pragma unroll
  for (int j = 0; j < kUnitsInFlight; ++j) {
    const int u = u0 + j * stride;
    if (u >= units) break;
    uint16_t* d = dst_of(u);
    if (d == nullptr) continue;
    if (u < rot_units)
      rotate_eight_pairs<kBf16>(lo[j], hi[j], d, 8 * (u % groups), half, cs);
    else
      *reinterpret_cast<uint4*>(d) = lo[j];
  }
  // shapes with more units than kUnitsInFlight per thread
  for (int u = u0 + kUnitsInFlight * stride; u < units; u += stride) {
    uint16_t* d = dst_of(u);
    if (d == nullptr) continue;
    const uint16_t* p;
    if (src_of(u, p)) {
      const int e = 8 * (u % groups);
      rotate_eight_pairs<kBf16>(__ldg(reinterpret_cast<const uint4*>(p + e)),
                           __ldg(reinterpret_cast<const uint4*>(p + e + half)), d, e, half, cs);
    } else {
      *reinterpret_cast<uint4*>(d) = __ldg(reinterpret_cast<const uint4*>(p));
    }
  }
}

}  // namespace

cudaError_t launch_append_rope(const AppendArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  const int heads = (a.q != nullptr ? a.num_q_heads : 0) + a.num_kv_heads;
  const int units = heads * (a.head_dim / 16) + a.num_kv_heads * (a.head_dim / 8);
  // a call with few tokens (a decode step) spreads each token over several
  // CTAs; a long one (a prefill chunk) keeps one CTA per token
  const int per_token = a.num_tokens >= 512 ? 1 : (units + kAppendThreads - 1) / kAppendThreads;
  dim3 grid(a.num_tokens, per_token), block(kAppendThreads);
  return a.dtype == KSHIPRA_DTYPE_BF16 ? launch_kernel(append_rope_kernel<true>, grid, block, 0, stream, true, a)
                                       : launch_kernel(append_rope_kernel<false>, grid, block, 0, stream, true, a);
}

}  // namespace kshipra
