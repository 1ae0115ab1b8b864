// Chunked-prefill attention over the block arena on tcgen05 tensor cores.
//
// Pages "Building Kshipra" part 3 (kshipra-3), section 4: a prompt chunk of
// new tokens sits at absolute positions after the cached prefix; each query
// attends to the cached prefix and to the earlier tokens of its own chunk
// (causal mask); attention runs an online softmax over KV blocks read in
// place from the arena.  Section 1: keys of position p live in slot
// p % block_size of physical block block_tables[s][p / block_size].
//
// Query tiles: 128 rows = 128/G consecutive tokens x the G query heads of one
// kv head (GQA packing: every K/V tile serves all G heads).  A work item is a
// pair of adjacent query tiles (A, B) of one (sequence, kv head); both walk
// the same 128-key tiles, keys 0 .. (last position of the pair), so each K/V
// tile is fetched once for 256 query rows.  Key tiles past the pair's last
// position are never visited; tiles that cross a row's position are masked
// element by element.
//
// A small planning kernel lists the items with their cost (key tiles) and
// sorts them, heaviest first; the persistent attention kernel (one CTA per
// SM) walks that list in snake order.
//
// Roles in the attention kernel (576 threads):
//  - warp 16 (one lane): TMA producer.  Q_A and Q_B are 3-D boxes (token x head
//    x 64 columns); each K/V tile is 128 / block_size arena-block boxes
//    addressed through the block table, double-buffered.
//  - warp 17 (one lane): tcgen05.mma issuer, ping-pong between the tiles:
//    S_X = Q_X K^T (M 128, N 128, K d) into TMEM, then O_X += P_X V (M 128,
//    N d, K 128) with P_X read from TMEM (written over S_X by the softmax) and
//    V read MN-major in its arena layout.  While one tile's softmax runs, the
//    tensor core works on the other tile.
//  - warps 0-7 / 8-15: softmax of tile A / B.  Two threads own row r (TMEM
//    lane r), one per 64-key half: each loads its half of the S row, masks,
//    and they swap partial row maxima through shared memory (a 64-thread
//    named barrier per warp pair); each keeps a running sum (the reference
//    max is only raised when the row max passes it by 2^8, so O is rarely
//    rescaled), writes P as fp16/bf16 back into TMEM, and at the end of the
//    item normalises O and stores the output row.
// Fused step (q_raw set): Q_A / Q_B are loaded from the raw q; the softmax
// threads rotate them in place (each its half of its row) and the MMA issuer
// starts on "Q ready" instead of "Q landed".
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,256+d), O_B [384,384+d);
// P_X (two 16-bit values per column) occupies columns [0,32) and [64,96) of
// S_X, the first half of each softmax thread's own 64 S columns.
// Every wait is bounded (mbar_wait); on a timeout all roles stop, drain their
// outstanding copies / MMAs and release tensor memory.
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "rope.cuh"

namespace kshipra {
namespace {

constexpr int kTile = 128;  // query rows per tile and keys per key tile
constexpr int kThreads = 576;  // 16 softmax warps, producer, MMA issuer
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr float kNegInf = -INFINITY;

template <int D>
struct PrefillLayout {
  static constexpr int kRegions = D / 64;
  static constexpr int kRegionBytes = kTile * 128;  // 128 rows x 128 B
  static constexpr int kTileBytes = kRegions * kRegionBytes;
  static constexpr int kQA = 0;
  static constexpr int kQB = kQA + kTileBytes;
  static constexpr int kK = kQB + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kX = kV + kStages * kTileBytes;  // row max / sum exchange between half-row threads
  static constexpr int kXBytes = (2 * 2 * 2 + 2 * 2) * kTile * 4;
  static constexpr int kBar = kX + kXBytes;
  // q_full, q_empty, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2],
  // p_full[2], o_full[2], o_free[2], drain, q_ready; then the TMEM base address
  static constexpr int kNumBars = 20;
  static constexpr int kBytes = kBar + kNumBars * 8 + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

struct Bars {
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* k_full;   // [2]
  uint64_t* k_empty;  // [2]
  uint64_t* v_full;   // [2]
  uint64_t* v_empty;  // [2]
  uint64_t* s_full;   // [2] per query tile
  uint64_t* p_full;   // [2]
  uint64_t* o_full;   // [2]
  uint64_t* o_free;   // [2]
  uint64_t* drain;
  uint64_t* q_ready;  // fused step: both query tiles rotated (one arrival per softmax thread)
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Waits for a phase ignoring other CTAs' timeouts (used to drain own work).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < kWaitLimitNs) {
  }
}

// A wait whose outcome is the same for all 32 lanes, so that warp-collective
// instructions after it never run with lanes missing.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

// ---------------------------------------------------------------- work items
//
// The planning kernel lists one entry per (sequence, tile pair): cost (key
// tiles, 16 bits) | sequence (24) | tile pair (16); sorting the 64-bit values
// in descending order puts the most expensive first.  Work item i is entry
// i / Hkv for kv head i % Hkv (the cost does not depend on the head).

__host__ __device__ constexpr uint64_t entry_pack(uint32_t cost, uint32_t s, uint32_t pair) {
  return (static_cast<uint64_t>(cost) << 40) | (static_cast<uint64_t>(s) << 16) | pair;
}

struct Item {
  int s, pair, h;
};

__device__ __forceinline__ Item item_at(const uint64_t* entries, int i, int num_kv_heads) {
  const uint64_t v = entries[i / num_kv_heads];
  return Item{static_cast<int>((v >> 16) & 0xFFFFFF), static_cast<int>(v & 0xFFFF), i % num_kv_heads};
}

// Index of this CTA's r-th item (snake order over the sorted list).
__device__ __forceinline__ int item_index(int r, int nc) {
  return r * nc + ((r & 1) ? nc - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
}

struct PairGeom {
  int q0;        // first token of the sequence
  int tok_a;     // first token (sequence-relative) of tile A
  int n_a, n_b;  // valid tokens in tiles A and B (n_b may be 0)
  int nkeys;     // keys 0..nkeys-1 cover every row of the pair
  int ntiles;    // 128-key tiles (0 when the item's lengths are inconsistent)
};

template <int G>
__device__ __forceinline__ PairGeom pair_geom(const AttnArgs& a, int s, int pair) {
  constexpr int TQ = kTile / G;
  PairGeom p{};
  p.q0 = __ldg(a.query_start_loc + s);
  const int qlen = __ldg(a.query_start_loc + s + 1) - p.q0;
  p.tok_a = 2 * pair * TQ;
  p.n_a = min(TQ, qlen - p.tok_a);
  p.n_b = max(0, min(TQ, qlen - p.tok_a - TQ));
  const int ctx = __ldg(a.context_lens + s);
  const bool shape_ok = p.q0 >= 0 && p.q0 + qlen <= a.num_tokens && p.n_a > 0;
  const int pos_first = shape_ok ? __ldg(a.positions + p.q0 + p.tok_a) : -1;
  const int pos_last = shape_ok ? __ldg(a.positions + p.q0 + p.tok_a + p.n_a + p.n_b - 1) : -1;
  const bool ok = shape_ok && ctx > 0 && ctx <= a.max_blocks_per_seq * a.block_size && pos_first >= 0 &&
                  pos_first <= pos_last && pos_last < ctx;
  p.nkeys = ok ? pos_last + 1 : 0;
  p.ntiles = ceil_div(p.nkeys, kTile);
  return p;
}

// Lists one entry per (prefill sequence, tile pair) -- sequences with
// query_len x group rows above the decode threshold -- sorts them by cost
// (rank sort, entries are distinct) and writes them to entries[]; *count
// receives entries x num_kv_heads, the number of work items.  One CTA.
constexpr int kPlanThreads = 256;
constexpr int kSortCapacity = 1024;  // longer lists keep plan order

template <int G>
__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const AttnArgs a, uint64_t* entries,
                                                                     int* count, int max_entries) {
  constexpr int TQ = kTile / G;
  __shared__ uint64_t buf[kSortCapacity];
  __shared__ int warp_total[kPlanThreads / 32];
  __shared__ int base;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) base = 0;
  __syncthreads();
  for (int s0 = 0; s0 < a.num_seqs; s0 += kPlanThreads) {
    const int s = s0 + threadIdx.x;
    int pairs = 0, q0 = 0, qlen = 0;
    if (s < a.num_seqs) {
      q0 = __ldg(a.query_start_loc + s);
      qlen = __ldg(a.query_start_loc + s + 1) - q0;
      if (q0 >= 0 && qlen > 0 && q0 + qlen <= a.num_tokens && qlen * G > a.decode_max_rows)
        pairs = ceil_div(ceil_div(qlen, TQ), 2);
    }
    int incl = pairs;  // inclusive scan within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) warp_total[warp] = incl;
    __syncthreads();
    int before = base;
    for (int w = 0; w < warp; ++w) before += warp_total[w];
    int out = before + incl - pairs;
    for (int p = 0; p < pairs; ++p, ++out) {
      const int last = min(qlen, (2 * p + 2) * TQ) - 1;
      const int nkeys = __ldg(a.positions + q0 + last) + 1;
      const uint32_t cost = static_cast<uint32_t>(min(max(ceil_div(nkeys, kTile), 0), 0xFFFF));
      if (out >= max_entries) continue;
      const uint64_t v = entry_pack(cost, s, p);
      if (out < kSortCapacity) buf[out] = v;
      entries[out] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0)
      for (int w = 0; w < kPlanThreads / 32; ++w) base += warp_total[w];
    __syncthreads();
  }
  const int total = min(base, max_entries);
  if (total <= kSortCapacity) {
    for (int i = threadIdx.x; i < total; i += kPlanThreads) {
      const uint64_t v = buf[i];
      int rank = 0;
      for (int k = 0; k < total; ++k) rank += buf[k] > v;
      entries[rank] = v;
    }
  }
  if (threadIdx.x == 0) *count = total * a.num_kv_heads;
}

// ---------------------------------------------------------------- producer

template <int D, int G>
__device__ __forceinline__ void producer_role(const CUtensorMap* kmap, const CUtensorMap* vmap,
                                              const CUtensorMap* qmap, const AttnArgs& a, uint8_t* smem,
                                              const Bars& b, const uint64_t* items, int count, int nc) {
  using L = PrefillLayout<D>;
  constexpr int TQ = kTile / G;
  prefetch_tensormap(qmap);
  prefetch_tensormap(kmap);
  prefetch_tensormap(vmap);
  const int bs = a.block_size;
  const int blocks_per_tile = kTile / bs;
  const int oob_row = a.num_blocks * a.num_kv_heads * bs;  // past the tensor: zero fill
  int g = 0;                                               // key tiles issued by this CTA
  int items_done = 0;
  int issued_k0 = 0, issued_k1 = 0, issued_v0 = 0, issued_v1 = 0;  // last tile + 1 per stage
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = item_index(r, nc);
    if (idx >= count) break;
    const Item it = item_at(items, idx, a.num_kv_heads);
    const PairGeom p = pair_geom<G>(a, it.s, it.pair);
    if (p.ntiles == 0) {
      report(a.status, KSHIPRA_DEV_BAD_POSITION);
      continue;
    }
    if (items_done > 0 && !mbar_wait(b.q_empty, (items_done - 1) & 1, a.status)) { ok = false; break; }
    mbar_arrive_expect_tx(b.q_full, 2 * L::kTileBytes);  // zero-filled rows still count
#pragma unroll
    for (int reg = 0; reg < L::kRegions; ++reg) {
      tma_load_3d(smem + L::kQA + reg * L::kRegionBytes, qmap, 64 * reg, it.h * G, p.q0 + p.tok_a, b.q_full);
      tma_load_3d(smem + L::kQB + reg * L::kRegionBytes, qmap, 64 * reg, it.h * G, p.q0 + p.tok_a + TQ, b.q_full);
    }
    ++items_done;
    const int32_t* table = a.block_tables + static_cast<size_t>(it.s) * a.max_blocks_per_seq;
    for (int j = 0; j < p.ntiles; ++j, ++g) {
      const int st = g & 1, use = g >> 1;
      const int nb = ceil_div(min(kTile * (j + 1), p.nkeys) - kTile * j, bs);
      const uint32_t bytes = static_cast<uint32_t>(nb * bs * 128 * L::kRegions);
      int rows[kTile / 16];
#pragma unroll
      for (int i = 0; i < kTile / 16; ++i) {
        rows[i] = oob_row;
        if (i < nb) {
          const int blk = __ldg(table + j * blocks_per_tile + i);
          if (blk < 0 || blk >= a.num_blocks)
            report(a.status, KSHIPRA_DEV_BAD_BLOCK_ID);
          else
            rows[i] = (blk * a.num_kv_heads + it.h) * bs;
        }
      }
      if (g >= kStages && !mbar_wait(&b.k_empty[st], (use - 1) & 1, a.status)) { ok = false; break; }
      mbar_arrive_expect_tx(&b.k_full[st], bytes);
      uint8_t* kdst = smem + L::kK + st * L::kTileBytes;
#pragma unroll
      for (int i = 0; i < kTile / 16; ++i)
        if (i < nb)
#pragma unroll
          for (int reg = 0; reg < L::kRegions; ++reg)
            tma_load_2d(kdst + reg * L::kRegionBytes + i * bs * 128, kmap, 64 * reg, rows[i], &b.k_full[st]);
      (st ? issued_k1 : issued_k0) = g + 1;
      if (g >= kStages && !mbar_wait(&b.v_empty[st], (use - 1) & 1, a.status)) { ok = false; break; }
      mbar_arrive_expect_tx(&b.v_full[st], bytes);
      uint8_t* vdst = smem + L::kV + st * L::kTileBytes;
#pragma unroll
      for (int i = 0; i < kTile / 16; ++i)
        if (i < nb)
#pragma unroll
          for (int reg = 0; reg < L::kRegions; ++reg)
            tma_load_2d(vdst + reg * L::kRegionBytes + i * bs * 128, vmap, 64 * reg, rows[i], &b.v_full[st]);
      (st ? issued_v1 : issued_v0) = g + 1;
    }
  }
  if (!ok) {  // let every copy this thread started land before the CTA moves on
    if (items_done) drain_wait(b.q_full, (items_done - 1) & 1);
    if (issued_k0) drain_wait(&b.k_full[0], ((issued_k0 - 1) >> 1) & 1);
    if (issued_k1) drain_wait(&b.k_full[1], ((issued_k1 - 1) >> 1) & 1);
    if (issued_v0) drain_wait(&b.v_full[0], ((issued_v0 - 1) >> 1) & 1);
    if (issued_v1) drain_wait(&b.v_full[1], ((issued_v1 - 1) >> 1) & 1);
  }
}

// ---------------------------------------------------------------- MMA issuer

// Descriptor words of the tiles the MMA issuer streams over.  The low word
// carries the start address (16-byte units), so stepping along a tile adds a
// constant to it; the high word (stride offset, version, swizzle) is fixed.
struct Descs {
  uint32_t q_lo[2], k_lo[2], v_lo[2];  // per query tile / per stage
  uint32_t qk_hi, v_hi;
};

__device__ __forceinline__ uint32_t lo_word(uint64_t d) { return static_cast<uint32_t>(d); }
__device__ __forceinline__ uint32_t hi_word(uint64_t d) { return static_cast<uint32_t>(d >> 32); }

// S_x = Q_x K^T for the key tile in stage st, then signal s_full[x].
template <int D, bool kBf16>
__device__ __forceinline__ void issue_qk(const Descs& dd, const Bars& b, uint32_t tmem, int x, int st) {
  using L = PrefillLayout<D>;
  constexpr uint32_t kIdescQK = idesc_f16(kBf16, kTile, kTile, false, false);
  const uint32_t q_lo = x ? dd.q_lo[1] : dd.q_lo[0];
  const uint32_t k_lo = st ? dd.k_lo[1] : dd.k_lo[0];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = ((ks >> 2) * L::kRegionBytes + (ks & 3) * 32) >> 4;
    umma_f16_ss_w(tmem + kTile * x, q_lo + off, dd.qk_hi, k_lo + off, dd.qk_hi, kIdescQK, ks > 0 ? 1u : 0u);
  }
  umma_commit(&b.s_full[x]);
}

// O_x (+)= P_x V.  P_x is read from TMEM over S_x: keys 16 kk.. of step kk in
// columns 8 kk (kk < 4) or 8 kk + 32 (kk >= 4).  V is MN-major: 64-column
// halves L::kRegionBytes apart (leading offset), 8-key row groups 1024 B
// apart (stride offset).
template <int D, bool kBf16>
__device__ __forceinline__ void issue_pv(const Descs& dd, uint32_t tmem, int x, int st, bool accumulate) {
  constexpr uint32_t kIdescPV = idesc_f16(kBf16, kTile, D, false, true);
  const uint32_t v_lo = st ? dd.v_lo[1] : dd.v_lo[0];
  const uint32_t acc = accumulate ? 1u : 0u;
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk)
    umma_f16_ts_w(tmem + 2 * kTile + kTile * x, tmem + kTile * x + 8 * kk + (kk >= 4 ? 32 : 0),
                  v_lo + ((kk * 16 * 128) >> 4), dd.v_hi, kIdescPV, kk > 0 ? 1u : acc);
}

template <int D, bool kBf16, int G>
__device__ __forceinline__ void mma_role(const AttnArgs& a, uint8_t* smem, const Bars& b, uint32_t tmem,
                                         const uint64_t* items, int count, int nc) {
  using L = PrefillLayout<D>;
  const uint32_t sb = smem_u32(smem);
  Descs dd;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    dd.q_lo[i] = lo_word(smem_desc_sw128(sb + L::kQA + i * L::kTileBytes, 16, 1024));
    dd.k_lo[i] = lo_word(smem_desc_sw128(sb + L::kK + i * L::kTileBytes, 16, 1024));
    dd.v_lo[i] = lo_word(smem_desc_sw128(sb + L::kV + i * L::kTileBytes, L::kRegionBytes, 1024));
  }
  dd.qk_hi = hi_word(smem_desc_sw128(sb, 16, 1024));
  dd.v_hi = hi_word(smem_desc_sw128(sb, L::kRegionBytes, 1024));
  bool ok = true, issued_any = false;
  int g = 0, items_done = 0;

  for (int r = 0; ok; ++r) {
    const int idx = item_index(r, nc);
    if (idx >= count) break;
    const Item it = item_at(items, idx, a.num_kv_heads);
    const PairGeom p = pair_geom<G>(a, it.s, it.pair);
    const int n = p.ntiles;
    if (n == 0) continue;
    if (!mbar_wait(a.q_raw != nullptr ? b.q_ready : b.q_full, items_done & 1, a.status)) { ok = false; break; }
    // the previous item's epilogues must have read O_A / O_B before PV overwrites them
    const bool wait_o = items_done > 0;
    const int g0 = g;
    if (!mbar_wait(&b.k_full[g0 & 1], (g0 >> 1) & 1, a.status)) { ok = false; break; }
    tc_fence_after();
    issue_qk<D, kBf16>(dd, b, tmem, 0, g0 & 1);
    issue_qk<D, kBf16>(dd, b, tmem, 1, g0 & 1);
    issued_any = true;
    umma_commit(&b.k_empty[g0 & 1]);
    if (n == 1) umma_commit(b.q_empty);
    for (int j = 0; j < n && ok; ++j) {
      const int gt = g0 + j, st = gt & 1;
      // tile A: PV(j), then QK(j + 1)
      if (!mbar_wait(&b.p_full[0], gt & 1, a.status) || !mbar_wait(&b.v_full[st], (gt >> 1) & 1, a.status) ||
          (j == 0 && wait_o && !mbar_wait(&b.o_free[0], (items_done - 1) & 1, a.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_pv<D, kBf16>(dd, tmem, 0, st, j > 0);
      if (j + 1 < n) {
        const int st1 = (gt + 1) & 1;
        if (!mbar_wait(&b.k_full[st1], ((gt + 1) >> 1) & 1, a.status)) { ok = false; break; }
        tc_fence_after();
        issue_qk<D, kBf16>(dd, b, tmem, 0, st1);
      } else {
        umma_commit(&b.o_full[0]);
      }
      // tile B: PV(j), then QK(j + 1)
      if (!mbar_wait(&b.p_full[1], gt & 1, a.status) ||
          (j == 0 && wait_o && !mbar_wait(&b.o_free[1], (items_done - 1) & 1, a.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_pv<D, kBf16>(dd, tmem, 1, st, j > 0);
      umma_commit(&b.v_empty[st]);
      if (j + 1 < n) {
        const int st1 = (gt + 1) & 1;
        issue_qk<D, kBf16>(dd, b, tmem, 1, st1);
        umma_commit(&b.k_empty[st1]);
        if (j + 2 == n) umma_commit(b.q_empty);
      } else {
        umma_commit(&b.o_full[1]);
      }
    }
    g += n;
    ++items_done;
  }
  if (!ok && issued_any) {  // wait for this thread's MMAs before TMEM is released
    umma_commit(b.drain);
    drain_wait(b.drain, 0);
  }
}

// ---------------------------------------------------------------- softmax

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// Named barrier for the two warps that share a row range (same TMEM lanes).
__device__ __forceinline__ void pair_sync(int id) {
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

// Each row of tile x is handled by two threads: `half` 0 takes key columns
// 0-63 (and O columns 0..d/2-1), half 1 the other halves.  They exchange
// their partial row maxima every key tile and their partial sums at the end.
template <int D, bool kBf16, int G>
__device__ __forceinline__ void softmax_role(const AttnArgs& a, uint8_t* smem, const Bars& b, uint32_t tmem,
                                             const uint64_t* items, int count, int nc, int x, int half) {
  using L = PrefillLayout<D>;
  constexpr int TQ = kTile / G;
  constexpr int HC = kTile / 2;  // key columns per thread
  constexpr int HD = D / 2;      // O columns per thread
  // the reference maximum of the exponents is raised only when the row
  // maximum passes it by more than 2^8 (exp2 units): probabilities stay below
  // 2^8, well inside fp16/bf16 range, and O / l is unchanged
  constexpr float kRescaleThreshold = 8.f;
  const int quarter = (threadIdx.x >> 5) & 3;
  const int r = 32 * quarter + (threadIdx.x & 31);  // row of tile x = TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
  const uint32_t s_tmem = tmem + kTile * x + lane_off;
  const uint32_t o_tmem = tmem + 2 * kTile + kTile * x + lane_off + HD * half;
  const int bar_id = 1 + 4 * x + quarter;
  float* xmax = reinterpret_cast<float*>(smem + L::kX) + x * 2 * 2 * kTile;  // [parity][half][row]
  float* xsum = reinterpret_cast<float*>(smem + L::kX) + 2 * 2 * 2 * kTile + x * 2 * kTile;  // [half][row]
  const float c2 = a.scale_log2;
  const int tl = r / G, gg = r % G;
  int g = 0, items_done = 0;
  bool ok = true;

  for (int ri = 0; ok; ++ri) {
    const int idx = item_index(ri, nc);
    if (idx >= count) break;
    const Item it = item_at(items, idx, a.num_kv_heads);
    const PairGeom p = pair_geom<G>(a, it.s, it.pair);
    const int n = p.ntiles;
    if (n == 0) continue;
    const int nvalid = x == 0 ? p.n_a : p.n_b;
    const bool row_valid = tl < nvalid;
    // rows past the last token compute on whatever the tile holds, at the
    // position of the pair's last token, and are never stored
    const int tok = row_valid ? p.q0 + p.tok_a + TQ * x + tl : p.q0 + p.tok_a + p.n_a + p.n_b - 1;
    const int pos = __ldg(a.positions + tok);
    float m_ref = kNegInf, l = 0.f;
    if (a.q_raw != nullptr) {
      // fused step: this thread's half of row r of the raw Q_x, rotated in
      // place (the append kernel's float32 arithmetic, bit for bit).  Element
      // e pairs with e + D/2, so 16-byte chunk c (elements 8c .. 8c+7) pairs
      // with chunk c + D/16 of the same row; half h takes chunks h D/32 ..
      // (h + 1) D/32 - 1 and their partners.  The rows go to q_rot when asked,
      // and every thread reports to the MMA issuer, which starts on "Q ready".
      if (!warp_wait(b.q_full, items_done & 1, a.status)) { ok = false; break; }
      if (row_valid) {
        if (pos < 0 || pos >= a.rope_max_pos) {
          report(a.status, KSHIPRA_DEV_BAD_POSITION);
        } else {
          constexpr int kPairs = D / 16;
          uint8_t* qrow = smem + (x ? L::kQB : L::kQA) + r * 128;
          const float* cs = a.rope_table + static_cast<size_t>(pos) * D;
          uint4* qr = a.q_rot_out == nullptr
                          ? nullptr
                          : reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.q_rot_out) +
                                                     (static_cast<size_t>(tok) * a.num_q_heads + it.h * G + gg) * D);
#pragma unroll
          for (int k = 0; k < kPairs / 2; ++k) {
            const int c = half * (kPairs / 2) + k, cp = c + kPairs;
            uint4* lo = reinterpret_cast<uint4*>(qrow + (c >> 3) * L::kRegionBytes + (((c & 7) ^ (r & 7)) << 4));
            uint4* hi = reinterpret_cast<uint4*>(qrow + (cp >> 3) * L::kRegionBytes + (((cp & 7) ^ (r & 7)) << 4));
            uint4 ylo, yhi;
            rotate_eight_pairs_vals<kBf16>(*lo, *hi, cs + 16 * c, ylo, yhi);
            *lo = ylo;
            *hi = yhi;
            if (qr != nullptr) {
              qr[c] = ylo;
              qr[cp] = yhi;
            }
          }
        }
      }
      fence_proxy_async_smem();  // the rotated rows visible to the tensor core
      mbar_arrive(b.q_ready);
    }

    for (int j = 0; j < n; ++j) {
      const int gt = g + j;
      if (!warp_wait(&b.s_full[x], gt & 1, a.status)) { ok = false; break; }
      tc_fence_after();
      // pass 1: the half row's maximum over visible keys.  Only tiles that
      // cross some row's position (warp-uniform test) pay for the mask.
      const int kb0 = kTile * j + HC * half;
      const bool diag = __any_sync(0xffffffffu, kb0 + HC - 1 > pos);
      float m_tile;
      {
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = kNegInf;
#pragma unroll
        for (int cc = 0; cc < HC / 32; ++cc) {
          uint32_t t[32];
          tmem_ld32(s_tmem + HC * half + 32 * cc, t);
          if (diag) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              mx[i & 7] = fmaxf(mx[i & 7], kb0 + 32 * cc + i > pos ? kNegInf : __uint_as_float(t[i]));
          } else {  // three operands at a time
#pragma unroll
            for (int i = 0; i < 16; ++i)
              mx[i & 7] = fmax3(mx[i & 7], __uint_as_float(t[2 * i]), __uint_as_float(t[2 * i + 1]));
          }
        }
        m_tile = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      }
      float* xm = xmax + (gt & 1) * 2 * kTile;
      xm[half * kTile + r] = m_tile;
      pair_sync(bar_id);
      m_tile = fmaxf(m_tile, xm[(1 - half) * kTile + r]);  // both halves now hold the row maximum
      const bool raise = m_tile != kNegInf && (m_ref == kNegInf || (m_tile - m_ref) * c2 > kRescaleThreshold);
      float alpha = 1.f;
      if (raise) {
        alpha = ex2((m_ref - m_tile) * c2);  // 0 on the first visible tile
        m_ref = m_tile;
      }
      const float ms = (m_ref == kNegInf ? 0.f : m_ref) * c2;
      // pass 2, 32 keys at a time: probabilities, their sum, and P (two per
      // column) written over this half's own, already read, S columns:
      // keys 32 cc + [0, 32) of half h go to columns 64 h + 16 cc + [0, 16)
      float sums[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int cc = 0; cc < HC / 32; ++cc) {
        uint32_t t[32];
        tmem_ld32(s_tmem + HC * half + 32 * cc, t);
        uint32_t pk[16];
        if (diag) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int k0 = kb0 + 32 * cc + 2 * i;
            const float p0 = k0 > pos ? 0.f : ex2(fmaf(__uint_as_float(t[2 * i]), c2, -ms));
            const float p1 = k0 + 1 > pos ? 0.f : ex2(fmaf(__uint_as_float(t[2 * i + 1]), c2, -ms));
            sums[i & 3] += p0 + p1;
            pk[i] = pack2<kBf16>(p0, p1);
          }
        } else {  // scale-and-shift and the sums on packed pairs (f32x2)
          const uint64_t c2x2 = f2_pack(c2, c2), msx2 = f2_pack(-ms, -ms);
          uint64_t s2[2] = {0, 0};
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2_unpack(f2_fma(f2_bits(t[2 * i], t[2 * i + 1]), c2x2, msx2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            s2[i & 1] = f2_add(s2[i & 1], f2_pack(p0, p1));
            pk[i] = pack2<kBf16>(p0, p1);
          }
          float a0, a1, b0, b1;
          f2_unpack(s2[0], a0, a1);
          f2_unpack(s2[1], b0, b1);
          sums[0] += a0 + a1;
          sums[1] += b0 + b1;
        }
        tmem_st16(s_tmem + HC * half + 16 * cc, pk);
      }
      l = fmaf(l, alpha, (sums[0] + sums[1]) + (sums[2] + sums[3]));
      // PV of the previous key tile completed before S of this one (same
      // issuing thread, committed in order), so O can be rescaled here
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t t[32];
          tmem_ld32(o_tmem + 32 * c, t);
#pragma unroll
          for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
          tmem_st32(o_tmem + 32 * c, t);
        }
      }
      if (x == 0 && j == n - 1 && p.nkeys < kTile * j + kTile && half < L::kRegions) {
        // value rows past the last needed key may hold anything (even NaN,
        // or nothing loaded at all): zero them so that P = 0 contributes 0
        // (tile A's PV, the first to read this stage, waits for p_full[0])
        const int st = gt & 1;
        if (!warp_wait(&b.v_full[st], (gt >> 1) & 1, a.status)) { ok = false; break; }
        if (r >= p.nkeys - kTile * j) {
          const uint32_t vrow = smem_u32(smem + L::kV + st * L::kTileBytes) + half * L::kRegionBytes + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) st_shared_zero16(vrow + c * 16);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&b.p_full[x]);
    }
    if (!ok) break;
    g += n;
    xsum[half * kTile + r] = l;
    pair_sync(bar_id);
    l += xsum[(1 - half) * kTile + r];
    if (!warp_wait(&b.o_full[x], items_done & 1, a.status)) { ok = false; break; }
    tc_fence_after();
    const float inv = 1.f / l;
    uint16_t* dst = static_cast<uint16_t*>(a.out) +
                    (static_cast<size_t>(tok) * a.num_q_heads + it.h * G + gg) * D + HD * half;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      uint32_t t[32];
      tmem_ld32(o_tmem + 32 * c, t);
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack2<kBf16>(__uint_as_float(t[2 * i]) * inv, __uint_as_float(t[2 * i + 1]) * inv);
      if (row_valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
    }
    tc_fence_before();
    mbar_arrive(&b.o_free[x]);
    pair_sync(bar_id);  // the partner has read xsum before it is written again
    ++items_done;
  }
}

// ---------------------------------------------------------------- share

// CTAs of this grid that take items when the kernel runs beside the decode
// kernel of the same call (the same rule as the head_dim 128 kernel's): the
// decode kernel, bound by HBM bandwidth, keeps the 56 SMs whose CTAs hold
// the ~10 MB of loads in flight that full bandwidth needs (its head_dim 64
// CTAs are half as large, so four fit per SM), and the prefill items take
// the rest -- unless they would then outlast the decode kernel (key tiles of
// a tile pair at 4 us per tile and SM beside the decode traffic, against the
// decode-class sequences' K/V bytes at 6.5 TB/s), when they take every SM.
// All threads of the CTA take part; every CTA gets the same answer.
constexpr int kDecodeSms = 56;

template <int D, int G>
__device__ int share_ctas(const AttnArgs& a, const uint64_t* items, int count, int nc) {
  __shared__ long long part[2][kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long keys = 0, tiles = 0;
  for (int s = threadIdx.x; s < a.num_seqs; s += kThreads) {
    const int q0 = __ldg(a.query_start_loc + s), ctx = __ldg(a.context_lens + s);
    const int qlen = __ldg(a.query_start_loc + s + 1) - q0;
    if (qlen > 0 && qlen * G <= a.decode_max_rows && ctx > 0) keys += ctx;
  }
  const int entries = count / a.num_kv_heads;
  for (int i = threadIdx.x; i < entries; i += kThreads) tiles += static_cast<long long>(items[i] >> 40);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    keys += __shfl_xor_sync(0xffffffffu, keys, off);
    tiles += __shfl_xor_sync(0xffffffffu, tiles, off);
  }
  if (lane == 0) {
    part[0][warp] = keys;
    part[1][warp] = tiles;
  }
  __syncthreads();
  keys = tiles = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    keys += part[0][w];
    tiles += part[1][w];
  }
  const int k = nc - kDecodeSms;
  if (k < 1) return nc;
  const double decode_us = static_cast<double>(keys) * a.num_kv_heads * D * 4 / 6.5e6;
  const double prefill_us = 4.0 * static_cast<double>(tiles) * a.num_kv_heads / k;
  return prefill_us <= decode_us ? k : nc;
}

// ---------------------------------------------------------------- kernel

template <int D, bool kBf16, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap qmap, const AttnArgs a, const uint64_t* items,
                   const int* count_ptr) {
  using L = PrefillLayout<D>;
  const int count = *count_ptr;
  // CTAs that take items: all of them, or beside the decode kernel only
  // those the prefill items' share of the call needs
  const int nc = a.beside_decode ? share_ctas<D, G>(a, items, count, static_cast<int>(gridDim.x))
                                 : static_cast<int>(gridDim.x);
  if (static_cast<int>(blockIdx.x) >= min(count, nc)) return;  // no item for this CTA
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  const Bars b{bar,      bar + 1,  bar + 2,  bar + 4,  bar + 6, bar + 8,
               bar + 10, bar + 12, bar + 14, bar + 16, bar + 18, bar + 19};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + L::kNumBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(b.q_full, 1);
    mbar_init(b.q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.k_full[i], 1);
      mbar_init(&b.k_empty[i], 1);
      mbar_init(&b.v_full[i], 1);
      mbar_init(&b.v_empty[i], 1);
      mbar_init(&b.s_full[i], 1);
      mbar_init(&b.p_full[i], 2 * kTile);
      mbar_init(&b.o_full[i], 1);
      mbar_init(&b.o_free[i], 2 * kTile);
    }
    mbar_init(b.drain, 1);
    mbar_init(b.q_ready, 4 * kTile);  // every softmax thread of both tiles
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 16) {
    softmax_role<D, kBf16, G>(a, smem, b, tmem, items, count, nc, warp >> 3, (warp >> 2) & 1);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role<D, G>(&kmap, &vmap, &qmap, a, smem, b, items, count, nc);
  } else {
    if (lane == 0) mma_role<D, kBf16, G>(a, smem, b, tmem, items, count, nc);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kBf16, int G>
cudaError_t launch_prefill_t(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const CUtensorMap& qmap, cudaStream_t stream) {
  using L = PrefillLayout<D>;
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = set_smem_limit_once(prefill_kernel<D, kBf16, G>, L::kAlloc, configured);
  if (e != cudaSuccess) return e;
  prefill_plan_kernel<G><<<1, kPlanThreads, 0, stream>>>(a, a.ws_items, a.ws_item_count, a.max_items);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  prefill_kernel<D, kBf16, G><<<a.sm_count, kThreads, L::kAlloc, stream>>>(kmap, vmap, qmap, a, a.ws_items,
                                                                            a.ws_item_count);
  return cudaGetLastError();
}

template <int D, bool kBf16>
cudaError_t launch_prefill_g(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const CUtensorMap& qmap, cudaStream_t stream) {
  switch (a.group) {
    case 1: return launch_prefill_t<D, kBf16, 1>(a, kmap, vmap, qmap, stream);
    case 2: return launch_prefill_t<D, kBf16, 2>(a, kmap, vmap, qmap, stream);
    case 4: return launch_prefill_t<D, kBf16, 4>(a, kmap, vmap, qmap, stream);
    case 8: return launch_prefill_t<D, kBf16, 8>(a, kmap, vmap, qmap, stream);
    case 16: return launch_prefill_t<D, kBf16, 16>(a, kmap, vmap, qmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int prefill_max_items(int num_seqs, int num_tokens, int num_q_heads, int num_kv_heads) {
  const int G = num_q_heads / (num_kv_heads > 0 ? num_kv_heads : 1);
  const int pair_tokens = 2 * (kTile / (G > 0 ? G : 1));
  return (num_tokens + pair_tokens - 1) / pair_tokens + num_seqs;  // (sequence, tile pair) entries
}

cudaError_t launch_prefill(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& qmap, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.max_query_len * a.group <= a.decode_max_rows) return cudaSuccess;
  if (a.head_dim == 128) return launch_prefill_pair(a, kmap, vmap, qmap, stream);
  const bool bf = a.dtype == KSHIPRA_DTYPE_BF16;
  return bf ? launch_prefill_g<64, true>(a, kmap, vmap, qmap, stream)
            : launch_prefill_g<64, false>(a, kmap, vmap, qmap, stream);
}

}  // namespace kshipra
