// Chunked-prefill attention over the block arena on CTA pairs (tcgen05
// cta_group::2), head_dim 128.
//
// Pages "Building Kshipra" part 3 (kshipra-3), section 4: a prompt chunk of
// new tokens sits at absolute positions after the cached prefix; each query
// attends to the cached prefix and to the earlier tokens of its own chunk
// (causal mask); attention runs an online softmax over KV blocks read in
// place from the arena.  Section 1: keys of position p live in slot
// p % block_size of physical block block_tables[s][p / block_size].
//
// Query tiles: 128 rows = 128/G consecutive tokens x the G query heads of one
// kv head (GQA packing).  A work item is a quad of adjacent query tiles of
// one (sequence, kv head), run by a cluster of two CTAs on neighbouring SMs:
// CTA r holds tiles 4q + 2r (its "A") and 4q + 2r + 1 (its "B").  The leader
// CTA issues M = 256 MMAs that cover both CTAs' A rows (or B rows) at once,
// so every 128-key K/V tile serves 512 query rows while each SM stages only
// half of it: CTA r loads keys 64r .. 64r+63 of each K tile (the columns of
// S split between the pair) and columns 64r .. 64r+63 of each V tile (the
// columns of O).  Loading K/V from L2 is what bounds a one-CTA version of
// this kernel on GB300; halving it per SM leaves the tensor core as the
// limit.
//
// Roles (352 threads per CTA):
//  - warp 8: TMA producer, 16 lanes issuing at once.  Q_A / Q_B as 3-D boxes
//    (token x head x 64 columns); this CTA's halves of each K/V tile as
//    arena-block boxes through the block table, three stages.  Completion is
//    counted on the leader's barriers, except the last V tile of an item,
//    which completes on a barrier of its own CTA so the softmax warps can
//    zero its tail.
//  - warps 9 / 10 (one lane each, leader only): MMA issuers of tiles A / B.
//    S_X = Q_X K^T (M 256, N 128, K 128) into TMEM; O_X += P_X V (M 256,
//    N 128, K 128) with P_X from shared memory.  The next key tile's S_X is
//    issued as soon as the softmax has read the current one, so scores and
//    softmax overlap within a tile; with an issuer per tile neither tile's
//    pipeline waits on the other's softmax.  Commits arrive on both CTAs'
//    barriers.
//  - warps 0-3 / 4-7: softmax of tile A / B of their own CTA, one thread per
//    row: the whole S row is read into registers once; P goes to shared
//    memory in the MMA's operand layout; each warp reports "S read", "P
//    ready" and "O read" to the leader with one remote arrival.  The
//    epilogue stages O / l in the tile's P buffer and each warp then writes
//    whole output rows (two per store instruction), as does the fused step's
//    q_rot store from Q_x.
// TMEM (each CTA): S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
// Fused step (q_raw set): Q_A / Q_B are loaded from the raw (unrotated) q
// and land on a barrier of their own CTA; each softmax thread rotates its row
// in shared memory (the append kernel's float32 arithmetic, bit for bit),
// optionally stores it to q_rot, and the MMA issuers start on "Q ready"
// instead of "Q landed".  Launched as a programmatic dependent of the step's
// K/V append, the kernel plans its work, loads and rotates Q and reads the
// cached-prefix key tiles while the append finishes, and waits for it only
// before the first key tile that reaches the sequence's new positions.
// Every wait is bounded; on a timeout all roles stop and drain their own
// outstanding copies / MMAs before the pair releases tensor memory.
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "rope.cuh"

namespace kshipra {
namespace {

constexpr int kTile = 128;  // query rows per tile and keys per key tile
constexpr int kD = 128;
constexpr int kThreads = 352;  // 8 softmax warps, producer warp, two MMA warps
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;  // and 10: the issuers of tiles A and B (leader); warp 9 also holds TMEM
constexpr int kStages = 3;           // K/V stages
constexpr int kSortCapacity = 128;   // work-list entries the kernel plans for itself
constexpr uint32_t kTmemCols = 512;
constexpr float kNegInf = -INFINITY;

struct Layout {
  static constexpr int kQRegion = kTile * 128;  // 128 rows x 64 columns (128-byte swizzle)
  static constexpr int kQTile = 2 * kQRegion;   // 32 KB
  static constexpr int kKRegion = 64 * 128;     // this CTA's 64 keys x 64 columns
  static constexpr int kKStage = 2 * kKRegion;  // 16 KB
  static constexpr int kVStage = kTile * 128;   // 128 keys x this CTA's 64 columns, 16 KB
  static constexpr int kPTile = 2 * kQRegion;   // P: 128 rows x 128 keys, K-major, 128-byte swizzle
  static constexpr int kQA = 0;
  static constexpr int kQB = kQA + kQTile;
  static constexpr int kPA = kQB + kQTile;
  static constexpr int kPB = kPA + kPTile;
  static constexpr int kK = kPB + kPTile;
  static constexpr int kV = kK + kStages * kKStage;
  static constexpr int kBar = kV + kStages * kVStage;
  static constexpr int kNumBars = 2 + 4 * kStages + 14 + 2 + 3;
  static constexpr int kPlan = kBar + kNumBars * 8 + 16;  // work list planned in the kernel
  static constexpr int kPlanSorted = kPlan;                 // [kSortCapacity] sorted entries
  static constexpr int kPlanBuf = kPlanSorted + kSortCapacity * 8;  // [kSortCapacity] listed entries
  static constexpr int kPlanWarp = kPlanBuf + kSortCapacity * 8;   // per-warp totals, running base
  static constexpr int kShare = kPlanWarp + 64;                     // [2 x 11] per-warp sums of the share
  static constexpr int kBytes = kShare + 2 * 11 * 8;
  // the dynamic shared memory of a kernel without static shared variables
  // starts at the base of the CTA's window (1024-aligned, checked at run time)
  static constexpr int kAlloc = kBytes;
};
static_assert(Layout::kAlloc <= 227 * 1024, "shared memory");

struct Bars {
  uint64_t* q_full;    // leader: both CTAs' Q tiles landed
  uint64_t* q_empty;   // both: the item's last QK MMAs completed (one arrival per issuer)
  uint64_t* kv_full;   // [kStages] leader: both CTAs' K (and V, but for an item's last tile) landed
  uint64_t* kv_empty;  // [kStages] both: the stage's PV MMAs completed (one arrival per issuer)
  uint64_t* v_last;    // [kStages] own CTA: one phase per use of the stage; an item's
                       // last V tile lands here (other uses complete it at once)
  uint64_t* v_zeroed;  // [kStages] leader, 8 warp arrivals (tile A's softmax warps) per use of
                       // the stage: the V rows past an item's last key are zeroed in both CTAs
  uint64_t* s_full;    // [2] both: S_x ready in TMEM
  uint64_t* s_free;    // [2] leader, 8 warp arrivals (4 per CTA): S_x read, its columns free
  uint64_t* p_full;    // [2] leader, 8 warp arrivals: P_x written to shared memory
  uint64_t* p_free;    // [2][2] both: the PV MMAs reading keys 0-63 / 64-127 of P_x completed
                       // (the second also: O_x holds this tile's PV)
  uint64_t* o_full;    // [2] both: O_x complete for the item
  uint64_t* o_free;    // [2] leader, 8 warp arrivals: O_x read by the epilogue
  uint64_t* drain;     // [2] leader: per issuer
  uint64_t* q_land;    // own CTA (fused step): this CTA's raw Q_A, Q_B landed
  uint64_t* q_ready;   // [2] leader (fused step), 8 warp arrivals: Q_x rotated in both CTAs
};

__device__ __forceinline__ Bars bars_at(uint8_t* smem) {
  uint64_t* p = reinterpret_cast<uint64_t*>(smem + Layout::kBar);
  Bars b;
  b.q_full = p;
  b.q_empty = p + 1;
  b.kv_full = p + 2;
  b.kv_empty = b.kv_full + kStages;
  b.v_last = b.kv_empty + kStages;
  b.v_zeroed = b.v_last + kStages;
  b.s_full = b.v_zeroed + kStages;
  b.s_free = b.s_full + 2;
  b.p_full = b.s_free + 2;
  b.p_free = b.p_full + 2;
  b.o_full = b.p_free + 4;
  b.o_free = b.o_full + 2;
  b.drain = b.o_free + 2;
  b.q_land = b.drain + 2;
  b.q_ready = b.q_land + 1;
  return b;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < kWaitLimitNs) {
  }
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

// ---------------------------------------------------------------- work items
//
// One entry per (sequence, quad of query tiles): cost (key tiles, 16 bits) |
// sequence (24) | quad (16); descending order puts the heaviest first.  Work
// item i is entry i / Hkv for kv head i % Hkv.  Cluster c takes items
// c, 2C-1-c, 2C+c, ... (snake order over C clusters).

__host__ __device__ constexpr uint64_t entry_pack(uint32_t cost, uint32_t s, uint32_t quad) {
  return (static_cast<uint64_t>(cost) << 40) | (static_cast<uint64_t>(s) << 16) | quad;
}

struct Item {
  int s, quad, h;
};

__device__ __forceinline__ Item item_at(const uint64_t* entries, int i, int num_kv_heads) {
  const uint64_t v = entries[i / num_kv_heads];
  return Item{static_cast<int>((v >> 16) & 0xFFFFFF), static_cast<int>(v & 0xFFFF), i % num_kv_heads};
}

__device__ __forceinline__ int item_index(int r, int nc) {
  const int c = blockIdx.x >> 1;
  return r * nc + ((r & 1) ? nc - 1 - c : c);
}

struct QuadGeom {
  int q0;        // first token of the sequence
  int tok;       // first token (sequence-relative) of this CTA's tile A
  int n_a, n_b;  // valid tokens in this CTA's tiles A and B (either may be 0)
  int last;      // last token (sequence-relative) of the quad
  int nkeys;     // keys 0..nkeys-1 cover every row of the quad
  int ntiles;    // 128-key tiles (0 when the item's lengths are inconsistent)
};

// Both CTAs of a pair compute the same nkeys / ntiles: they walk the same
// key tiles.
template <int G>
__device__ __forceinline__ QuadGeom quad_geom(const AttnArgs& a, int s, int quad, int rank) {
  constexpr int TQ = kTile / G;
  QuadGeom p{};
  p.q0 = __ldg(a.query_start_loc + s);
  const int qlen = __ldg(a.query_start_loc + s + 1) - p.q0;
  const int quad_tok = 4 * TQ * quad;
  p.tok = quad_tok + 2 * TQ * rank;
  p.n_a = max(0, min(TQ, qlen - p.tok));
  p.n_b = max(0, min(TQ, qlen - p.tok - TQ));
  p.last = min(qlen, quad_tok + 4 * TQ) - 1;
  const int ctx = __ldg(a.context_lens + s);
  const bool shape_ok = p.q0 >= 0 && p.q0 + qlen <= a.num_tokens && quad_tok < qlen;
  const int pos_first = shape_ok ? __ldg(a.positions + p.q0 + quad_tok) : -1;
  const int pos_last = shape_ok ? __ldg(a.positions + p.q0 + p.last) : -1;
  const bool ok = shape_ok && ctx > 0 && ctx <= a.max_blocks_per_seq * a.block_size && pos_first >= 0 &&
                  pos_first <= pos_last && pos_last < ctx;
  p.nkeys = ok ? pos_last + 1 : 0;
  p.ntiles = ceil_div(p.nkeys, kTile);
  return p;
}

// Lists one entry per (prefill sequence, quad) -- sequences with query_len x
// group rows above the decode threshold -- into buf[] (unsorted), sorts them
// by cost (rank sort, entries are distinct) into out[], and returns the
// number of entries to every thread.  Run by one whole CTA of NT threads.
// Lists longer than kSortCapacity keep plan order (written to out[] as they
// are listed), which the caller allows only when out[] is in global memory.

template <int G, int NT>
__device__ int plan_entries(const AttnArgs& a, uint64_t* buf, int* warp_total, int* base, uint64_t* out,
                            int max_entries) {
  constexpr int TQ = kTile / G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) *base = 0;
  __syncthreads();
  for (int s0 = 0; s0 < a.num_seqs; s0 += NT) {
    const int s = s0 + threadIdx.x;
    int quads = 0, q0 = 0, qlen = 0;
    if (s < a.num_seqs) {
      q0 = __ldg(a.query_start_loc + s);
      qlen = __ldg(a.query_start_loc + s + 1) - q0;
      if (q0 >= 0 && qlen > 0 && q0 + qlen <= a.num_tokens && qlen * G > a.decode_max_rows) {
        quads = ceil_div(qlen, 4 * TQ);
        // read again by every CTA's roles for their items' geometry
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.context_lens + s));
      }
    }
    int incl = quads;  // inclusive scan within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) warp_total[warp] = incl;
    __syncthreads();
    int before = *base;
    for (int w = 0; w < warp; ++w) before += warp_total[w];
    int o = before + incl - quads;
    for (int q = 0; q < quads; ++q, ++o) {
      const int last = min(qlen, 4 * TQ * (q + 1)) - 1;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a.positions + q0 + 4 * TQ * q));
      const int nkeys = __ldg(a.positions + q0 + last) + 1;
      const uint32_t cost = static_cast<uint32_t>(min(max(ceil_div(nkeys, kTile), 0), 0xFFFF));
      if (o >= max_entries) continue;
      const uint64_t v = entry_pack(cost, s, q);
      if (o < kSortCapacity) buf[o] = v;
      else out[o] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0)
      for (int w = 0; w < NT / 32; ++w) *base += warp_total[w];
    __syncthreads();
  }
  const int total = min(*base, max_entries);
  for (int i = threadIdx.x; i < min(total, kSortCapacity); i += NT) {
    const uint64_t v = buf[i];
    int rank = 0;
    if (total <= kSortCapacity)
      for (int k = 0; k < total; ++k) rank += buf[k] > v;
    else
      rank = i;
    out[rank] = v;
  }
  __syncthreads();
  return total;
}

// Planning on its own (lists longer than the attention kernel plans for
// itself): one CTA, entries and *count (entries x Hkv) to global memory.
constexpr int kPlanThreads = 256;

template <int G>
__global__ void __launch_bounds__(kPlanThreads) prefill_pair_plan_kernel(const AttnArgs a, uint64_t* entries,
                                                                          int* count, int max_entries) {
  __shared__ uint64_t buf[kSortCapacity];
  __shared__ int warp_total[kPlanThreads / 32];
  __shared__ int base;
  grid_launch_dependents();
  if (!a.early_inputs) grid_dependency_wait();  // the lengths may come from the previous grid
  const int total = plan_entries<G, kPlanThreads>(a, buf, warp_total, &base, entries, max_entries);
  if (threadIdx.x == 0) *count = total * a.num_kv_heads;
  grid_dependency_wait();  // this grid completes after the one it depends on
}

// ---------------------------------------------------------------- producer

// The producer is a whole warp: one TMA copy takes its issuing thread about
// a hundred cycles, so the copies of a key tile go out from 16 lanes at once
// (lanes 0-7: this CTA's K boxes, block lane / 2 of its 64 keys, 64-column
// half lane % 2; lanes 8-15: V block lane - 8 of the tile, this CTA's 64
// columns).  Each lane loads the block id of its box one tile ahead.
__device__ __forceinline__ int lane_block_id(const int32_t* table, int j, int nkeys, int bs, int blk) {
  return (blk >= 0 && kTile * j + blk * bs < nkeys) ? __ldg(table + kTile * j / bs + blk) : -1;
}

template <int G>
__device__ __forceinline__ void producer_role(const CUtensorMap* kmap, const CUtensorMap* vmap,
                                              const CUtensorMap* qmap, const AttnArgs& a, uint8_t* smem,
                                              const Bars& b, const uint64_t* items, int count, int nc,
                                              uint32_t rank) {
  using L = Layout;
  constexpr int TQ = kTile / G;
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    prefetch_tensormap(qmap);
    prefetch_tensormap(kmap);
    prefetch_tensormap(vmap);
  }
  const bool leader = rank == 0;
  const int bs = a.block_size;
  const uint32_t box = static_cast<uint32_t>(bs * 128);  // bytes of one 64-column arena-block box
  const int oob_row = a.num_blocks * a.num_kv_heads * bs;  // past the tensor: zero fill
  const bool k_lane = lane < 8, v_lane = lane >= 8 && lane < 16;
  const int kblk = lane >> 1, kreg = lane & 1, vblk = lane - 8;
  const int k_first = 64 * static_cast<int>(rank) / bs;  // this CTA's first block of a key tile
  const int my_blk = k_lane ? k_first + kblk : (v_lane ? vblk : -1);
  int g = 0;  // key tiles issued by this CTA
  int items_done = 0;
  // outside the fused step the kernel waited for its predecessor at the start
  bool ok = true, waited = !a.early_inputs;
  const bool rotate = a.q_raw != nullptr;
  for (int r = 0; ok; ++r) {
    const int idx = item_index(r, nc);
    if (idx >= count) break;
    const Item it = item_at(items, idx, a.num_kv_heads);
    const QuadGeom p = quad_geom<G>(a, it.s, it.quad, static_cast<int>(rank));
    if (p.ntiles == 0) {
      if (leader && lane == 0) report(a.status, KSHIPRA_DEV_BAD_POSITION);
      continue;
    }
    const int32_t* table = a.block_tables + static_cast<size_t>(it.s) * a.max_blocks_per_seq;
    int next_id = lane_block_id(table, 0, p.nkeys, bs, my_blk);
    if (items_done > 0 && !warp_wait(b.q_empty, (items_done - 1) & 1, a.status)) { ok = false; break; }
    if (rotate) {  // raw Q onto this CTA's own barrier: the softmax warps rotate it in place
      if (lane == 0) mbar_arrive_expect_tx(b.q_land, 2 * L::kQTile);
    } else if (leader && lane == 0) {
      mbar_arrive_expect_tx(b.q_full, 4 * L::kQTile);  // both CTAs, zero-filled rows included
    }
    __syncwarp();
    if (lane < 4) {
      const int reg = lane & 1, tb = lane >> 1;
      uint8_t* qdst = smem + (tb ? L::kQB : L::kQA) + reg * L::kQRegion;
      if (rotate)
        tma_load_3d(qdst, qmap, 64 * reg, it.h * G, p.q0 + p.tok + TQ * tb, b.q_land);
      else
        tma_load_3d_pair(qdst, qmap, 64 * reg, it.h * G, p.q0 + p.tok + TQ * tb, map_to_rank(b.q_full, 0));
    }
    ++items_done;
    // fused step: the K/V append this grid depends on writes the sequence's
    // positions from p_new on (its query tokens); key tiles below p_new hold
    // earlier appends only and are read while the append still runs
    const int p_new = waited ? 0 : __ldg(a.positions + p.q0);
    for (int j = 0; j < p.ntiles; ++j, ++g) {
      const int st = g % kStages, use = g / kStages;
      const int id = next_id;
      if (j + 1 < p.ntiles) next_id = lane_block_id(table, j + 1, p.nkeys, bs, my_blk);
      const bool last = j + 1 == p.ntiles;
      const int nv = ceil_div(min(kTile, p.nkeys - kTile * j), bs);
      const int k_own = 64 * static_cast<int>(rank), k_peer = 64 - k_own;
      const int nk_own = p.nkeys > kTile * j + k_own ? ceil_div(min(64, p.nkeys - kTile * j - k_own), bs) : 0;
      const int nk_peer = p.nkeys > kTile * j + k_peer ? ceil_div(min(64, p.nkeys - kTile * j - k_peer), bs) : 0;
      const bool has_k = k_lane && kblk < nk_own;
      const bool has_v = v_lane && vblk < nv;
      int row = oob_row;
      if (has_k || has_v) {
        if (id < 0 || id >= a.num_blocks)
          report(a.status, KSHIPRA_DEV_BAD_BLOCK_ID);
        else
          row = (id * a.num_kv_heads + it.h) * bs;
      }
      if (g >= kStages && !warp_wait(&b.kv_empty[st], (use - 1) & 1, a.status)) { ok = false; break; }
      if (!waited && kTile * (j + 1) > p_new) {  // the tile reaches the new positions
        grid_dependency_wait();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        waited = true;
      }
      if (lane == 0) {
        // the leader expects both CTAs' K halves and, but for the last tile,
        // both V halves; an item's last V tile lands on each CTA's v_last,
        // where tile A's softmax warps zero the rows past the last key before
        // reporting P ready (which is what that tile's PV MMAs wait for)
        const uint32_t kv_bytes = static_cast<uint32_t>(nk_own + nk_peer) * 2 * box +
                                  (last ? 0u : static_cast<uint32_t>(2 * nv) * box);
        if (leader) mbar_arrive_expect_tx(&b.kv_full[st], kv_bytes);
        // a phase of v_last[st] per use of the stage, so that the softmax
        // waiting for an item's last tile can never see a later phase (the
        // stage is reused only after that wait)
        if (last)
          mbar_arrive_expect_tx(&b.v_last[st], static_cast<uint32_t>(nv) * box);
        else
          mbar_arrive(&b.v_last[st]);
      }
      __syncwarp();
      const uint32_t kv_bar = map_to_rank(&b.kv_full[st], 0);
      if (has_k)
        tma_load_2d_pair(smem + L::kK + st * L::kKStage + kreg * L::kKRegion + kblk * bs * 128, kmap, 64 * kreg,
                         row, kv_bar);
      if (has_v) {
        uint8_t* vdst = smem + L::kV + st * L::kVStage + vblk * bs * 128;
        if (!last)
          tma_load_2d_pair(vdst, vmap, 64 * static_cast<int>(rank), row, kv_bar);
        else
          tma_load_2d(vdst, vmap, 64 * static_cast<int>(rank), row, &b.v_last[st]);
      }
    }
  }
  if (!ok) {
    // copies in flight complete on the leader's barriers, which this warp
    // may not be able to observe: give them time to land (they take
    // microseconds) before the pair tears down
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) {
    }
  }
}

// ---------------------------------------------------------------- MMA issuer

// Descriptor words of the tiles the MMA issuer streams over (the low word
// carries the start address, so stepping along a tile adds a constant).
struct Descs {
  uint32_t q_lo[2], p_lo[2], k_lo, v_lo;  // K and V: stage 0; stage st adds st x the stage size
  uint32_t qk_hi, v_hi;
};

__device__ __forceinline__ uint32_t lo_word(uint64_t d) { return static_cast<uint32_t>(d); }
__device__ __forceinline__ uint32_t hi_word(uint64_t d) { return static_cast<uint32_t>(d >> 32); }

// S_x = Q_x K^T over both CTAs (rows: leader then peer; columns: the
// leader's 64 keys then the peer's), then signal s_full[x] in both CTAs.
template <bool kBf16>
__device__ __forceinline__ void issue_qk(const Descs& dd, const Bars& b, uint32_t tmem, int x, int st) {
  using L = Layout;
  constexpr uint32_t kIdescQK = idesc_f16(kBf16, 2 * kTile, kTile, false, false);
  const uint32_t q_lo = x ? dd.q_lo[1] : dd.q_lo[0];
  const uint32_t k_lo = dd.k_lo + static_cast<uint32_t>(st) * (L::kKStage >> 4);
#pragma unroll
  for (int ks = 0; ks < kD / 16; ++ks) {
    const uint32_t q_off = ((ks >> 2) * L::kQRegion + (ks & 3) * 32) >> 4;
    const uint32_t k_off = ((ks >> 2) * L::kKRegion + (ks & 3) * 32) >> 4;
    umma_pair_ss_w(tmem + kTile * x, q_lo + q_off, dd.qk_hi, k_lo + k_off, dd.qk_hi, kIdescQK, ks > 0 ? 1u : 0u);
  }
  umma_commit_pair(&b.s_full[x]);
}

// O_x (+)= P_x V.  P_x is K-major in shared memory like Q (keys 64 g .. in
// 64-key region g); V is MN-major, one 64-column swizzle atom per CTA (the
// leader's columns of O, then the peer's), 8-key row groups 1024 B apart,
// 16 keys = 2048 B per step.  Each half of P (64 keys) is released to the
// softmax as soon as its MMAs complete.
template <bool kBf16>
__device__ __forceinline__ void issue_pv(const Descs& dd, const Bars& b, uint32_t tmem, int x, int st,
                                         bool accumulate) {
  using L = Layout;
  constexpr uint32_t kIdescPV = idesc_f16(kBf16, 2 * kTile, kD, false, true);
  const uint32_t p_lo = x ? dd.p_lo[1] : dd.p_lo[0];
  const uint32_t v_lo = dd.v_lo + static_cast<uint32_t>(st) * (L::kVStage >> 4);
  const uint32_t acc = accumulate ? 1u : 0u;
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk) {
    const uint32_t p_off = ((kk >> 2) * L::kQRegion + (kk & 3) * 32) >> 4;
    umma_pair_ss_w(tmem + 2 * kTile + kTile * x, p_lo + p_off, dd.qk_hi, v_lo + ((kk * 16 * 128) >> 4), dd.v_hi,
                   kIdescPV, kk > 0 ? 1u : acc);
    if (kk == 3) umma_commit_pair(&b.p_free[2 * x]);
  }
  umma_commit_pair(&b.p_free[2 * x + 1]);
}

// The MMAs of query tile x (one issuing thread per tile, so that neither
// tile's pipeline waits on the other's softmax): per key tile j of an item,
// S_x(j + 1) = Q_x K(j + 1)^T as soon as the softmax has read S_x(j) (the
// next scores are computed while the softmax of this tile runs), then
// O_x += P_x(j) V(j) once P_x(j) is in shared memory.  Barriers that cover
// both tiles (stage empty, Q empty) count one arrival from each issuer.
template <bool kBf16, int G>
__device__ __forceinline__ void mma_role(const AttnArgs& a, uint8_t* smem, const Bars& b, uint32_t tmem,
                                         const uint64_t* items, int count, int nc, int x) {
  using L = Layout;
  const uint32_t sb = smem_u32(smem);
  Descs dd;
  dd.q_lo[0] = lo_word(smem_desc_sw128(sb + L::kQA, 16, 1024));
  dd.q_lo[1] = lo_word(smem_desc_sw128(sb + L::kQB, 16, 1024));
  dd.p_lo[0] = lo_word(smem_desc_sw128(sb + L::kPA, 16, 1024));
  dd.p_lo[1] = lo_word(smem_desc_sw128(sb + L::kPB, 16, 1024));
  dd.k_lo = lo_word(smem_desc_sw128(sb + L::kK, 16, 1024));
  dd.v_lo = lo_word(smem_desc_sw128(sb + L::kV, L::kVStage, 1024));
  dd.qk_hi = hi_word(smem_desc_sw128(sb, 16, 1024));
  dd.v_hi = hi_word(smem_desc_sw128(sb, L::kVStage, 1024));
  bool ok = true, issued_any = false;
  int g = 0, items_done = 0;

  for (int r = 0; ok; ++r) {
    const int idx = item_index(r, nc);
    if (idx >= count) break;
    const Item it = item_at(items, idx, a.num_kv_heads);
    const QuadGeom p = quad_geom<G>(a, it.s, it.quad, 0);
    const int n = p.ntiles;
    if (n == 0) continue;
    if (!mbar_wait_cluster(a.q_raw != nullptr ? &b.q_ready[x] : b.q_full, items_done & 1, a.status)) {
      ok = false;
      break;
    }
    const int g0 = g;
    // the item's first scores, once the previous tile's S columns are read
    if (!mbar_wait_cluster(&b.kv_full[g0 % kStages], (g0 / kStages) & 1, a.status) ||
        (g0 > 0 && !mbar_wait_cluster(&b.s_free[x], (g0 - 1) & 1, a.status))) {
      ok = false;
      break;
    }
    tc_fence_after();
    issue_qk<kBf16>(dd, b, tmem, x, g0 % kStages);
    issued_any = true;
    if (n == 1) umma_commit_pair(b.q_empty);
    for (int j = 0; j < n; ++j) {
      const int gt = g0 + j, st = gt % kStages, st1 = (gt + 1) % kStages;
      if (j + 1 < n) {
        if (!mbar_wait_cluster(&b.s_free[x], gt & 1, a.status) ||
            !mbar_wait_cluster(&b.kv_full[st1], ((gt + 1) / kStages) & 1, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_qk<kBf16>(dd, b, tmem, x, st1);
        if (j + 2 == n) umma_commit_pair(b.q_empty);
      }
      // the previous item's epilogue must have read O_x before PV overwrites it
      // (tile B's last PV also waits for tile A's warps to have zeroed the V
      // rows past the item's last key, which both tiles read)
      if (!mbar_wait_cluster(&b.p_full[x], gt & 1, a.status) ||
          (x == 1 && j + 1 == n && !mbar_wait_cluster(&b.v_zeroed[st], (gt / kStages) & 1, a.status)) ||
          (j == 0 && items_done > 0 && !mbar_wait_cluster(&b.o_free[x], (items_done - 1) & 1, a.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_pv<kBf16>(dd, b, tmem, x, st, j > 0);
      umma_commit_pair(&b.kv_empty[st]);  // this tile's last use of K(j), V(j)
      if (j + 1 == n) umma_commit_pair(&b.o_full[x]);
    }
    g += n;
    ++items_done;
  }
  if (!ok && issued_any) {  // wait for this thread's MMAs before tensor memory is released
    umma_commit_pair(&b.drain[x]);
    drain_wait(&b.drain[x], 0);
  }
}

// ---------------------------------------------------------------- softmax

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// One arrival per warp on a barrier of the leader CTA, after every lane's
// tensor-memory and shared-memory writes.
__device__ __forceinline__ void warp_arrive_leader(uint32_t bar_cluster) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive_cluster(bar_cluster);
}

// A whole S row (128 key columns) into registers: four loads in flight, one
// wait.
__device__ __forceinline__ void load_row(uint32_t taddr, uint32_t (&t0)[32], uint32_t (&t1)[32],
                                         uint32_t (&t2)[32], uint32_t (&t3)[32]) {
  tmem_ld32_async(taddr, t0);
  tmem_ld32_async(taddr + 32, t1);
  tmem_ld32_async(taddr + 64, t2);
  tmem_ld32_async(taddr + 96, t3);
  tmem_wait_ld(t0);
  reg_fence(t1);
  reg_fence(t2);
  reg_fence(t3);
}

// Masked scores become -inf (exp2 gives 0); the running maximum of 32 of them.
__device__ __forceinline__ void mask_max(uint32_t (&t)[32], int k0, int pos, bool diag, float (&mx)[8]) {
  if (diag) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (k0 + i > pos) t[i] = __float_as_uint(kNegInf);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) mx[i & 7] = fmax3(mx[i & 7], __uint_as_float(t[2 * i]), __uint_as_float(t[2 * i + 1]));
}

// Probabilities of 32 scores (keys 32 cc ..), their sum, and P into row r of
// the P tile in shared memory: K-major, 128-byte swizzle (16-byte chunk c of
// a 128-byte row segment stored at chunk c ^ (r % 8)), keys 64 g .. in
// region g -- the layout TMA gives Q, which the MMA reads the same way.
// Scaling, shifting and summing work on pairs (f32x2 instructions) and the
// row maximum takes three operands at a time: the softmax warps are bound by
// instruction issue, not by the special-function unit (moving some of the
// exponentials to a polynomial on the FMA pipe measured slower at every
// fraction tried).
template <bool kBf16>
__device__ __forceinline__ void exp_store(const uint32_t (&t)[32], uint64_t c2x2, uint64_t msx2,
                                          uint64_t (&sums)[2], uint32_t p_row, int cc, int r) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float x0, x1;
    f2_unpack(f2_fma(f2_bits(t[2 * i], t[2 * i + 1]), c2x2, msx2), x0, x1);
    const float p0 = ex2(x0), p1 = ex2(x1);
    sums[i & 1] = f2_add(sums[i & 1], f2_pack(p0, p1));
    pk[i] = pack2<kBf16>(p0, p1);
  }
  const uint32_t seg = p_row + (cc >> 1) * Layout::kQRegion;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t c = static_cast<uint32_t>((cc & 1) * 4 + q);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(seg + ((c ^ (r & 7)) << 4)), "r"(pk[4 * q]),
                 "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                 : "memory");
  }
}

// Rows 32 w .. 32 w + 31 of a 128-row tile held in shared memory in the Q
// layout (columns 0-63 in region 0, 64-127 in region 1, 128-byte swizzle) to
// their global rows: row t G + gg goes to dst0 + t tok_stride + gg D.  Each
// half-warp writes one whole 256-byte row per pass (lane L: 16-byte chunk
// L % 16 of row 32 w + 2 k + L / 16), so that a store instruction covers two
// rows instead of 32 scattered pieces; rows of tokens t >= nvalid are
// skipped.  Called by warp w after its lanes wrote their rows (and a warp
// synchronisation).
template <int G>
__device__ __forceinline__ void store_rows(const uint8_t* tile, int w, uint16_t* dst0, size_t tok_stride,
                                           int nvalid) {
  const int lane = threadIdx.x & 31, c = lane & 15;
  const uint8_t* src = tile + (c >> 3) * Layout::kQRegion;
  uint4 v[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int row = 32 * w + 2 * k + (lane >> 4);
    v[k] = *reinterpret_cast<const uint4*>(src + row * 128 + (((c & 7) ^ (row & 7)) << 4));
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int row = 32 * w + 2 * k + (lane >> 4);
    if (row / G < nvalid)
      *reinterpret_cast<uint4*>(dst0 + (row / G) * tok_stride + (row % G) * kD + 8 * c) = v[k];
  }
}

// Thread r of tile x owns row r (TMEM lane r): it reads its whole S row once
// (releasing the S columns to the next QK MMAs at once), masks, finds the row
// maximum, and writes P to row r of its P tile in shared memory.  The
// reference maximum of the exponents is
// raised only when the row maximum passes it by more than 2^8 (exp2 units):
// probabilities stay below 2^8, well inside fp16/bf16 range, O is rarely
// rescaled, and O / l is unchanged.
template <bool kBf16, int G>
__device__ __forceinline__ void softmax_role(const AttnArgs& a, uint8_t* smem, const Bars& b, uint32_t tmem,
                                             const uint64_t* items, int count, int nc, int x, uint32_t rank) {
  using L = Layout;
  constexpr int TQ = kTile / G;
  constexpr float kRescaleThreshold = 8.f;
  const int quarter = (threadIdx.x >> 5) & 3;
  const int r = 32 * quarter + (threadIdx.x & 31);  // row of tile x = TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
  const uint32_t s_tmem = tmem + kTile * x + lane_off;
  const uint32_t o_tmem = tmem + 2 * kTile + kTile * x + lane_off;
  const uint32_t p_row = smem_u32(smem + (x ? L::kPB : L::kPA)) + r * 128;
  const float c2 = a.scale_log2;
  const int tl = r / G;
  const size_t tok_stride = static_cast<size_t>(a.num_q_heads) * kD;
  uint8_t* const q_tile = smem + (x ? L::kQB : L::kQA);
  uint8_t* const p_tile = smem + (x ? L::kPB : L::kPA);
  int g = 0, items_done = 0;
  bool ok = true;

  // The first non-empty item from round ri on, with this row's token and
  // position (-1 when there is none).  The next item's is read while the last
  // PV MMAs of the current one run, ahead of its epilogue.
  struct RowItem {
    Item it;
    QuadGeom p;
    int nvalid, pos;
  };
  auto find = [&](int ri, RowItem& w) -> int {
    for (;; ++ri) {
      const int idx = item_index(ri, nc);
      if (idx >= count) return -1;
      w.it = item_at(items, idx, a.num_kv_heads);
      w.p = quad_geom<G>(a, w.it.s, w.it.quad, static_cast<int>(rank));
      if (w.p.ntiles == 0) continue;
      w.nvalid = x == 0 ? w.p.n_a : w.p.n_b;
      // rows past the last token compute on whatever the tile holds, at the
      // position of the quad's last token, and are never stored
      const int tok = tl < w.nvalid ? w.p.q0 + w.p.tok + TQ * x + tl : w.p.q0 + w.p.last;
      w.pos = __ldg(a.positions + tok);
      return ri;
    }
  };

  RowItem cur;
  int ri = find(0, cur);
  while (ri >= 0) {
    const Item it = cur.it;
    const QuadGeom p = cur.p;
    const int n = p.ntiles, nvalid = cur.nvalid, pos = cur.pos;
    const bool row_valid = tl < nvalid;
    // this tile's first row in the [token][head][D] outputs
    const size_t row0 = (static_cast<size_t>(p.q0 + p.tok + TQ * x) * a.num_q_heads + it.h * G) * kD;
    float m_ref = kNegInf, l = 0.f;
    if (a.q_raw != nullptr) {
      // fused step: rotate this row of the raw Q_x in place (both 64-column
      // regions: element e in region 0 pairs with e + 64 in region 1, at the
      // same swizzled chunk), store the tile to q_rot when asked, and report
      // Q_x ready to the issuer
      if (!warp_wait(b.q_land, items_done & 1, a.status)) { ok = false; break; }
      if (row_valid) {
        if (pos < 0 || pos >= a.rope_max_pos) {
          report(a.status, KSHIPRA_DEV_BAD_POSITION);
        } else {
          uint8_t* qrow = q_tile + r * 128;
          const float* cs = a.rope_table + static_cast<size_t>(pos) * kD;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4* lo = reinterpret_cast<uint4*>(qrow + ((c ^ (r & 7)) << 4));
            uint4* hi = reinterpret_cast<uint4*>(qrow + L::kQRegion + ((c ^ (r & 7)) << 4));
            uint4 ylo, yhi;
            rotate_eight_pairs_vals<kBf16>(*lo, *hi, cs + 16 * c, ylo, yhi);
            *lo = ylo;
            *hi = yhi;
          }
        }
      }
      if (a.q_rot_out != nullptr) {
        __syncwarp();
        store_rows<G>(q_tile, quarter, static_cast<uint16_t*>(a.q_rot_out) + row0, tok_stride, nvalid);
      }
      fence_proxy_async_smem();  // the rotated rows visible to the tensor cores
      warp_arrive_leader(map_to_rank(&b.q_ready[x], 0));
    }

    for (int j = 0; j < n; ++j) {
      const int gt = g + j;
      if (!warp_wait(&b.s_full[x], gt & 1, a.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t t0[32], t1[32], t2[32], t3[32];
      load_row(s_tmem, t0, t1, t2, t3);
      warp_arrive_leader(map_to_rank(&b.s_free[x], 0));  // the next scores may overwrite S_x
      // only tiles that cross some row's position (warp-uniform test) pay
      // for the mask
      const int kb0 = kTile * j;
      const bool diag = __any_sync(0xffffffffu, kb0 + kTile - 1 > pos);
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = kNegInf;
      mask_max(t0, kb0, pos, diag, mx);
      mask_max(t1, kb0 + 32, pos, diag, mx);
      mask_max(t2, kb0 + 64, pos, diag, mx);
      mask_max(t3, kb0 + 96, pos, diag, mx);
      const float m_tile =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const bool raise = m_tile != kNegInf && (m_ref == kNegInf || (m_tile - m_ref) * c2 > kRescaleThreshold);
      float alpha = 1.f;
      if (raise) {
        alpha = ex2((m_ref - m_tile) * c2);  // 0 on the first visible tile
        m_ref = m_tile;
      }
      const float ms = (m_ref == kNegInf ? 0.f : m_ref) * c2;
      // the previous tile's PV MMAs must be done with each half of P_x (and
      // with O_x, which may be rescaled below) before it is written
      if (gt > 0 && !warp_wait(&b.p_free[2 * x], (gt - 1) & 1, a.status)) { ok = false; break; }
      const uint64_t c2x2 = f2_pack(c2, c2), msx2 = f2_pack(-ms, -ms);
      uint64_t sums[2] = {0, 0};
      exp_store<kBf16>(t0, c2x2, msx2, sums, p_row, 0, r);
      exp_store<kBf16>(t1, c2x2, msx2, sums, p_row, 1, r);
      if (gt > 0 && !warp_wait(&b.p_free[2 * x + 1], (gt - 1) & 1, a.status)) { ok = false; break; }
      exp_store<kBf16>(t2, c2x2, msx2, sums, p_row, 2, r);
      exp_store<kBf16>(t3, c2x2, msx2, sums, p_row, 3, r);
      float s00, s01, s10, s11;
      f2_unpack(sums[0], s00, s01);
      f2_unpack(sums[1], s10, s11);
      l = fmaf(l, alpha, (s00 + s01) + (s10 + s11));
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t t[32];
          tmem_ld32(o_tmem + 32 * c, t);
#pragma unroll
          for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
          tmem_st32(o_tmem + 32 * c, t);
        }
      }
      if (x == 0 && j == n - 1) {
        // the item's last V tile lands on this CTA's v_last; value rows past
        // the last needed key may hold anything (even NaN, or nothing loaded
        // at all): zero them so that P = 0 contributes 0.  The PV MMAs of
        // both tiles wait for tile A's warps ("P ready" / "V zeroed").
        const int st = gt % kStages;
        if (!warp_wait(&b.v_last[st], (gt / kStages) & 1, a.status)) { ok = false; break; }
        if (r >= p.nkeys - kTile * j) {
          const uint32_t vrow = smem_u32(smem + L::kV + st * L::kVStage) + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) st_shared_zero16(vrow + c * 16);
        }
      }
      fence_proxy_async_smem();  // P (and zeroed V rows) visible to the tensor cores
      warp_arrive_leader(map_to_rank(&b.p_full[x], 0));
      if (x == 0) warp_arrive_leader(map_to_rank(&b.v_zeroed[gt % kStages], 0));
    }
    if (!ok) break;
    g += n;
    RowItem nxt;
    const int ri_next = find(ri + 1, nxt);
    // epilogue: O_x / l through P_x (free once O_x is final: every PV MMA of
    // the item is done), then whole rows to the output
    if (!warp_wait(&b.o_full[x], items_done & 1, a.status)) { ok = false; break; }
    tc_fence_after();
    const float inv = 1.f / l;
#pragma unroll
    for (int c = 0; c < kD / 32; ++c) {
      uint32_t t[32];
      tmem_ld32(o_tmem + 32 * c, t);
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack2<kBf16>(__uint_as_float(t[2 * i]) * inv, __uint_as_float(t[2 * i + 1]) * inv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ch = 4 * c + i;  // 16-byte chunk of the row
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(p_row + (ch >> 3) * L::kQRegion +
                                                                    (((ch & 7) ^ (r & 7)) << 4)),
                     "r"(w[4 * i]), "r"(w[4 * i + 1]), "r"(w[4 * i + 2]), "r"(w[4 * i + 3])
                     : "memory");
      }
    }
    warp_arrive_leader(map_to_rank(&b.o_free[x], 0));  // O_x is read (the warp is synchronised)
    store_rows<G>(p_tile, quarter, static_cast<uint16_t*>(a.out) + row0, tok_stride, nvalid);
    __syncwarp();  // every lane's reads of P_x done before the next item writes it
    ++items_done;
    cur = nxt;
    ri = ri_next;
  }
}

// ---------------------------------------------------------------- share

// Clusters of this grid that take items when the pair kernel runs beside the
// decode kernel of the same call.  The decode kernel is bound by HBM
// bandwidth and needs only part of the SMs to reach it: two CTAs per SM with
// 96 KB of loads in flight each, against the ~10 MB that HBM needs in flight
// at full bandwidth, is 56 SMs; it keeps kDecodeClusters clusters' worth and
// the prefill items take the rest -- unless they would then outlast the
// decode kernel (the items' key tiles at 4 us per tile and cluster, the rate
// measured beside the decode kernel's traffic, against the decode-class
// sequences' K/V bytes at 6.5 TB/s), in which case they take every cluster
// and the decode kernel fills the SMs they leave.  All threads of the CTA
// take part; every CTA gets the same answer.
constexpr int kDecodeClusters = 28;

template <int G>
__device__ int share_clusters(const AttnArgs& a, const uint64_t* items, int count, int nc, long long* scratch) {
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
    scratch[warp] = keys;
    scratch[kThreads / 32 + warp] = tiles;
  }
  __syncthreads();
  keys = tiles = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    keys += scratch[w];
    tiles += scratch[kThreads / 32 + w];
  }
  __syncthreads();  // scratch may be reused
  const int k = nc - kDecodeClusters;
  if (k < 1) return nc;
  const double decode_us = static_cast<double>(keys) * a.num_kv_heads * kD * 4 / 6.5e6;
  const double prefill_us = 4.0 * static_cast<double>(tiles) * a.num_kv_heads / k;
  return prefill_us <= decode_us ? k : nc;
}

// ---------------------------------------------------------------- kernel

template <bool kBf16, int G>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap qmap, const AttnArgs a, const uint64_t* planned,
                        const int* planned_count, int plan_here) {
  using L = Layout;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1024-byte alignment
    grid_dependency_wait();
    if (threadIdx.x == 0) report(a.status, KSHIPRA_DEV_TIMEOUT);
    return;
  }
  const Bars b = bars_at(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + L::kNumBars * 8);
  const uint32_t rank = cluster_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_launch_dependents();
  // barriers, tensor memory and the cluster handshake touch no global memory:
  // they run before the wait for the previous grid (launched as its
  // programmatic dependent, this CTA may start while that grid finishes)
  if (threadIdx.x == 0) {
    mbar_init(b.q_full, 1);
    mbar_init(b.q_empty, 2);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&b.kv_full[i], 1);
      mbar_init(&b.kv_empty[i], 2);
      mbar_init(&b.v_last[i], 1);
      mbar_init(&b.v_zeroed[i], 2 * 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.s_full[i], 1);
      mbar_init(&b.s_free[i], 2 * 4);  // four softmax warps per tile in each CTA
      mbar_init(&b.p_full[i], 2 * 4);
      mbar_init(&b.p_free[2 * i], 1);
      mbar_init(&b.p_free[2 * i + 1], 1);
      mbar_init(&b.o_full[i], 1);
      mbar_init(&b.o_free[i], 2 * 4);
    }
    mbar_init(&b.drain[0], 1);
    mbar_init(&b.drain[1], 1);
    mbar_init(b.q_land, 1);
    mbar_init(&b.q_ready[0], 2 * 4);
    mbar_init(&b.q_ready[1], 2 * 4);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrival or copy
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // the work list: planned here, in shared memory, when it is short enough
  // (saves a launch), else by the planning kernel.  Wait for the previous
  // grid before touching memory, unless this is the fused step (predecessor:
  // the library's K/V append) and the work list is planned here, when only
  // the arena must wait (the producer waits before its first K/V load).
  // A pair without an item runs its roles zero times.
  const uint64_t* items = planned;
  int count;
  if (!a.early_inputs || !plan_here) grid_dependency_wait();
  if (plan_here) {
    uint64_t* sorted = reinterpret_cast<uint64_t*>(smem + L::kPlanSorted);
    int* warp_total = reinterpret_cast<int*>(smem + L::kPlanWarp);
    const int total = plan_entries<G, kThreads>(a, reinterpret_cast<uint64_t*>(smem + L::kPlanBuf), warp_total,
                                                warp_total + 12, sorted, kSortCapacity);
    count = total * a.num_kv_heads;
    items = sorted;
  } else {
    count = *planned_count;
  }

  // clusters that take items: all of them, or beside the decode kernel only
  // those its share of the call needs (the others run their roles zero times)
  int nc = static_cast<int>(gridDim.x >> 1);
  if (a.beside_decode) nc = share_clusters<G>(a, items, count, nc, reinterpret_cast<long long*>(smem + L::kShare));
  if (static_cast<int>(blockIdx.x >> 1) >= nc) count = 0;
  if (warp < 8) {
    softmax_role<kBf16, G>(a, smem, b, tmem, items, count, nc, warp >> 2, rank);
  } else if (warp == kProducerWarp) {
    producer_role<G>(&kmap, &vmap, &qmap, a, smem, b, items, count, nc, rank);
  } else if (rank == 0) {
    if (lane == 0) mma_role<kBf16, G>(a, smem, b, tmem, items, count, nc, warp - kMmaWarp);
  }
  grid_dependency_wait();  // (at once when the producer has waited already)
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal its barriers
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Clusters of the persistent grid: as many pairs as fit at once (at most
// one per two SMs), probed once per device.
template <typename Kernel>
int pair_clusters(Kernel* kernel, int sm_count) {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const int c = cached[dev & 63].load(std::memory_order_relaxed);
  if (c > 0) return c;
  int n = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count / 2 > 0 ? sm_count / 2 : 1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Layout::kAlloc;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sm_count / 2;
  }
  n = max(1, min(n, max(1, sm_count / 2)));
  cached[dev & 63].store(n, std::memory_order_relaxed);
  return n;
}

template <bool kBf16, int G>
cudaError_t launch_pair_t(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const CUtensorMap& qmap, cudaStream_t stream) {
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = set_smem_limit_once(prefill_pair_kernel<kBf16, G>, Layout::kAlloc, configured);
  if (e != cudaSuccess) return e;
  const int clusters = pair_clusters(prefill_pair_kernel<kBf16, G>, a.sm_count);
  const bool plan_here = a.max_items <= kSortCapacity;  // an upper bound on the entries
  // both launch as programmatic dependents; the attention kernel waits for
  // the planning kernel before reading the planned list
  if (!plan_here) {
    e = launch_kernel(prefill_pair_plan_kernel<G>, dim3(1), dim3(kPlanThreads), 0, stream, true, a, a.ws_items,
                      a.ws_item_count, a.max_items);
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(prefill_pair_kernel<kBf16, G>, dim3(2 * clusters), dim3(kThreads), Layout::kAlloc, stream,
                       true, kmap, vmap, qmap, a, static_cast<const uint64_t*>(a.ws_items),
                       static_cast<const int*>(a.ws_item_count), plan_here ? 1 : 0);
}

template <bool kBf16>
cudaError_t launch_pair_g(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const CUtensorMap& qmap, cudaStream_t stream) {
  switch (a.group) {
    case 1: return launch_pair_t<kBf16, 1>(a, kmap, vmap, qmap, stream);
    case 2: return launch_pair_t<kBf16, 2>(a, kmap, vmap, qmap, stream);
    case 4: return launch_pair_t<kBf16, 4>(a, kmap, vmap, qmap, stream);
    case 8: return launch_pair_t<kBf16, 8>(a, kmap, vmap, qmap, stream);
    case 16: return launch_pair_t<kBf16, 16>(a, kmap, vmap, qmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill_pair(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                const CUtensorMap& qmap, cudaStream_t stream) {
  if (a.head_dim != kD) return cudaErrorInvalidValue;
  return a.dtype == KSHIPRA_DTYPE_BF16 ? launch_pair_g<true>(a, kmap, vmap, qmap, stream)
                                       : launch_pair_g<false>(a, kmap, vmap, qmap, stream);
}

}  // namespace kshipra
