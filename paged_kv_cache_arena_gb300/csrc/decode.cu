// Split-KV decode attention over the block arena, with the split combine.
//
// Pages "Building Kshipra" part 3 (kshipra-3), section 4: attention runs an
// online softmax (running max m, running sum l, rescaled accumulator o) over
// KV blocks read in place from the arena, and the merge is exact, so the key
// range of one sequence can be cut into splits whose partial (m, l, o) are
// merged afterwards with the same rescaling rule.  Section 1: keys of
// position p sit in slot p % block_size of physical block
// block_tables[s][p / block_size].
//
// Work unit (one CTA): (sequence s, kv head h, split).  All query rows that
// share kv head h -- query_len x group rows, at most 16 -- are served from one
// read of each K/V tile.  The CTAs take the units longest first: every full
// split of every decode-class sequence (kv heads of one split next to each
// other, so the heads of one arena block are read together), then the
// sequences' shorter last splits in decreasing length, so that the last wave
// holds the shortest work (batches of up to 256 sequences; larger ones, many
// waves long, take the units in index order).
//  - Each of the 4 warps owns every 4th 16-key chunk of the split and keeps a
//    3-deep ring of shared-memory stages.  Lane 0 fills a stage with four TMA
//    tile loads (K and V, two 64-column halves each, 128-byte swizzle)
//    straight from the arena block, completing on the stage's mbarrier.
//  - Scores are computed as S^T = K q^T with mma.sync m16n8k16 (keys on the
//    16-row side, query rows on the 8-column side), so no query padding to 16
//    rows is needed; fp32 accumulation.
//  - Online softmax in registers with quad-lane shuffles for the row max; the
//    running sum stays per lane until the end.
//  - P^T is turned into the B operand of O^T = V^T P^T with movmatrix, V^T
//    comes from ldmatrix.trans; keys past the context (possibly NaN) get
//    zeroed value rows.
//  - Warps merge through shared memory; a single-split sequence writes its
//    rounded output directly, otherwise the partial (m, l, o) goes to the
//    workspace, and the CTA that finishes last for its (sequence, kv head)
//    (atomic ticket) merges all splits.
//  - Fused decode step (kshipra_decode_step): the kernel also does the
//    RoPE-and-append of the step's new tokens (or, in a mixed step whose
//    append ran as its own kernel, only the query rotation).  Each CTA rotates its own query
//    rows from the raw q in registers; in the CTA whose split holds a new
//    token's position, the warp that loads the chunk holding it writes that
//    token's rotated K and raw V (its kv head) into the arena before it loads
//    anything -- no other warp or CTA reads that position -- so the step is
//    one launch.  The rotation is the append kernel's, bit for bit.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "internal.h"
#include "rope.cuh"

namespace kshipra {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kChunk = 16;  // keys per stage
constexpr float kNegInf = -INFINITY;

// Generic-proxy global writes of this thread ordered before later async-proxy
// (TMA) reads that a barrier orders after them.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

template <int D>
struct DecodeLayout {
  static constexpr int kRegions = D / 64;                      // 64-column swizzle regions
  static constexpr int kRegionBytes = kChunk * 128;            // 16 rows x 128 B
  static constexpr int kTileBytes = kRegions * kRegionBytes;   // K (or V) of one chunk
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kWarpBytes = kStages * kStageBytes;
  static constexpr int kBarOffset = kWarps * kWarpBytes;
  static constexpr int kBytes = kBarOffset + kWarps * kStages * 8;
  static constexpr int kMergeBytes = kWarps * (2 * 16 + 16 * D) * 4;
  static_assert(kMergeBytes <= kBarOffset, "merge scratch must fit in the stage buffers");
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 B
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

template <int D, bool kBf16, bool kFused, int NT>
__device__ __forceinline__ void decode_body(const CUtensorMap* kmap, const CUtensorMap* vmap, const AttnArgs& a,
                                            uint8_t* smem, int s, int h, int split, int q0, int qlen, int ctx,
                                            int nsplit) {
  const int nrows = qlen * a.group;
  using L = DecodeLayout<D>;
  constexpr int KS = D / 16;  // 16-wide steps over the head dimension
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int G = a.group;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset) + warp * kStages;
  uint8_t* wbase = smem + warp * L::kWarpBytes;

  const int tok_begin = split * a.split_tokens;
  const int tok_end = min(ctx, tok_begin + a.split_tokens);
  const int nchunks = ceil_div(tok_end - tok_begin, kChunk);
  const int my_chunks = nchunks > warp ? ceil_div(nchunks - warp, kWarps) : 0;
  const int oob_row = a.num_blocks * a.num_kv_heads * a.block_size;  // past the tensor: zero fill

  if constexpr (kFused) {
    // the step's new tokens whose positions fall in this split: rotated K and
    // raw V of kv head h into their arena slots, each written by the warp
    // that loads the 16-key chunk holding it, before that warp loads any
    // tile; the other warps start at once
    constexpr int half = D / 2;
    bool wrote = false;
    for (int i = 0; a.k_new != nullptr && i < qlen; ++i) {
      const int t = q0 + i;
      const int pos = __ldg(a.positions + t);
      if (pos < tok_begin || pos >= tok_end || ((pos - tok_begin) / kChunk) % kWarps != warp) continue;
      if (pos >= a.rope_max_pos) {
        if (lane == 0) report(a.status, KSHIPRA_DEV_BAD_POSITION);
        continue;
      }
      const int blk = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + pos / a.block_size);
      if (blk < 0 || blk >= a.num_blocks) {
        if (lane == 0) report(a.status, KSHIPRA_DEV_BAD_BLOCK_ID);
        continue;
      }
      const size_t src = (static_cast<size_t>(t) * a.num_kv_heads + h) * D;
      const size_t dst = ((static_cast<size_t>(blk) * a.num_kv_heads + h) * a.block_size + pos % a.block_size) * D;
      if (2 * lane < half)
        rotate_two_pairs<kBf16>(static_cast<const uint16_t*>(a.k_new) + src, static_cast<uint16_t*>(a.k_arena_w) + dst,
                                2 * lane, half, a.rope_table + static_cast<size_t>(pos) * D);
      if (lane < D / 8)  // value row: bit copy in 16-byte pieces
        reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.v_arena_w) + dst)[lane] =
            reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.v_new) + src)[lane];
      wrote = true;
    }
    if (wrote) fence_proxy_async_global();  // the rows above, before this warp's tile loads below
    __syncwarp();
  }

  if (lane == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](int i) {  // lane 0 only: load this warp's i-th chunk
    const int c = warp + kWarps * i;
    const int tok = tok_begin + c * kChunk;
    const int blk = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + tok / a.block_size);
    int row;
    if (blk < 0 || blk >= a.num_blocks) {
      report(a.status, KSHIPRA_DEV_BAD_BLOCK_ID);
      row = oob_row;
    } else {
      row = (blk * a.num_kv_heads + h) * a.block_size + (tok % a.block_size);
    }
    uint8_t* stg = wbase + (i % kStages) * L::kStageBytes;
    uint64_t* bar = &bars[i % kStages];
    mbar_arrive_expect_tx(bar, L::kStageBytes);
#pragma unroll
    for (int r = 0; r < L::kRegions; ++r) {
      tma_load_2d(stg + r * L::kRegionBytes, kmap, 64 * r, row, bar);
      tma_load_2d(stg + L::kTileBytes + r * L::kRegionBytes, vmap, 64 * r, row, bar);
    }
  };
  int issued = 0;
  if (lane == 0) {
    for (; issued < min(kStages, my_chunks); ++issued) issue(issued);
  }
  if constexpr (kFused) {
    // split 0 also stores the rotated query rows when asked to, while the
    // first tiles are in flight
    constexpr int half = D / 2;
    if (split == 0 && a.q_rot_out != nullptr)
      for (int n = warp; n < nrows; n += kWarps) {
        const int t = q0 + n / a.group;
        const int pos = __ldg(a.positions + t);
        if (pos < 0 || pos >= a.rope_max_pos) continue;
        const size_t row = (static_cast<size_t>(t) * a.num_q_heads + h * a.group + n % a.group) * D;
        if (2 * lane < half)
          rotate_two_pairs<kBf16>(static_cast<const uint16_t*>(a.q_raw) + row,
                                  static_cast<uint16_t*>(a.q_rot_out) + row, 2 * lane, half,
                                  a.rope_table + static_cast<size_t>(pos) * D);
      }
  }

  // Query fragments: B operand of S^T = K q^T.  Column n of n-tile nt is
  // query row 8 nt + g = (token q0 + n / G, q head h G + n % G).
  uint32_t qb[NT][KS][2];
  int rpos[NT][2];
  const uint16_t* qrot = static_cast<const uint16_t*>(kFused ? a.q_raw : a.q_rot);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n = 8 * nt + g;
    const uint16_t* qp = nullptr;
    if (n < nrows)
      qp = qrot + (static_cast<size_t>(q0 + n / G) * a.num_q_heads + h * G + n % G) * D;
    if constexpr (kFused) {
      // rotate the row's elements e, e + 1 with their partners e +- d/2
      const int pos = qp ? __ldg(a.positions + q0 + n / G) : -1;
      const bool pos_ok = pos >= 0 && pos < a.rope_max_pos;
      const float* cs = a.rope_table + static_cast<size_t>(pos_ok ? pos : 0) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int e = 16 * ks + 8 * hb + 2 * t4;
          const bool upper = e >= D / 2;
          const int f = upper ? e - D / 2 : e;
          uint32_t v = 0u;
          if (qp && pos_ok)
            v = rope_pair<kBf16>(__ldg(reinterpret_cast<const uint32_t*>(qp + e)),
                                 __ldg(reinterpret_cast<const uint32_t*>(qp + (upper ? f : e + D / 2))),
                                 __ldg(reinterpret_cast<const float4*>(cs + 2 * f)), upper);
          qb[nt][ks][hb] = v;
        }
    } else {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qb[nt][ks][0] = qp ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * ks + 2 * t4)) : 0u;
        qb[nt][ks][1] = qp ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * ks + 8 + 2 * t4)) : 0u;
      }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 8 * nt + 2 * t4 + e;
      rpos[nt][e] = r < nrows ? __ldg(a.positions + q0 + r / G) : -1;
    }
  }

  float m[NT][2], l[NT][2], o[NT][KS][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      m[nt][e] = kNegInf;
      l[nt][e] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[nt][mt][k] = 0.f;
  }
  const float c2 = a.scale_log2;
  bool ok = true;
  int consumed = 0;

  for (int i = 0; i < my_chunks; ++i) {
    const int st = i % kStages;
    if (!mbar_wait(&bars[st], (i / kStages) & 1, a.status)) {
      ok = false;
      break;
    }
    consumed = i + 1;
    const uint32_t kb = smem_u32(wbase + st * L::kStageBytes);
    const uint32_t vb = kb + L::kTileBytes;
    const int tok0 = tok_begin + (warp + kWarps * i) * kChunk;

    // S^T (16 keys x 8 query rows per n-tile)
    float sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) sacc[nt][k] = 0.f;
    {
      const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
      const uint32_t rbase = kb + row * 128;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int ch = 2 * (ks & 3) + (lane >> 4);
        uint32_t af[4];
        ldsm_x4(rbase + (ks >> 2) * L::kRegionBytes + ((ch ^ (row & 7)) << 4), af);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816<kBf16>(sacc[nt], af, qb[nt][ks][0], qb[nt][ks][1]);
      }
    }

    // causal mask (key j visible iff j <= the row's position) and online softmax
    const int j0 = tok0 + g, j1 = j0 + 8;
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float s0 = j0 <= rpos[nt][e] ? sacc[nt][e] : kNegInf;
        const float s1 = j1 <= rpos[nt][e] ? sacc[nt][e + 2] : kNegInf;
        float mx = fmaxf(s0, s1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(m[nt][e], mx);
        const float ms = (mnew == kNegInf ? 0.f : mnew) * c2;
        const float alpha = ex2(fmaf(m[nt][e], c2, -ms));
        p[e] = ex2(fmaf(s0, c2, -ms));
        p[e + 2] = ex2(fmaf(s1, c2, -ms));
        l[nt][e] = fmaf(l[nt][e], alpha, p[e] + p[e + 2]);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[nt][mt][e] *= alpha;
          o[nt][mt][e + 2] *= alpha;
        }
        m[nt][e] = mnew;
      }
      pb[nt][0] = movmatrix_trans(pack2<kBf16>(p[0], p[1]));
      pb[nt][1] = movmatrix_trans(pack2<kBf16>(p[2], p[3]));
    }

    // O^T (head dim x query rows) += V^T P^T
    const bool tail = tok0 + kChunk > ctx;
    uint32_t vmask_a = 0xFFFFFFFFu, vmask_b = 0xFFFFFFFFu;
    if (tail) {  // value rows of keys past the context may hold anything
      const int ta = tok0 + 2 * t4, tb = ta + 8;
      vmask_a = (ta < ctx ? 0x0000FFFFu : 0u) | (ta + 1 < ctx ? 0xFFFF0000u : 0u);
      vmask_b = (tb < ctx ? 0x0000FFFFu : 0u) | (tb + 1 < ctx ? 0xFFFF0000u : 0u);
    }
    {
      const int row = (lane & 7) + 8 * (lane >> 4);
      const uint32_t rbase = vb + row * 128;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int ch = 2 * mt + ((lane >> 3) & 1);
        uint32_t vf[4];
        ldsm_x4_trans(rbase + (ch >> 3) * L::kRegionBytes + (((ch & 7) ^ (row & 7)) << 4), vf);
        vf[0] &= vmask_a;
        vf[1] &= vmask_a;
        vf[2] &= vmask_b;
        vf[3] &= vmask_b;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816<kBf16>(o[nt][mt], vf, pb[nt][0], pb[nt][1]);
      }
    }
    __syncwarp();
    if (lane == 0 && issued < my_chunks) issue(issued++);
  }

  if (!ok) {
    // a wait gave up: let this warp's outstanding loads land before the CTA
    // reuses or releases its shared memory
    if (lane == 0)
      for (int i = consumed; i < issued; ++i) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&bars[i % kStages], (i / kStages) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    __syncwarp();
  }

#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = l[nt][e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l[nt][e] = v;
    }

  __syncthreads();  // every warp's stages are drained: reuse them for the merge
  const bool any_fail = __syncthreads_or(!ok);
  float* mbuf = reinterpret_cast<float*>(smem);
  float* lbuf = mbuf + kWarps * 16;
  float* obuf = lbuf + kWarps * 16;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 8 * nt + 2 * t4 + e;
      if (g == 0) {
        mbuf[warp * 16 + r] = m[nt][e];
        lbuf[warp * 16 + r] = l[nt][e];
      }
      float* orow = obuf + (warp * 16 + r) * D;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        orow[16 * mt + g] = o[nt][mt][e];
        orow[16 * mt + g + 8] = o[nt][mt][e + 2];
      }
    }
  __syncthreads();
  if (any_fail) return;

  const size_t split_stride = static_cast<size_t>(a.num_tokens) * a.num_q_heads;
  for (int idx = threadIdx.x; idx < nrows * D; idx += kThreads) {
    const int r = idx / D, d = idx % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mbuf[w * 16 + r]);
    float Lsum = 0.f, O = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = mbuf[w * 16 + r];
        const float f = mw == kNegInf ? 0.f : ex2((mw - M) * c2);
        Lsum = fmaf(lbuf[w * 16 + r], f, Lsum);
        O = fmaf(obuf[(w * 16 + r) * D + d], f, O);
      }
    }
    const int tok = q0 + r / G, head = h * G + r % G;
    const size_t orow = static_cast<size_t>(tok) * a.num_q_heads + head;
    if (nsplit == 1) {
      static_cast<uint16_t*>(a.out)[orow * D + d] = round_f32<kBf16>(O / Lsum);
    } else {
      const size_t prow = static_cast<size_t>(split) * split_stride + orow;
      a.ws_o[prow * D + d] = O;
      if (d == 0) {
        a.ws_ml[prow * 2] = M;
        a.ws_ml[prow * 2 + 1] = Lsum;
      }
    }
  }
  if (nsplit == 1) return;

  // Split combine, done by whichever CTA of this (sequence, kv head) finishes
  // last: M = max_i m_i, L = sum_i l_i 2^{(m_i - M) c}, out = sum_i o_i 2^{(m_i - M) c} / L.
  __shared__ unsigned is_last;
  __threadfence();  // this CTA's partials are visible before its ticket
  __syncthreads();
  if (threadIdx.x == 0)
    is_last = atomicAdd(a.ws_counters + static_cast<size_t>(s) * a.num_kv_heads + h, 1u) ==
              static_cast<unsigned>(nsplit - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int idx = threadIdx.x; idx < nrows * D; idx += kThreads) {
    const int r = idx / D, d = idx % D;
    const size_t orow = static_cast<size_t>(q0 + r / G) * a.num_q_heads + h * G + r % G;
    float M = kNegInf;
    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(a.ws_ml + (sp * split_stride + orow) * 2));
    float Lsum = 0.f, O = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) {
      const size_t prow = sp * split_stride + orow;
      const float mi = __ldcg(a.ws_ml + prow * 2);
      const float f = mi == kNegInf ? 0.f : ex2((mi - M) * c2);
      Lsum = fmaf(__ldcg(a.ws_ml + prow * 2 + 1), f, Lsum);
      O = fmaf(__ldcg(a.ws_o + prow * D + d), f, O);
    }
    static_cast<uint16_t*>(a.out)[orow * D + d] = round_f32<kBf16>(O / Lsum);
  }
}

// Exclusive prefix sum of v over the CTA's threads in thread order, and the
// CTA total.  Every thread calls it.
__device__ __forceinline__ int cta_exclusive_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int t = warp_tot[w];
    if (w < warp) before += t;
    total += t;
  }
  __syncthreads();  // warp_tot may be reused
  return before + incl - v;
}

constexpr int kRemBuckets = 256;  // last-split lengths, in 1/256ths of a split

// Context length of sequence s when it is of the decode class and its
// lengths are consistent, else 0 (inconsistent ones reported by CTA 0).
__device__ __forceinline__ int decode_ctx(const AttnArgs& a, int s) {
  // the three loads go out together (s < num_seqs: every address is in bounds)
  const int q0 = __ldg(a.query_start_loc + s);
  const int qlen = __ldg(a.query_start_loc + s + 1) - q0;
  const int ctx = __ldg(a.context_lens + s);
  if (q0 < 0 || q0 + qlen > a.num_tokens) {  // query_start_loc inconsistent with num_tokens
    if (blockIdx.x == 0) report(a.status, KSHIPRA_DEV_BAD_LENGTHS);
    return 0;
  }
  if (qlen <= 0 || qlen * a.group > a.decode_max_rows) return 0;  // empty, or handled by the prefill kernel
  if (ctx <= 0 || ctx > a.max_blocks_per_seq * a.block_size || ceil_div(ctx, a.split_tokens) > a.max_splits) {
    if (blockIdx.x == 0) report(a.status, KSHIPRA_DEV_BAD_LENGTHS);
    return 0;
  }
  return ctx;
}

// The unit of CTA blockIdx.x.  Batches of up to kDecodeOrderedMaxSeqs
// sequences take the order described at the top -- full splits (sequence,
// split, kv head), then last splits by decreasing length bucket (sequence
// order within a bucket), kv head fastest -- found by scanning the batch's
// lengths, kThreads sequences per round.  Larger batches (many waves, a
// small tail) take the grid in index order -- sequence, kv head, split --
// with no scan.  False when the index names no unit.
__device__ bool decode_unit(const AttnArgs& a, int& s_out, int& h_out, int& split_out) {
  const int L = a.split_tokens, H = a.num_kv_heads;
  const int i = static_cast<int>(blockIdx.x);
  if (!a.decode_ordered) {
    const int s = i / (H * a.max_splits), h = (i / a.max_splits) % H, split = i % a.max_splits;
    if (s >= a.num_seqs) return false;
    const int ctx = decode_ctx(a, s);
    if (ctx == 0 || split >= ceil_div(ctx, L)) return false;
    s_out = s;
    h_out = h;
    split_out = split;
    return true;
  }
  __shared__ int warp_tot[kWarps];
  __shared__ int hist[kRemBuckets];
  __shared__ int found[3];
  for (int b = threadIdx.x; b < kRemBuckets; b += kThreads) hist[b] = 0;
  if (threadIdx.x == 0) found[0] = -1;
  __syncthreads();
  int full_before = 0;  // full-split units of the sequences scanned so far
  for (int b0 = 0; b0 < a.num_seqs; b0 += kThreads) {
    const int s = b0 + static_cast<int>(threadIdx.x);
    const int ctx = s < a.num_seqs ? decode_ctx(a, s) : 0;
    const int nfull = ctx / L, rem = ctx - nfull * L;
    int t;
    const int start = full_before + H * cta_exclusive_scan(nfull, warp_tot, t);
    if (i >= start && i < start + H * nfull) {
      found[0] = s;
      found[1] = (i - start) / H;
      found[2] = (i - start) % H;
    }
    if (rem > 0) atomicAdd(&hist[static_cast<int>((static_cast<long long>(rem) * kRemBuckets) / L)], 1);
    full_before += H * t;
  }
  __syncthreads();
  if (found[0] >= 0) {
    s_out = found[0];
    split_out = found[1];
    h_out = found[2];
    return true;
  }
  // a last split: the r-th sequence with one in (bucket descending, sequence) order
  const int r = (i - full_before) / H, h = (i - full_before) % H;
  // buckets in descending order: thread k holds buckets 2k (after) and 2k + 1
  static_assert(kRemBuckets == 2 * kThreads, "two buckets per thread");
  const int b_hi = kRemBuckets - 1 - 2 * static_cast<int>(threadIdx.x), b_lo = b_hi - 1;
  int nrem;
  const int before = cta_exclusive_scan(hist[b_hi] + hist[b_lo], warp_tot, nrem);
  if (r >= nrem) return false;  // past the last unit
  __shared__ int pick[2];
  if (r >= before && r < before + hist[b_hi]) {
    pick[0] = b_hi;
    pick[1] = r - before;
  } else if (r >= before + hist[b_hi] && r < before + hist[b_hi] + hist[b_lo]) {
    pick[0] = b_lo;
    pick[1] = r - before - hist[b_hi];
  }
  __syncthreads();
  const int bucket = pick[0], k = pick[1];
  int seen = 0;
  for (int b0 = 0; b0 < a.num_seqs; b0 += kThreads) {
    const int s = b0 + static_cast<int>(threadIdx.x);
    const int ctx = s < a.num_seqs ? decode_ctx(a, s) : 0;
    const int rem = ctx % L;
    const bool in = rem > 0 && static_cast<int>((static_cast<long long>(rem) * kRemBuckets) / L) == bucket;
    int t;
    const int idx = seen + cta_exclusive_scan(in ? 1 : 0, warp_tot, t);
    if (in && idx == k) {
      found[0] = s;
      found[1] = ctx / L;
    }
    seen += t;
    if (seen > k) break;
  }
  __syncthreads();
  s_out = found[0];
  split_out = found[1];
  h_out = h;
  return s_out >= 0;
}

template <int D, bool kBf16, bool kFused>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const AttnArgs a) {
  // launched as a programmatic dependent of the previous grid on the stream:
  // the next grid may start its own launch now, and every CTA waits for the
  // previous one (so this grid completes after it) before touching memory
  grid_launch_dependents();
  grid_dependency_wait();
  int s, h, split;
  if (!decode_unit(a, s, h, split)) return;
  const int q0 = __ldg(a.query_start_loc + s);
  const int qlen = __ldg(a.query_start_loc + s + 1) - q0;
  const int ctx = __ldg(a.context_lens + s);
  const int nsplit = ceil_div(ctx, a.split_tokens);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (qlen * a.group <= 8)
    decode_body<D, kBf16, kFused, 1>(&kmap, &vmap, a, smem, s, h, split, q0, qlen, ctx, nsplit);
  else
    decode_body<D, kBf16, kFused, 2>(&kmap, &vmap, a, smem, s, h, split, q0, qlen, ctx, nsplit);
}

template <int D, bool kBf16, bool kFused>
cudaError_t launch_decode_f(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t stream) {
  using L = DecodeLayout<D>;
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = set_smem_limit_once(decode_kernel<D, kBf16, kFused>, L::kAlloc, configured);
  if (e != cudaSuccess) return e;
  // at most max_splits units per (sequence, kv head); CTAs past the last unit exit at once
  const long long units = static_cast<long long>(a.max_splits) * a.num_kv_heads * a.num_seqs;
  if (units > INT_MAX) return cudaErrorInvalidConfiguration;
  return launch_kernel(decode_kernel<D, kBf16, kFused>, dim3(static_cast<unsigned>(units)), dim3(kThreads), L::kAlloc,
                       stream, !a.beside_decode, kmap, vmap, a);
}

template <int D, bool kBf16>
cudaError_t launch_decode_t(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t stream) {
  return a.q_raw ? launch_decode_f<D, kBf16, true>(a, kmap, vmap, stream)
                 : launch_decode_f<D, kBf16, false>(a, kmap, vmap, stream);
}

}  // namespace

cudaError_t launch_decode(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t stream) {
  if (a.num_seqs == 0 || a.decode_max_rows == 0) return cudaSuccess;
  const bool bf = a.dtype == KSHIPRA_DTYPE_BF16;
  if (a.head_dim == 128)
    return bf ? launch_decode_t<128, true>(a, kmap, vmap, stream) : launch_decode_t<128, false>(a, kmap, vmap, stream);
  return bf ? launch_decode_t<64, true>(a, kmap, vmap, stream) : launch_decode_t<64, false>(a, kmap, vmap, stream);
}

}  // namespace kshipra
