// Chunked-prefill attention over the block arena on tcgen05 tensor cores.
//
// Pages "Building Kshipra" part 3 (kshipra-3), section 4: a prompt chunk of
// new tokens sits at absolute positions after the cached prefix; each query
// attends to the cached prefix and to the earlier tokens of its own chunk
// (causal mask); attention runs an online softmax over KV blocks read in
// place from the arena.  Section 1: keys of position p live in slot
// p % block_size of physical block block_tables[s][p / block_size].
//
// Work unit (one CTA): 128 query rows = 128/G consecutive tokens x the G
// query heads of one kv head (GQA packing: every K/V tile is loaded once for
// all G heads), against 128-key tiles of that sequence.  Key tiles that lie
// entirely past the tile's last position are never visited; only tiles that
// cross a row's position are masked element by element.
//
// Roles (192 threads):
//  - warp 4 (one lane): TMA producer.  The Q tile is one 3-D box per 64-column
//    half; each K/V tile is 128 / block_size boxes of one arena block each,
//    addressed through the block table, double-buffered.
//  - warp 5 (one lane): tcgen05.mma issuer.  S = Q K^T (M 128, N 128, K d)
//    into TMEM columns [0, 128); O += P V (M 128, N d, K 128) into TMEM
//    columns [128, 128 + d), V read MN-major straight from its arena layout.
//    Completion is signalled with tcgen05.commit on mbarriers.
//  - warps 0-3: softmax.  Thread r owns row r (TMEM lane r): loads its S row,
//    applies the causal mask, updates the running max / sum, writes the
//    probabilities as fp16/bf16 into shared memory (K-major, 128-byte
//    swizzle) for the PV MMA, rescales its O row in TMEM when the max grows,
//    and finally normalises and stores the output row.
// Every wait is bounded (see mbar_wait); on a timeout all roles stop, drain
// their outstanding copies / MMAs and release tensor memory.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace kshipra {
namespace {

constexpr int kTile = 128;  // query rows per CTA and keys per tile
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 256;
constexpr float kNegInf = -INFINITY;

template <int D>
struct PrefillLayout {
  static constexpr int kRegions = D / 64;
  static constexpr int kRegionBytes = kTile * 128;  // 128 rows x 128 B
  static constexpr int kTileBytes = kRegions * kRegionBytes;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kP = kV + kStages * kTileBytes;
  static constexpr int kBar = kP + 2 * kRegionBytes;  // P: 128 rows x 128 keys
  // barriers: q, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full, s_free,
  // p_full, o_done, drain; then the TMEM base address
  static constexpr int kNumBars = 14;
  static constexpr int kBytes = kBar + kNumBars * 8 + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

struct Bars {
  uint64_t* q;
  uint64_t* k_full;
  uint64_t* k_empty;
  uint64_t* v_full;
  uint64_t* v_empty;
  uint64_t* s_full;
  uint64_t* s_free;
  uint64_t* p_full;
  uint64_t* o_done;
  uint64_t* drain;
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Waits for a phase ignoring other CTAs' timeouts (used to drain own work).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < kWaitLimitNs) {
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// ---------------------------------------------------------------- producer

template <int D, int G>
__device__ __forceinline__ void producer_role(const CUtensorMap* kmap, const CUtensorMap* vmap,
                                              const CUtensorMap* qmap, const AttnArgs& a, uint8_t* smem,
                                              const Bars& b, int s, int h, int tok0, int nkeys, int ntiles) {
  using L = PrefillLayout<D>;
  prefetch_tensormap(qmap);
  prefetch_tensormap(kmap);
  prefetch_tensormap(vmap);
  mbar_arrive_expect_tx(b.q, L::kTileBytes);  // out-of-range tokens are zero-filled, bytes still count
#pragma unroll
  for (int r = 0; r < L::kRegions; ++r) tma_load_3d(smem + L::kQ + r * L::kRegionBytes, qmap, 64 * r, h * G, tok0, b.q);

  const int bs = a.block_size;
  const int blocks_per_tile = kTile / bs;
  const int oob_row = a.num_blocks * a.num_kv_heads * bs;
  const int32_t* table = a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq;
  int issued_k[kStages] = {0, 0}, issued_v[kStages] = {0, 0};
  bool ok = true;
  for (int j = 0; j < ntiles && ok; ++j) {
    const int st = j & 1, use = j >> 1;
    const int kend = min(kTile * (j + 1), nkeys);
    const int nb = ceil_div(kend - kTile * j, bs);
    const uint32_t bytes = static_cast<uint32_t>(nb * bs * 128 * L::kRegions);
    int rows[kTile / 16];
    for (int i = 0; i < nb; ++i) {
      const int blk = __ldg(table + j * blocks_per_tile + i);
      if (blk < 0 || blk >= a.num_blocks) {
        report(a.status, KSHIPRA_DEV_BAD_BLOCK_ID);
        rows[i] = oob_row;
      } else {
        rows[i] = (blk * a.num_kv_heads + h) * bs;
      }
    }
    if (j >= kStages && !mbar_wait(&b.k_empty[st], (use - 1) & 1, a.status)) { ok = false; break; }
    mbar_arrive_expect_tx(&b.k_full[st], bytes);
    uint8_t* kdst = smem + L::kK + st * L::kTileBytes;
    for (int i = 0; i < nb; ++i)
#pragma unroll
      for (int r = 0; r < L::kRegions; ++r)
        tma_load_2d(kdst + r * L::kRegionBytes + i * bs * 128, kmap, 64 * r, rows[i], &b.k_full[st]);
    issued_k[st] = j + 1;
    if (j >= kStages && !mbar_wait(&b.v_empty[st], (use - 1) & 1, a.status)) { ok = false; break; }
    mbar_arrive_expect_tx(&b.v_full[st], bytes);
    uint8_t* vdst = smem + L::kV + st * L::kTileBytes;
    for (int i = 0; i < nb; ++i)
#pragma unroll
      for (int r = 0; r < L::kRegions; ++r)
        tma_load_2d(vdst + r * L::kRegionBytes + i * bs * 128, vmap, 64 * r, rows[i], &b.v_full[st]);
    issued_v[st] = j + 1;
  }
  if (!ok) {  // let every copy this thread started land before the CTA moves on
    drain_wait(b.q, 0);
    for (int st = 0; st < kStages; ++st) {
      if (issued_k[st]) drain_wait(&b.k_full[st], ((issued_k[st] - 1) >> 1) & 1);
      if (issued_v[st]) drain_wait(&b.v_full[st], ((issued_v[st] - 1) >> 1) & 1);
    }
  }
}

// ---------------------------------------------------------------- MMA issuer

template <int D, bool kBf16>
__device__ __forceinline__ void mma_role(const AttnArgs& a, uint8_t* smem, const Bars& b, uint32_t tmem,
                                         int ntiles) {
  using L = PrefillLayout<D>;
  constexpr uint32_t kIdescQK = idesc_f16(kBf16, kTile, kTile, false, false);
  constexpr uint32_t kIdescPV = idesc_f16(kBf16, kTile, D, false, true);
  const uint32_t s_tmem = tmem, o_tmem = tmem + kTile;
  const uint32_t q_addr = smem_u32(smem + L::kQ);
  const uint32_t p_addr = smem_u32(smem + L::kP);
  bool ok = mbar_wait(b.q, 0, a.status);
  bool issued_any = false;
  for (int j = 0; ok && j <= ntiles; ++j) {
    if (j < ntiles) {
      const int st = j & 1, use = j >> 1;
      if (!mbar_wait(&b.k_full[st], use & 1, a.status)) { ok = false; break; }
      if (j >= 1 && !mbar_wait(b.s_free, (j - 1) & 1, a.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t k_addr = smem_u32(smem + L::kK + st * L::kTileBytes);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks >> 2) * L::kRegionBytes + (ks & 3) * 32;
        umma_f16_ss(s_tmem, smem_desc_sw128(q_addr + off, 16, 1024), smem_desc_sw128(k_addr + off, 16, 1024),
                    kIdescQK, ks > 0 ? 1u : 0u);
      }
      issued_any = true;
      umma_commit(b.s_full);
      umma_commit(&b.k_empty[st]);
    }
    if (j >= 1) {
      const int i = j - 1, st = i & 1, use = i >> 1;
      if (!mbar_wait(b.p_full, i & 1, a.status)) { ok = false; break; }
      if (!mbar_wait(&b.v_full[st], use & 1, a.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t v_addr = smem_u32(smem + L::kV + st * L::kTileBytes);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        const uint64_t pdesc = smem_desc_sw128(p_addr + (kk >> 2) * L::kRegionBytes + (kk & 3) * 32, 16, 1024);
        // V tile [key][d] is MN-major for O += P V: 64-column halves L::kRegionBytes
        // apart (leading offset), 8-key row groups 1024 B apart (stride offset)
        const uint64_t vdesc = smem_desc_sw128(v_addr + kk * 16 * 128, L::kRegionBytes, 1024);
        umma_f16_ss(o_tmem, pdesc, vdesc, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(b.o_done);
      umma_commit(&b.v_empty[st]);
    }
  }
  if (!ok && issued_any) {  // wait for this thread's MMAs before TMEM is released
    umma_commit(b.drain);
    drain_wait(b.drain, 0);
  }
}

// ---------------------------------------------------------------- softmax

// A wait whose outcome is the same for all 32 lanes, so that warp-collective
// instructions after it never run with lanes missing.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

template <int D, bool kBf16, int G>
__device__ __forceinline__ void softmax_role(const AttnArgs& a, uint8_t* smem, const Bars& b, uint32_t tmem, int q0,
                                             int t_begin, int ntok, int h, int nkeys, int ntiles) {
  using L = PrefillLayout<D>;
  const int r = threadIdx.x;  // row = TMEM lane
  const int warp = r >> 5;
  const int tl = r / G, g = r % G;
  const bool row_valid = tl < ntok;
  const int tok = q0 + t_begin + min(tl, ntok - 1);
  const int pos = __ldg(a.positions + tok);
  const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
  const uint32_t s_tmem = tmem + lane_off, o_tmem = tmem + kTile + lane_off;
  const uint32_t p_addr = smem_u32(smem + L::kP);
  const float c2 = a.scale_log2;
  float m = kNegInf, l = 0.f;
  bool ok = true;

  for (int j = 0; j < ntiles; ++j) {
    if (!warp_wait(b.s_full, j & 1, a.status)) { ok = false; break; }
    tc_fence_after();
    float sv[kTile];
#pragma unroll
    for (int c = 0; c < kTile / 32; ++c) {
      uint32_t t[32];
      tmem_ld32(s_tmem + 32 * c, t);
#pragma unroll
      for (int i = 0; i < 32; ++i) sv[32 * c + i] = __uint_as_float(t[i]);
    }
    tc_fence_before();
    mbar_arrive(b.s_free);

    // causal mask: key k is visible to this row iff k <= pos
    const int kb0 = kTile * j;
    if (kb0 + kTile - 1 > pos) {
#pragma unroll
      for (int i = 0; i < kTile; ++i)
        if (kb0 + i > pos) sv[i] = kNegInf;
    }
    float mx = sv[0];
#pragma unroll
    for (int i = 1; i < kTile; ++i) mx = fmaxf(mx, sv[i]);
    const float m_new = fmaxf(m, mx);
    const float ms = (m_new == kNegInf ? 0.f : m_new) * c2;
    const float alpha = ex2(fmaf(m, c2, -ms));
    float sum = 0.f;
    uint32_t pk[kTile / 2];
#pragma unroll
    for (int i = 0; i < kTile / 2; ++i) {
      const float p0 = ex2(fmaf(sv[2 * i], c2, -ms));
      const float p1 = ex2(fmaf(sv[2 * i + 1], c2, -ms));
      sum += p0 + p1;
      pk[i] = pack2<kBf16>(p0, p1);
    }
    l = fmaf(l, alpha, sum);
    m = m_new;

    if (j > 0) {  // PV of the previous tile must be done before O is rescaled and P rewritten
      if (!warp_wait(b.o_done, (j - 1) & 1, a.status)) { ok = false; break; }
      tc_fence_after();
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t t[32];
          tmem_ld32(o_tmem + 32 * c, t);
#pragma unroll
          for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
          tmem_st32(o_tmem + 32 * c, t);
        }
      }
    }
    if (j == ntiles - 1 && nkeys < kb0 + kTile) {
      // value rows past the last needed key may hold anything (even NaN, or
      // nothing loaded at all): zero them so that P = 0 contributes 0
      const int st = j & 1;
      if (!warp_wait(&b.v_full[st], (j >> 1) & 1, a.status)) { ok = false; break; }
      if (r >= nkeys - kb0) {
        const uint32_t vrow = smem_u32(smem + L::kV + st * L::kTileBytes) + r * 128;
#pragma unroll
        for (int reg = 0; reg < L::kRegions; ++reg)
#pragma unroll
          for (int c = 0; c < 8; ++c) st_shared_v4(vrow + reg * L::kRegionBytes + c * 16, 0, 0, 0, 0);
      }
    }
    // P row r, K-major with the 128-byte swizzle: keys 0-63 in region 0, 64-127 in region 1
#pragma unroll
    for (int half = 0; half < 2; ++half)
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int k = half * 32 + 4 * c;
        st_shared_v4(p_addr + half * L::kRegionBytes + r * 128 + ((c ^ (r & 7)) << 4), pk[k], pk[k + 1], pk[k + 2],
                     pk[k + 3]);
      }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(b.p_full);
  }

  if (ok && ntiles > 0 && warp_wait(b.o_done, (ntiles - 1) & 1, a.status)) {
    tc_fence_after();
    const float inv = 1.f / l;
    uint16_t* dst = static_cast<uint16_t*>(a.out) + (static_cast<size_t>(tok) * a.num_q_heads + h * G + g) * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
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
  }
}

// ---------------------------------------------------------------- kernel

template <int D, bool kBf16, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap qmap, const AttnArgs a) {
  using L = PrefillLayout<D>;
  constexpr int TQ = kTile / G;  // tokens per tile
  const int qt = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int q0 = __ldg(a.query_start_loc + s);
  const int qlen = __ldg(a.query_start_loc + s + 1) - q0;
  if (q0 < 0 || qlen < 0 || q0 + qlen > a.num_tokens) {
    if (qt == 0 && h == 0 && threadIdx.x == 0) report(a.status, KSHIPRA_DEV_BAD_LENGTHS);
    return;
  }
  if (qlen == 0 || qlen * G <= a.decode_max_rows) return;  // empty, or served by the decode kernel
  const int t_begin = qt * TQ;
  if (t_begin >= qlen) return;
  const int ntok = min(TQ, qlen - t_begin);
  const int ctx = __ldg(a.context_lens + s);
  const int pos_last = __ldg(a.positions + q0 + t_begin + ntok - 1);
  const int pos_first = __ldg(a.positions + q0 + t_begin);
  if (ctx <= 0 || ctx > a.max_blocks_per_seq * a.block_size || pos_last >= ctx || pos_first < 0 ||
      pos_first > pos_last) {
    if (h == 0 && threadIdx.x == 0) report(a.status, KSHIPRA_DEV_BAD_POSITION);
    return;
  }
  const int nkeys = pos_last + 1;  // keys 0..pos_last cover every row of the tile
  const int ntiles = ceil_div(nkeys, kTile);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  Bars b{bar, bar + 1, bar + 3, bar + 5, bar + 7, bar + 9, bar + 10, bar + 11, bar + 12, bar + 13};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + L::kNumBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(b.q, 1);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&b.k_full[st], 1);
      mbar_init(&b.k_empty[st], 1);
      mbar_init(&b.v_full[st], 1);
      mbar_init(&b.v_empty[st], 1);
    }
    mbar_init(b.s_full, 1);
    mbar_init(b.s_free, kTile);
    mbar_init(b.p_full, kTile);
    mbar_init(b.o_done, 1);
    mbar_init(b.drain, 1);
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

  if (warp < 4) {
    softmax_role<D, kBf16, G>(a, smem, b, tmem, q0, t_begin, ntok, h, nkeys, ntiles);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role<D, G>(&kmap, &vmap, &qmap, a, smem, b, s, h, q0 + t_begin, nkeys, ntiles);
  } else {
    if (lane == 0) mma_role<D, kBf16>(a, smem, b, tmem, ntiles);
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
  constexpr int TQ = kTile / G;
  dim3 grid((a.max_query_len + TQ - 1) / TQ, a.num_kv_heads, a.num_seqs);
  prefill_kernel<D, kBf16, G><<<grid, kThreads, L::kAlloc, stream>>>(kmap, vmap, qmap, a);
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

cudaError_t launch_prefill(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& qmap, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.max_query_len * a.group <= a.decode_max_rows) return cudaSuccess;
  const bool bf = a.dtype == KSHIPRA_DTYPE_BF16;
  if (a.head_dim == 128)
    return bf ? launch_prefill_g<128, true>(a, kmap, vmap, qmap, stream)
              : launch_prefill_g<128, false>(a, kmap, vmap, qmap, stream);
  return bf ? launch_prefill_g<64, true>(a, kmap, vmap, qmap, stream)
            : launch_prefill_g<64, false>(a, kmap, vmap, qmap, stream);
}

}  // namespace kshipra
