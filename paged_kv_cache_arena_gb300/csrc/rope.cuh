// RoPE rotation shared by the append kernel, the fused decode step and the
// prefill kernel's in-place query rotation.
//
// Pages "Building Kshipra" part 3 (kshipra-3), section 4: new tokens are
// rotated at their absolute positions.  Pairs (i, i + d/2) rotate by the
// angle of frequency i:
//   y_i = x_i c - x_{i+d/2} s,  y_{i+d/2} = x_{i+d/2} c + x_i s
// computed in float32 from the caller's (cos, sin) table with separately
// rounded products and one rounded add or subtract, then rounded once to the
// storage type, so every path that rotates a row gets the same bits.
#pragma once

#include "common.cuh"

namespace kshipra {

// Storage bits -> float32 (exact).
template <bool kBf16>
__device__ __forceinline__ float bits_to_float(uint32_t h) {
  if constexpr (kBf16)
    return __uint_as_float(h << 16);
  else
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// Rotated values of elements e, e + 1 (e even) of one head row, packed two per
// word.  own: the row's elements e, e + 1; partner: elements e +- d/2, e + 1 +-
// d/2; cs: (c, s) of frequencies f, f + 1 with f = e mod d/2; upper: e >= d/2.
template <bool kBf16>
__device__ __forceinline__ uint32_t rope_pair(uint32_t own, uint32_t partner, float4 cs, bool upper) {
  const float x0 = bits_to_float<kBf16>(own & 0xFFFF), x1 = bits_to_float<kBf16>(own >> 16);
  const float y0 = bits_to_float<kBf16>(partner & 0xFFFF), y1 = bits_to_float<kBf16>(partner >> 16);
  float r0, r1;
  if (upper) {  // y_{i+d/2} = x_{i+d/2} c + x_i s
    r0 = __fadd_rn(__fmul_rn(x0, cs.x), __fmul_rn(y0, cs.y));
    r1 = __fadd_rn(__fmul_rn(x1, cs.z), __fmul_rn(y1, cs.w));
  } else {  // y_i = x_i c - x_{i+d/2} s
    r0 = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(y0, cs.y));
    r1 = __fsub_rn(__fmul_rn(x1, cs.z), __fmul_rn(y1, cs.w));
  }
  return static_cast<uint32_t>(round_f32<kBf16>(r0)) | (static_cast<uint32_t>(round_f32<kBf16>(r1)) << 16);
}

// Rotates pairs (i, i + d/2) and (i + 1, i + 1 + d/2) of one head row from src
// into dst (i even, i < d/2); cs is the position's [d/2][2] table row.
template <bool kBf16>
__device__ __forceinline__ void rotate_two_pairs(const uint16_t* src, uint16_t* dst, int i, int half,
                                                 const float* cs) {
  const uint32_t lo = *reinterpret_cast<const uint32_t*>(src + i);
  const uint32_t hi = *reinterpret_cast<const uint32_t*>(src + i + half);
  const float4 t = *reinterpret_cast<const float4*>(cs + 2 * i);  // c_i, s_i, c_i+1, s_i+1
  *reinterpret_cast<uint32_t*>(dst + i) = rope_pair<kBf16>(lo, hi, t, false);
  *reinterpret_cast<uint32_t*>(dst + i + half) = rope_pair<kBf16>(hi, lo, t, true);
}

// Rotated pairs (e + k, e + k + d/2), k = 0..7, of one head row: lo holds
// elements e.., hi elements e + d/2..; cs_e points at the (cos, sin) entries
// of frequencies e.. (the position's table row + 2 e).  Each element is
// rotated exactly as rope_pair rotates it.
template <bool kBf16>
__device__ __forceinline__ void rotate_eight_pairs_vals(uint4 lo, uint4 hi, const float* cs_e, uint4& ylo,
                                                        uint4& yhi) {
  const float4* c4 = reinterpret_cast<const float4*>(cs_e);
  const float4 t0 = __ldg(c4), t1 = __ldg(c4 + 1), t2 = __ldg(c4 + 2), t3 = __ldg(c4 + 3);
  ylo.x = rope_pair<kBf16>(lo.x, hi.x, t0, false);
  ylo.y = rope_pair<kBf16>(lo.y, hi.y, t1, false);
  ylo.z = rope_pair<kBf16>(lo.z, hi.z, t2, false);
  ylo.w = rope_pair<kBf16>(lo.w, hi.w, t3, false);
  yhi.x = rope_pair<kBf16>(hi.x, lo.x, t0, true);
  yhi.y = rope_pair<kBf16>(hi.y, lo.y, t1, true);
  yhi.z = rope_pair<kBf16>(hi.z, lo.z, t2, true);
  yhi.w = rope_pair<kBf16>(hi.w, lo.w, t3, true);
}

// Rotates pairs (e + k, e + k + d/2), k = 0..7, of one head row into dst
// with 16-byte stores (e a multiple of 8, e < d/2; rows 16-byte aligned),
// from the row's words already loaded (lo: elements e.., hi: e + d/2..); cs
// is the position's [d/2][2] table row.
template <bool kBf16>
__device__ __forceinline__ void rotate_eight_pairs(uint4 lo, uint4 hi, uint16_t* dst, int e, int half,
                                                   const float* cs) {
  uint4 ylo, yhi;
  rotate_eight_pairs_vals<kBf16>(lo, hi, cs + 2 * e, ylo, yhi);
  *reinterpret_cast<uint4*>(dst + e) = ylo;
  *reinterpret_cast<uint4*>(dst + e + half) = yhi;
}

}  // namespace kshipra
