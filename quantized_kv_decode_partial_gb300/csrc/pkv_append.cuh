// One appended K/V row written into its page, quantising affine pages on the
// way: the per-row step of the pages' PagedKVCache.append, which splits a
// step's rows along block boundaries, and BlockPool.writeBlock, which quantises
// each piece ("@mlx-bun/inference 0.0.0-stage -> 1.0.0", state/paged/cache.ts).
// Used by the append kernel and by the fused append-then-attend prologue of the
// partial kernel, so both write the same bits.
//
// Affine quantisation per row and 64-dim group, every step in f32 (the pages do
// not give the quantiser's formula; this is the plain min/max reading):
//     scale = bf16((max - min) / (2^bits - 1)), bias = bf16(min)
//     code  = clamp(rint((x - bias) / scale), 0, 2^bits - 1)   (0 when scale is 0)
// packed lowest bits first into u32 words.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

// Writes one row of D values from `src` (bf16) into pool row `row` of one plane: a
// bf16 row, or codes plus the row's per-group scale and bias. Warp-collective: lane
// l handles dims [l*E, l*E + E), E = D / 32; every lane of the warp must call it.
template <int BITS, int D>
__device__ __forceinline__ void append_plane(const __nv_bfloat16* src_row, __nv_bfloat16* pool_bf16,
                                             uint32_t* pool_words, __nv_bfloat16* scales, __nv_bfloat16* biases,
                                             size_t row, int lane) {
  constexpr int E = D / 32;  // elements per lane
  static_assert(D % 64 == 0 || (BITS == 16 && D % 32 == 0), "whole lanes (and whole 64-dim groups for affine)");
  const __nv_bfloat16* src = src_row + lane * E;
  if constexpr (BITS == 16) {
    __nv_bfloat16* out = pool_bf16 + row * D + lane * E;
    if constexpr (E == 8) {
      *reinterpret_cast<uint4*>(out) = *reinterpret_cast<const uint4*>(src);
    } else if constexpr (E == 4) {
      *reinterpret_cast<uint2*>(out) = *reinterpret_cast<const uint2*>(src);
    } else {
#pragma unroll
      for (int w = 0; w < E / 2; ++w)
        reinterpret_cast<uint32_t*>(out)[w] = reinterpret_cast<const uint32_t*>(src)[w];
    }
  } else {
    static_assert(D == 128 || D == 256, "affine head dims 128 or 256");
    constexpr int kLanesPerGroup = 64 / E;
    constexpr float kLevels = static_cast<float>((1 << BITS) - 1);
    float x[E];
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(src + e);
      x[e] = __low2float(v);
      x[e + 1] = __high2float(v);
    }
    float lo = x[0], hi = x[0];
#pragma unroll
    for (int e = 1; e < E; ++e) {
      lo = fminf(lo, x[e]);
      hi = fmaxf(hi, x[e]);
    }
#pragma unroll
    for (int off = 1; off < kLanesPerGroup; off <<= 1) {  // the group's lanes are consecutive
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    }
    const __nv_bfloat16 s16 = __float2bfloat16_rn(__fdiv_rn(hi - lo, kLevels));
    const __nv_bfloat16 b16 = __float2bfloat16_rn(lo);
    const float s = __bfloat162float(s16), bias = __bfloat162float(b16);
    // (x - bias) / s correctly rounded decides each code. The product with the correctly
    // rounded reciprocal is within 1.5 * 2^-23 relative of that quotient. Outside
    // [-0.5, 2^bits - 0.5] both clamp to the same code; inside, the two differ by less
    // than 2^-14, so the product rounds to the same integer unless it lies within 2^-13
    // of a half-integer. Those few take the division itself.
    const float rs = s != 0.f ? __frcp_rn(s) : 0.f;
    uint32_t packed[E * BITS / 32 > 0 ? E * BITS / 32 : 1] = {};
    uint32_t half_word = 0;  // 4-bit codes of a lane with E = 4 fill 16 bits
#pragma unroll
    for (int e = 0; e < E; ++e) {
      uint32_t code = 0;
      if (s != 0.f) {
        const float d = x[e] - bias;
        float qt = d * rs;
        if (fabsf(qt - floorf(qt) - 0.5f) < 1.f / 8192.f) qt = __fdiv_rn(d, s);
        code = static_cast<uint32_t>(fminf(fmaxf(rintf(qt), 0.f), kLevels));
      }
      if constexpr (E * BITS >= 32) {
        packed[(e * BITS) / 32] |= code << ((e * BITS) % 32);
      } else {
        half_word |= code << (e * BITS);
      }
    }
    uint32_t* words = pool_words + row * (D * BITS / 32);
    if constexpr (E * BITS >= 32) {
#pragma unroll
      for (int w = 0; w < E * BITS / 32; ++w) words[lane * (E * BITS / 32) + w] = packed[w];
    } else {  // two lanes per word: the even lane holds the low half
      const uint32_t other = __shfl_xor_sync(0xffffffffu, half_word, 1);
      if ((lane & 1) == 0) words[lane >> 1] = half_word | (other << 16);
    }
    if (lane % kLanesPerGroup == 0) {
      const int grp = lane / kLanesPerGroup;
      scales[row * (D / 64) + grp] = s16;
      biases[row * (D / 64) + grp] = b16;
    }
  }
}

// Writes K row `k_src` (DK values) and V row `v_src` (DV values) to pool row `row`
// (= (phys * HK + h) * BS + offset in block) of their planes. Warp-collective.
template <int BITS, int DK, int DV>
__device__ __forceinline__ void append_row(const __nv_bfloat16* k_src, const __nv_bfloat16* v_src,
                                           const AppendTarget& dst, size_t row, int lane) {
  append_plane<BITS, DK>(k_src, dst.k_pool_bf16, dst.k_pool_words, dst.k_scales, dst.k_biases, row, lane);
  append_plane<BITS, DV>(v_src, dst.v_pool_bf16, dst.v_pool_words, dst.v_scales, dst.v_biases, row, lane);
}

}  // namespace pkv
