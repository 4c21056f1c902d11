// Write side of the paged cache: append a step's new K/V rows into their pages,
// quantising affine pages on the way (the pages' PagedKVCache.append splitting
// rows along block boundaries and BlockPool.writeBlock quantising each piece,
// "@mlx-bun/inference 0.0.0-stage -> 1.0.0", state/paged/cache.ts).
//
// Affine quantisation per row and 64-dim group, every step in f32 (the pages do
// not give the quantiser's formula; this is the plain min/max reading):
//     scale = bf16((max - min) / (2^bits - 1)), bias = bf16(min)
//     code  = clamp(rint((x - bias) / scale), 0, 2^bits - 1)   (0 when scale is 0)
// packed lowest bits first into u32 words.
#include "pkv_launch.h"

namespace pkv {

namespace {

constexpr int kAppendWarps = 4;  // KV heads per CTA

// One warp per (sequence, new row, KV head); lane l holds dims [l*E, l*E + E).
template <int BITS, int D>
__global__ void __launch_bounds__(kAppendWarps * 32) pkv_append_kernel(const __grid_constant__ AppendParams p) {
  constexpr int E = D / 32;  // elements per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * kAppendWarps + warp;
  const int j = blockIdx.y, b = blockIdx.z;
  if (h >= p.num_kv_heads) return;
  const int len = p.seq_lens[b];
  if (len < 0 || len + p.n_new > p.max_blocks * p.block_size) {
    if (lane == 0 && h == 0 && j == 0 && p.error_flag) atomicOr(p.error_flag, kDevErrBadSeqLen);
    return;
  }
  const int t = len + j;
  const int phys = p.block_tables[static_cast<size_t>(b) * p.max_blocks + t / p.block_size];
  if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
    if (lane == 0 && p.error_flag) atomicOr(p.error_flag, kDevErrBadBlock);
    return;
  }
  const size_t row = (static_cast<size_t>(phys) * p.num_kv_heads + h) * p.block_size + t % p.block_size;
  const size_t src_row = ((static_cast<size_t>(b) * p.num_kv_heads + h) * p.n_new + j);

#pragma unroll
  for (int plane = 0; plane < 2; ++plane) {
    const __nv_bfloat16* src = (plane == 0 ? p.k_new : p.v_new) + src_row * D + lane * E;
    if constexpr (BITS == 16) {
      __nv_bfloat16* dst = (plane == 0 ? p.k_pool_bf16 : p.v_pool_bf16) + row * D + lane * E;
      if constexpr (E == 8) {
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
      } else if constexpr (E == 4) {
        *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(src);
      } else {
        *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
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
      uint32_t packed[E * BITS / 32 > 0 ? E * BITS / 32 : 1] = {};
      uint32_t half_word = 0;  // 4-bit codes of a lane with E = 4 fill 16 bits
#pragma unroll
      for (int e = 0; e < E; ++e) {
        uint32_t code = 0;
        if (s != 0.f) code = static_cast<uint32_t>(fminf(fmaxf(rintf(__fdiv_rn(x[e] - bias, s)), 0.f), kLevels));
        if constexpr (E * BITS >= 32) {
          packed[(e * BITS) / 32] |= code << ((e * BITS) % 32);
        } else {
          half_word |= code << (e * BITS);
        }
      }
      uint32_t* words = (plane == 0 ? p.k_pool_words : p.v_pool_words) + row * (D * BITS / 32);
      if constexpr (E * BITS >= 32) {
#pragma unroll
        for (int w = 0; w < E * BITS / 32; ++w) words[lane * (E * BITS / 32) + w] = packed[w];
      } else {  // two lanes per word: the even lane holds the low half
        const uint32_t other = __shfl_xor_sync(0xffffffffu, half_word, 1);
        if ((lane & 1) == 0) words[lane >> 1] = half_word | (other << 16);
      }
      if (lane % kLanesPerGroup == 0) {
        const int grp = lane / kLanesPerGroup;
        (plane == 0 ? p.k_scales : p.v_scales)[row * (D / 64) + grp] = s16;
        (plane == 0 ? p.k_biases : p.v_biases)[row * (D / 64) + grp] = b16;
      }
    }
  }
}

template <int BITS, int D>
cudaError_t launch_append_of(const AppendParams& p, int num_seqs, cudaStream_t stream) {
  dim3 grid((p.num_kv_heads + kAppendWarps - 1) / kAppendWarps, p.n_new, num_seqs);
  pkv_append_kernel<BITS, D><<<grid, kAppendWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool append_supported(int bits, int head_dim) {
  if (bits == 16) return head_dim == 64 || head_dim == 128 || head_dim == 256;
  return (bits == 4 || bits == 8) && (head_dim == 128 || head_dim == 256);
}

cudaError_t launch_append(const AppendParams& p, int bits, int head_dim, int num_seqs, cudaStream_t stream) {
  if (p.n_new == 0) return cudaSuccess;
  if (bits == 16 && head_dim == 64) return launch_append_of<16, 64>(p, num_seqs, stream);
  if (bits == 16 && head_dim == 128) return launch_append_of<16, 128>(p, num_seqs, stream);
  if (bits == 16 && head_dim == 256) return launch_append_of<16, 256>(p, num_seqs, stream);
  if (bits == 4 && head_dim == 128) return launch_append_of<4, 128>(p, num_seqs, stream);
  if (bits == 4 && head_dim == 256) return launch_append_of<4, 256>(p, num_seqs, stream);
  if (bits == 8 && head_dim == 128) return launch_append_of<8, 128>(p, num_seqs, stream);
  if (bits == 8 && head_dim == 256) return launch_append_of<8, 256>(p, num_seqs, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
