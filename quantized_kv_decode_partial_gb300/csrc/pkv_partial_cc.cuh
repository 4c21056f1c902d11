// CUDA-core contraction for the partial kernel: bf16 pages, at most 4 query rows per
// KV head. The form of the pages' direct paged kernel ("@mlx-bun/inference
// 0.0.0-stage -> 1.0.0", kernels/attention/paged.ts, paged_attention_partial: per key,
// a dot product of q with the key row reduced across the SIMD group, then the
// weighted sum of value rows with f32 weights), on a chunk staged in shared memory.
//
// Layout: a lane owns 8 consecutive head dims (one 16-byte vector of a row), so a
// row of D dims spans D/8 lanes and one warp-wide load covers 256/D rows. Per chunk of
// 16 rows a lane therefore sees 16*D/256 keys; it accumulates its 8-dim partial dot
// products for those keys and every query row with packed f32 FMAs (two lanes of
// f32 per instruction), and a transposed butterfly across the lanes of a row (each
// step halves the keys a lane keeps and adds its partner's half) leaves every lane
// with the full score of one key. The weights p = 2^(x - m) stay in f32 (the online
// softmax as in the tensor-core form), go through a small per-warp buffer in shared
// memory to the lanes that hold that key's value rows, and the value rows are
// accumulated with packed f32 FMAs, each lane into its own 8 dims.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

template <int D, int NQC>
struct CcShape {
  static_assert(D == 64 || D == 128 || D == 256, "head dims 64, 128, 256");
  static_assert(NQC == 2 || NQC == 4, "2 or 4 query rows per KV head (padded)");
  static constexpr int kLanesPerRow = D / 8;               // 16-byte vectors per row
  static constexpr int kRowsPerLoad = 32 / kLanesPerRow;   // rows one warp-wide load covers
  static constexpr int kLoads = 16 / kRowsPerLoad;         // loads per 16-row chunk = keys per lane
  static constexpr int kBoxBytes = 16 * 128;               // one 128-byte segment of 16 rows
  static constexpr int kPBufFloats = 16 * 4;               // weights of one chunk: [row][query]
  // After the transposed butterfly, lane bits below kDupBit name the key slot, bit kDupBit
  // tells the two lanes of a row that hold the same key apart (a row spans twice as many
  // lanes as it has keys per lane), and the bits above are the row within a load.
  static constexpr int kDupBit = kLoads == 16 ? 4 : kLoads == 8 ? 3 : 2;
  static_assert(kLanesPerRow == 2 * kLoads, "two lanes per key after the butterfly");
};

// Shared-memory address of the 16-byte vector holding dims d0 .. d0+7 of row r of a
// plane staged as 128-byte segments ([segment][16 rows][128 B], 128-byte swizzle).
__device__ __forceinline__ uint32_t cc_vec_addr(uint32_t plane, int r, int d0) {
  const int c16 = d0 >> 3;  // 16-byte vector index within the row
  return plane + (c16 >> 3) * (16 * 128) + r * 128 + (((c16 & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// The two bf16 values of a word (low half first) as an f32 pair, exactly.
__device__ __forceinline__ float2 bf16x2_pair(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Index (0 .. kLoads-1) of the key a lane holds after the transposed butterfly: at
// step b the lanes with bit b set keep the upper half of the keys.
template <int D, int NQC>
__device__ __forceinline__ int cc_key_slot(int lane) {
  using S = CcShape<D, NQC>;
  int slot = 0;
#pragma unroll
  for (int b = 0; (S::kLoads >> b) > 1; ++b) slot += ((lane >> b) & 1) * (S::kLoads >> (b + 1));
  return slot;
}

// Sums each value over the kLanesPerRow lanes of a row, transposed: on entry v[j][qi]
// is this lane's partial for key slot j; on exit v[0][qi] is the full sum for slot
// cc_key_slot(lane).
template <int D, int NQC>
__device__ __forceinline__ void cc_transpose_reduce(float (&v)[CcShape<D, NQC>::kLoads][NQC], int lane) {
  using S = CcShape<D, NQC>;
#pragma unroll
  for (int b = 0; (1 << b) < S::kLanesPerRow; ++b) {
    const int delta = 1 << b;
    const int n = S::kLoads >> b;  // values this lane still holds (1 once the keys are spread)
    if (n > 1) {
      const int half = n >> 1;
      const bool upper = (lane >> b) & 1;
#pragma unroll
      for (int i = 0; i < half; ++i)
#pragma unroll
        for (int qi = 0; qi < NQC; ++qi) {
          const float send = upper ? v[i][qi] : v[i + half][qi];
          const float keep = upper ? v[i + half][qi] : v[i][qi];
          v[i][qi] = keep + __shfl_xor_sync(0xffffffffu, send, delta);
        }
    } else {
#pragma unroll
      for (int qi = 0; qi < NQC; ++qi) v[0][qi] += __shfl_xor_sync(0xffffffffu, v[0][qi], delta);
    }
  }
}

// One staged chunk of 16 bf16 rows (first cache row kbase) for NQC query rows:
// online-softmax update of (m, l, o). m and l are per query row (m warp-uniform; l
// this lane's share: only the first of the lanes that hold a key adds its weight), o
// this lane's 8 dims. pbuf is this warp's 16 x 4 floats of shared memory.
template <int D, int NQC>
__device__ __forceinline__ void cc_chunk(uint32_t kpl, uint32_t vpl, float* pbuf, const float2 (&qv)[NQC][4],
                                         float2 (&o)[NQC][4], float (&m)[NQC], float (&l)[NQC], int lane, int kbase,
                                         int len, int vis_base, int win, int n_query, bool full_vis, bool stale,
                                         float score_scale) {
  using S = CcShape<D, NQC>;
  const int d0 = (lane % S::kLanesPerRow) * 8;
  const int rsub = lane / S::kLanesPerRow;

  // ---- partial dot products of this lane's 8 dims, for each of its keys
  float sc[S::kLoads][NQC];
#pragma unroll
  for (int j = 0; j < S::kLoads; ++j) {
    const uint4 w = lds128(cc_vec_addr(kpl, j * S::kRowsPerLoad + rsub, d0));
    const float2 k0 = bf16x2_pair(w.x), k1 = bf16x2_pair(w.y), k2 = bf16x2_pair(w.z), k3 = bf16x2_pair(w.w);
#pragma unroll
    for (int qi = 0; qi < NQC; ++qi) {
      float2 a = __fmul2_rn(k0, qv[qi][0]);
      a = __ffma2_rn(k1, qv[qi][1], a);
      a = __ffma2_rn(k2, qv[qi][2], a);
      a = __ffma2_rn(k3, qv[qi][3], a);
      sc[j][qi] = a.x + a.y;
    }
  }
  cc_transpose_reduce<D, NQC>(sc, lane);

  // ---- scores of this lane's key (base 2), causal tail / window / stale rows
  const int row = cc_key_slot<D, NQC>(lane) * S::kRowsPerLoad + rsub;
  const int key = kbase + row;
  float x[NQC];
#pragma unroll
  for (int qi = 0; qi < NQC; ++qi) {
    x[qi] = sc[0][qi] * score_scale;
    if (!full_vis) {
      const int qpos = qi % n_query;
      const bool vis = key < vis_base + qpos && (win == 0 || key >= vis_base + qpos - win);
      x[qi] = vis ? x[qi] : -INFINITY;
    }
  }

  // ---- online softmax: the lazy running maximum of the tensor-core form
  bool below = true;
#pragma unroll
  for (int qi = 0; qi < NQC; ++qi) below &= x[qi] <= m[qi];
  if (!__all_sync(0xffffffffu, below)) {
#pragma unroll
    for (int qi = 0; qi < NQC; ++qi) {
      float mx = x[qi];
#pragma unroll
      for (int delta = 1; delta < 32; delta <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, delta));
      const float mnew = fmaxf(m[qi], mx);
      if (mnew != m[qi]) {
        const float c = fast_exp2(m[qi] - mnew);  // 0 when m was -inf
        l[qi] *= c;
        const float2 cc = make_float2(c, c);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[qi][i] = __fmul2_rn(o[qi][i], cc);
        m[qi] = mnew;
      }
    }
  }
  // the first of the two lanes holding a key counts and publishes its weights
  const bool first = ((lane >> S::kDupBit) & 1) == 0;
  float p[NQC];
#pragma unroll
  for (int qi = 0; qi < NQC; ++qi) {
    const float muse = m[qi] == -INFINITY ? 0.f : m[qi];
    p[qi] = fast_exp2(x[qi] - muse);
    l[qi] += first ? p[qi] : 0.f;
  }
  if (first) {
    if constexpr (NQC == 4) {
      *reinterpret_cast<float4*>(pbuf + 4 * row) = make_float4(p[0], p[1], p[2], p[3]);
    } else {
      *reinterpret_cast<float2*>(pbuf + 4 * row) = make_float2(p[0], p[1]);
    }
  }
  __syncwarp();

  // ---- o += p * V over this lane's value rows and 8 dims
#pragma unroll
  for (int j = 0; j < S::kLoads; ++j) {
    const int r = j * S::kRowsPerLoad + rsub;
    uint4 w = lds128(cc_vec_addr(vpl, r, d0));
    if (stale && kbase + r >= len) w = make_uint4(0u, 0u, 0u, 0u);  // stale storage may hold NaN
    const float2 v0 = bf16x2_pair(w.x), v1 = bf16x2_pair(w.y), v2 = bf16x2_pair(w.z), v3 = bf16x2_pair(w.w);
    float pw[NQC];
    if constexpr (NQC == 4) {
      const float4 t = *reinterpret_cast<const float4*>(pbuf + 4 * r);
      pw[0] = t.x;
      pw[1] = t.y;
      pw[2] = t.z;
      pw[3] = t.w;
    } else {
      const float2 t = *reinterpret_cast<const float2*>(pbuf + 4 * r);
      pw[0] = t.x;
      pw[1] = t.y;
    }
#pragma unroll
    for (int qi = 0; qi < NQC; ++qi) {
      const float2 pp = make_float2(pw[qi], pw[qi]);
      o[qi][0] = __ffma2_rn(v0, pp, o[qi][0]);
      o[qi][1] = __ffma2_rn(v1, pp, o[qi][1]);
      o[qi][2] = __ffma2_rn(v2, pp, o[qi][2]);
      o[qi][3] = __ffma2_rn(v3, pp, o[qi][3]);
    }
  }
}

}  // namespace pkv
