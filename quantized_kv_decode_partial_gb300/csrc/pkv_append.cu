// Write side of the paged cache: append a step's new K/V rows into their pages,
// quantising affine pages on the way (the pages' PagedKVCache.append splitting
// rows along block boundaries and BlockPool.writeBlock quantising each piece,
// "@mlx-bun/inference 0.0.0-stage -> 1.0.0", state/paged/cache.ts). The row
// writer and its quantiser live in pkv_append.cuh.
#include "pkv_append.cuh"
#include "pkv_launch.h"

namespace pkv {

namespace {

constexpr int kAppendWarps = 4;  // KV heads per CTA

// One warp per (sequence, new row, KV head).
template <int BITS, int DK, int DV>
__global__ void __launch_bounds__(kAppendWarps * 32) pkv_append_kernel(const __grid_constant__ AppendParams p) {
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
  const size_t src_row = (static_cast<size_t>(b) * p.num_kv_heads + h) * p.n_new + j;
  append_row<BITS, DK, DV>(p.k_new + src_row * DK, p.v_new + src_row * DV, p.dst, row, lane);
}

template <int BITS, int DK, int DV>
cudaError_t launch_append_of(const AppendParams& p, int num_seqs, cudaStream_t stream) {
  dim3 grid((p.num_kv_heads + kAppendWarps - 1) / kAppendWarps, p.n_new, num_seqs);
  pkv_append_kernel<BITS, DK, DV><<<grid, kAppendWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

// (bits, key head dim, value head dim) combinations of the append kernel: every
// layout the partial kernel reads.
#define PKV_APPEND_SHAPES(X)                                                       \
  X(16, 64, 64) X(16, 128, 128) X(16, 256, 256) X(16, 192, 128) X(16, 256, 128) \
  X(16, 128, 256) X(4, 128, 128) X(4, 256, 256) X(4, 256, 128) X(4, 128, 256)   \
  X(8, 128, 128) X(8, 256, 256) X(8, 256, 128) X(8, 128, 256)

}  // namespace

bool append_supported(int bits, int head_dim, int v_head_dim) {
#define X(B_, DK_, DV_) \
  if (bits == B_ && head_dim == DK_ && v_head_dim == DV_) return true;
  PKV_APPEND_SHAPES(X)
#undef X
  return false;
}

cudaError_t launch_append(const AppendParams& p, int bits, int head_dim, int v_head_dim, int num_seqs,
                          cudaStream_t stream) {
  if (p.n_new == 0) return cudaSuccess;
#define X(B_, DK_, DV_) \
  if (bits == B_ && head_dim == DK_ && v_head_dim == DV_) return launch_append_of<B_, DK_, DV_>(p, num_seqs, stream);
  PKV_APPEND_SHAPES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace pkv
