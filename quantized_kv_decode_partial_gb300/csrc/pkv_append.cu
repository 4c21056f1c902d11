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
template <int BITS, int D>
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
  append_row<BITS, D>(p.k_new + src_row * D, p.v_new + src_row * D, p.dst, row, lane);
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
