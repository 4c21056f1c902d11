// Internal launch interface between the C-ABI host code and the kernel
// translation units (one per page format, compiled in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "pkv_common.cuh"

namespace pkv {

// Static shape of one partial-kernel instantiation.
struct PartialInfo {
  bool exists;
  int threads;
  int smem_bytes;
  int chunk_rows;
  int box_row_bytes;    // bytes of one TMA box row of the K plane (64 or 128)
  int box_row_bytes_v;  // ... of the V plane
  int tensor_elem_bytes;  // element size of the pool tensor maps (2 bf16, 1 affine codes)
  int page_groups;        // page groups per CTA (rings of stages, each read by its query-group warps)
};

// Partial-kernel instantiation for key head dim dk, value head dim dv and `nq` query
// rows per KV head; `solo` selects the variant for grids of at most one CTA per SM
// (exists = false where there is none).
PartialInfo partial_info_bf16(int dk, int dv, int nq, bool solo);
PartialInfo partial_info_u4(int dk, int dv, int nq, bool solo);
PartialInfo partial_info_u8(int dk, int dv, int nq, bool solo);
// bf16 pages with the CUDA-core contraction (up to 4 query rows per KV head, equal head dims)
PartialInfo partial_info_bf16_cc(int dk, int dv, int nq, bool solo);

cudaError_t launch_partial_bf16(int dk, int dv, int nq, bool solo, const PartialParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, dim3 grid, cudaStream_t stream, int device);
cudaError_t launch_partial_u4(int dk, int dv, int nq, bool solo, const PartialParams& p, const CUtensorMap& tk,
                              const CUtensorMap& tv, dim3 grid, cudaStream_t stream, int device);
cudaError_t launch_partial_u8(int dk, int dv, int nq, bool solo, const PartialParams& p, const CUtensorMap& tk,
                              const CUtensorMap& tv, dim3 grid, cudaStream_t stream, int device);
cudaError_t launch_partial_bf16_cc(int dk, int dv, int nq, bool solo, const PartialParams& p, const CUtensorMap& tk,
                                   const CUtensorMap& tv, dim3 grid, cudaStream_t stream, int device);

// Balanced-schedule instantiations (kModeBalanced) for the same shapes' grids of several
// CTAs per SM; the CTAs of one per SM on `device` (the current device; 0 on an error).
PartialInfo partial_info_bf16_bal(int dk, int dv, int nq);
PartialInfo partial_info_u4_bal(int dk, int dv, int nq);
PartialInfo partial_info_u8_bal(int dk, int dv, int nq);
int partial_bal_ctas_per_sm_bf16(int dk, int dv, int nq, int device);
int partial_bal_ctas_per_sm_u4(int dk, int dv, int nq, int device);
int partial_bal_ctas_per_sm_u8(int dk, int dv, int nq, int device);
cudaError_t launch_partial_bf16_bal(int dk, int dv, int nq, const PartialParams& p, const CUtensorMap& tk,
                                    const CUtensorMap& tv, dim3 grid, cudaStream_t stream, int device);
cudaError_t launch_partial_u4_bal(int dk, int dv, int nq, const PartialParams& p, const CUtensorMap& tk,
                                  const CUtensorMap& tv, dim3 grid, cudaStream_t stream, int device);
cudaError_t launch_partial_u8_bal(int dk, int dv, int nq, const PartialParams& p, const CUtensorMap& tk,
                                  const CUtensorMap& tv, dim3 grid, cudaStream_t stream, int device);

// Instantiations for pools of blocks smaller than a chunk (PartialParams.piece_log2 > 0) of
// the same shapes' grids of several CTAs per SM; their PartialInfo is that of those grids.
cudaError_t launch_partial_bf16_pc(int dk, int dv, int nq, const PartialParams& p, const CUtensorMap& tk,
                                   const CUtensorMap& tv, dim3 grid, cudaStream_t stream, int device);
cudaError_t launch_partial_u4_pc(int dk, int dv, int nq, const PartialParams& p, const CUtensorMap& tk,
                                 const CUtensorMap& tv, dim3 grid, cudaStream_t stream, int device);
cudaError_t launch_partial_u8_pc(int dk, int dv, int nq, const PartialParams& p, const CUtensorMap& tk,
                                 const CUtensorMap& tv, dim3 grid, cudaStream_t stream, int device);

int merge_groups(int head_dim, int max_partitions);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
cudaError_t launch_gather(const GatherParams& p, int num_seqs, cudaStream_t stream);

bool append_supported(int bits, int head_dim, int v_head_dim);
cudaError_t launch_append(const AppendParams& p, int bits, int head_dim, int v_head_dim, int num_seqs,
                          cudaStream_t stream);

}  // namespace pkv
