// bf16 pages: head_dim 64 (up to 32 query rows per KV head), 128 (up to 16), 256 (up to 8).
#include "pkv_partial_instances.cuh"

namespace pkv {

PartialInfo partial_info_bf16(int d, int nt) {
  if (d == 64 && nt == 1) return info_of<16, 64, 1>();
  if (d == 64 && nt == 2) return info_of<16, 64, 2>();
  if (d == 64 && nt == 4) return info_of<16, 64, 4>();
  if (d == 128 && nt == 1) return info_of<16, 128, 1>();
  if (d == 128 && nt == 2) return info_of<16, 128, 2>();
  if (d == 256 && nt == 1) return info_of<16, 256, 1>();
  return PartialInfo{false, 0, 0, 0, 0, 0};
}

cudaError_t launch_partial_bf16(int d, int nt, const PartialParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, dim3 grid, cudaStream_t s) {
  if (d == 64 && nt == 1) return launch_of<16, 64, 1>(p, tk, tv, grid, s);
  if (d == 64 && nt == 2) return launch_of<16, 64, 2>(p, tk, tv, grid, s);
  if (d == 64 && nt == 4) return launch_of<16, 64, 4>(p, tk, tv, grid, s);
  if (d == 128 && nt == 1) return launch_of<16, 128, 1>(p, tk, tv, grid, s);
  if (d == 128 && nt == 2) return launch_of<16, 128, 2>(p, tk, tv, grid, s);
  if (d == 256 && nt == 1) return launch_of<16, 256, 1>(p, tk, tv, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
