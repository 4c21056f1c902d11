// Affine 8-bit pages: head_dim 128 (up to 16 query rows per KV head) and 256 (up to 8).
#include "pkv_partial_instances.cuh"

namespace pkv {

PartialInfo partial_info_u8(int d, int nt) {
  if (d == 128 && nt == 1) return info_of<8, 128, 1>();
  if (d == 128 && nt == 2) return info_of<8, 128, 2>();
  if (d == 256 && nt == 1) return info_of<8, 256, 1>();
  return PartialInfo{false, 0, 0, 0, 0, 0};
}

cudaError_t launch_partial_u8(int d, int nt, const PartialParams& p, const CUtensorMap& tk,
                              const CUtensorMap& tv, dim3 grid, cudaStream_t s) {
  if (d == 128 && nt == 1) return launch_of<8, 128, 1>(p, tk, tv, grid, s);
  if (d == 128 && nt == 2) return launch_of<8, 128, 2>(p, tk, tv, grid, s);
  if (d == 256 && nt == 1) return launch_of<8, 256, 1>(p, tk, tv, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
