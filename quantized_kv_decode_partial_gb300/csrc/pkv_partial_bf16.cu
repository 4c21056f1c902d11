// bf16 pages: head_dim 64 / 128 / 256 with up to 64 / 64 / 32 query rows per KV head.
#include "pkv_partial_instances.cuh"

namespace pkv {

#define PKV_BF16_INSTANCES(X) \
  X(64, 1, 1) X(64, 2, 1) X(64, 4, 1) X(64, 4, 2) \
  X(128, 1, 1) X(128, 2, 1) X(128, 2, 2) X(128, 2, 4) \
  X(256, 1, 1) X(256, 1, 2) X(256, 1, 4)

PartialInfo partial_info_bf16(int d, int nq) {
  int nt, wq;
  tiles_for(d, nq, nt, wq);
#define X(D_, NT_, WQ_) \
  if (d == D_ && nt == NT_ && wq == WQ_) return info_of<16, D_, NT_, WQ_>();
  PKV_BF16_INSTANCES(X)
#undef X
  return PartialInfo{false, 0, 0, 0, 0, 0};
}

cudaError_t launch_partial_bf16(int d, int nq, const PartialParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                dim3 grid, cudaStream_t s, int dev) {
  int nt, wq;
  tiles_for(d, nq, nt, wq);
#define X(D_, NT_, WQ_) \
  if (d == D_ && nt == NT_ && wq == WQ_) return launch_of<16, D_, NT_, WQ_>(p, tk, tv, grid, s, dev);
  PKV_BF16_INSTANCES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace pkv
