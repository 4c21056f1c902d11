// Affine 8-bit pages: head_dim 128 / 256 with up to 64 / 32 query rows per KV head.
#include "pkv_partial_instances.cuh"

namespace pkv {

#define PKV_U8_INSTANCES(X) \
  X(128, 1, 1) X(128, 2, 1) X(128, 2, 2) X(128, 2, 4) \
  X(256, 1, 1) X(256, 1, 2) X(256, 1, 4)

PartialInfo partial_info_u8(int d, int nq) {
  int nt, wq;
  tiles_for(d, nq, nt, wq);
#define X(D_, NT_, WQ_) \
  if (d == D_ && nt == NT_ && wq == WQ_) return info_of<8, D_, NT_, WQ_>();
  PKV_U8_INSTANCES(X)
#undef X
  return PartialInfo{false, 0, 0, 0, 0, 0};
}

cudaError_t launch_partial_u8(int d, int nq, const PartialParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              dim3 grid, cudaStream_t s, int dev) {
  int nt, wq;
  tiles_for(d, nq, nt, wq);
#define X(D_, NT_, WQ_) \
  if (d == D_ && nt == NT_ && wq == WQ_) return launch_of<8, D_, NT_, WQ_>(p, tk, tv, grid, s, dev);
  PKV_U8_INSTANCES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace pkv
