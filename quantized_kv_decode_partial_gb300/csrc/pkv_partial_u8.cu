// Affine 8-bit pages: head_dim 128 / 256 with up to 64 / 32 query rows per KV head.
// The SOLO instances serve grids of at most one CTA per SM (see PartialCfg).
#include "pkv_partial_instances.cuh"

namespace pkv {

#define PKV_U8_INSTANCES(X) \
  X(128, 1, 1, false) X(128, 2, 1, false) X(128, 2, 2, false) X(128, 2, 4, false) \
  X(256, 1, 1, false) X(256, 1, 2, false) X(256, 1, 4, false) \
  X(128, 1, 1, true) X(256, 1, 1, true)

PartialInfo partial_info_u8(int d, int nq, bool solo) {
  int nt, wq;
  tiles_for(d, nq, nt, wq);
#define X(D_, NT_, WQ_, SOLO_) \
  if (d == D_ && nt == NT_ && wq == WQ_ && solo == SOLO_) return info_of<8, D_, NT_, WQ_, SOLO_>();
  PKV_U8_INSTANCES(X)
#undef X
  return PartialInfo{false, 0, 0, 0, 0, 0};
}

cudaError_t launch_partial_u8(int d, int nq, bool solo, const PartialParams& p, const CUtensorMap& tk,
                              const CUtensorMap& tv, dim3 grid, cudaStream_t s, int dev) {
  int nt, wq;
  tiles_for(d, nq, nt, wq);
#define X(D_, NT_, WQ_, SOLO_) \
  if (d == D_ && nt == NT_ && wq == WQ_ && solo == SOLO_) \
    return launch_of<8, D_, NT_, WQ_, SOLO_>(p, tk, tv, grid, s, dev);
  PKV_U8_INSTANCES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace pkv
