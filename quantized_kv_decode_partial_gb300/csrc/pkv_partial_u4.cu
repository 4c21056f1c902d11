// Affine 4-bit pages: head dims 128 / 256 and key/value head dims 256/128 and 128/256,
// each with up to 64 query rows per KV head.
// The SOLO instances serve grids of at most one CTA per SM (see PartialCfg).
#include "pkv_partial_instances.cuh"

namespace pkv {

#define PKV_U4_INSTANCES(X) \
  X(128, 128, 1, 1, false) X(128, 128, 2, 1, false) X(128, 128, 2, 2, false) X(128, 128, 2, 4, false) \
  X(256, 256, 1, 1, false) X(256, 256, 1, 2, false) X(256, 256, 1, 4, false) X(256, 256, 1, 8, false) \
  X(256, 128, 1, 1, false) X(256, 128, 1, 2, false) X(256, 128, 1, 4, false) X(256, 128, 1, 8, false) \
  X(128, 256, 1, 1, false) X(128, 256, 1, 2, false) X(128, 256, 1, 4, false) X(128, 256, 1, 8, false) \
  X(128, 128, 1, 1, true) X(256, 256, 1, 1, true)

// Up to 4 query rows per KV head with equal head dims: the paired-value-group form (PV in
// pkv_partial_kernel), one weight fragment per pair of 64-dim groups.
#define PKV_U4_PV_INSTANCES(X) X(128, false) X(256, false) X(128, true) X(256, true)

PartialInfo partial_info_u4(int dk, int dv, int nq, bool solo) {
  int nt, wq;
  tiles_for(dk, dv, nq, nt, wq);
  if (nq >= 1 && nq <= 4 && dk == dv) {
#define X(D_, SOLO_) \
    if (dk == D_ && solo == SOLO_) return info_of<4, D_, D_, 1, 1, SOLO_, 0>();  /* the layout of the unpaired form */
    PKV_U4_PV_INSTANCES(X)
#undef X
  }
#define X(DK_, DV_, NT_, WQ_, SOLO_) \
  if (dk == DK_ && dv == DV_ && nt == NT_ && wq == WQ_ && solo == SOLO_) \
    return info_of<4, DK_, DV_, NT_, WQ_, SOLO_>();
  PKV_U4_INSTANCES(X)
#undef X
  return PartialInfo{};
}

cudaError_t launch_partial_u4(int dk, int dv, int nq, bool solo, const PartialParams& p, const CUtensorMap& tk,
                              const CUtensorMap& tv, dim3 grid, cudaStream_t s, int dev) {
  int nt, wq;
  tiles_for(dk, dv, nq, nt, wq);
  if (nq >= 1 && nq <= 4 && dk == dv) {
#define X(D_, SOLO_) \
    if (dk == D_ && solo == SOLO_) return launch_of<4, D_, D_, 1, 1, SOLO_, 0, true>(p, tk, tv, grid, s, dev);
    PKV_U4_PV_INSTANCES(X)
#undef X
  }
#define X(DK_, DV_, NT_, WQ_, SOLO_) \
  if (dk == DK_ && dv == DV_ && nt == NT_ && wq == WQ_ && solo == SOLO_) \
    return launch_of<4, DK_, DV_, NT_, WQ_, SOLO_>(p, tk, tv, grid, s, dev);
  PKV_U4_INSTANCES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace pkv
