// Instantiations of the affine 8-bit shapes whose grids hold several CTAs per SM for pools of
// blocks smaller than a chunk (PC): the same kernels, copying each chunk block piece by
// block piece. Their layout is that of the instantiations without PC.
#include "pkv_partial_instances.cuh"

namespace pkv {

#define PKV_U8_PC_INSTANCES(X) \
  X(128, 128, 1, 1) X(128, 128, 2, 1) X(128, 128, 2, 2) X(128, 128, 2, 4) \
  X(256, 256, 1, 1) X(256, 256, 1, 2) X(256, 256, 1, 4) X(256, 256, 1, 8) \
  X(256, 128, 1, 1) X(256, 128, 1, 2) X(256, 128, 1, 4) X(256, 128, 1, 8) \
  X(128, 256, 1, 1) X(128, 256, 1, 2) X(128, 256, 1, 4) X(128, 256, 1, 8)

cudaError_t launch_partial_u8_pc(int dk, int dv, int nq, const PartialParams& p, const CUtensorMap& tk,
                                 const CUtensorMap& tv, dim3 grid, cudaStream_t s, int dev) {
  int nt, wq;
  tiles_for(dk, dv, nq, nt, wq);
#define X(DK_, DV_, NT_, WQ_) \
  if (dk == DK_ && dv == DV_ && nt == NT_ && wq == WQ_) \
    return launch_of<8, DK_, DV_, NT_, WQ_, false, 0, false, false, true>(p, tk, tv, grid, s, dev);
  PKV_U8_PC_INSTANCES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace pkv
