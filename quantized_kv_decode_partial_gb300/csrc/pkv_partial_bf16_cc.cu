// bf16 pages with the CUDA-core contraction (pkv_partial_cc.cuh): head dims 64 / 128 / 256
// with up to 4 query rows per KV head, padded to 2 or 4. The SOLO instances serve grids of
// at most one CTA per SM (see PartialCfg).
#include "pkv_partial_instances.cuh"

namespace pkv {

#define PKV_BF16_CC_INSTANCES(X) \
  X(64, 2, false) X(64, 4, false) X(128, 2, false) X(128, 4, false) X(256, 2, false) X(256, 4, false) \
  X(64, 2, true) X(64, 4, true) X(128, 2, true) X(128, 4, true) X(256, 2, true) X(256, 4, true)

namespace {
int padded_rows(int nq) { return nq <= 2 ? 2 : nq <= 4 ? 4 : 0; }
}  // namespace

PartialInfo partial_info_bf16_cc(int dk, int dv, int nq, bool solo) {
  const int q = nq >= 1 && dk == dv ? padded_rows(nq) : 0;
#define X(D_, Q_, SOLO_) \
  if (dk == D_ && q == Q_ && solo == SOLO_) return info_of<16, D_, D_, 1, 1, SOLO_, Q_>();
  PKV_BF16_CC_INSTANCES(X)
#undef X
  return PartialInfo{};
}

cudaError_t launch_partial_bf16_cc(int dk, int dv, int nq, bool solo, const PartialParams& p, const CUtensorMap& tk,
                                   const CUtensorMap& tv, dim3 grid, cudaStream_t s, int dev) {
  const int q = nq >= 1 && dk == dv ? padded_rows(nq) : 0;
#define X(D_, Q_, SOLO_) \
  if (dk == D_ && q == Q_ && solo == SOLO_) return launch_of<16, D_, D_, 1, 1, SOLO_, Q_>(p, tk, tv, grid, s, dev);
  PKV_BF16_CC_INSTANCES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace pkv
