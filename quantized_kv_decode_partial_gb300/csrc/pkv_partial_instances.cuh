// Explicit instantiations of the partial kernel for one page format. Included by
// pkv_partial_bf16.cu / pkv_partial_u4.cu / pkv_partial_u8.cu with PKV_BITS set.
#pragma once

#include "pkv_launch.h"
#include "pkv_partial.cuh"

namespace pkv {
namespace {

template <int BITS, int D, int NT>
PartialInfo info_of() {
  using C = PartialCfg<BITS, D, NT>;
  return PartialInfo{true, C::kThreads, C::kSmemBytes, C::kCh, C::kRB, C::kElemBytes};
}

template <int BITS, int D, int NT>
cudaError_t launch_of(const PartialParams& p, const CUtensorMap& tk, const CUtensorMap& tv, dim3 grid,
                      cudaStream_t stream) {
  using C = PartialCfg<BITS, D, NT>;
  auto kern = pkv_partial_kernel<BITS, D, NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(p, tk, tv);
  return cudaGetLastError();
}

}  // namespace
}  // namespace pkv
