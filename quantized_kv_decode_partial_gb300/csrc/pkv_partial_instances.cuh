// Explicit instantiations of the partial kernel for one page format. Included by
// pkv_partial_bf16.cu / pkv_partial_u4.cu / pkv_partial_u8.cu with PKV_BITS set.
#pragma once

#include <atomic>

#include "pkv_launch.h"
#include "pkv_partial.cuh"

namespace pkv {
namespace {

template <int BITS, int D, int DV, int NT, int WQ, bool SOLO, int CCQ = 0, bool BAL = false>
PartialInfo info_of() {
  using C = PartialCfg<BITS, D, DV, NT, WQ, SOLO, CCQ, BAL>;
  return PartialInfo{true, C::kThreads, C::kSmemBytes, C::kCh, C::kRB, C::kRBV, C::kElemBytes, C::kWP};
}

// Devices on which an instantiation's function attributes are set (bit per device < 64).
template <int BITS, int D, int DV, int NT, int WQ, bool SOLO, bool HOSTIN, int CCQ, bool PV, bool BAL, bool PC>
std::atomic<unsigned long long> g_configured{0};

template <int BITS, int D, int DV, int NT, int WQ, bool SOLO, bool HOSTIN, int CCQ = 0, bool PV = false,
          bool BAL = false, bool PC = false>
cudaError_t configure_once(int device) {
  using C = PartialCfg<BITS, D, DV, NT, WQ, SOLO, CCQ, BAL>;
  auto kern = pkv_partial_kernel<BITS, D, DV, NT, WQ, SOLO, HOSTIN, CCQ, PV, BAL, PC>;
  const unsigned long long bit = device >= 0 && device < 64 ? (1ull << device) : 0ull;
  if (bit &&
      (g_configured<BITS, D, DV, NT, WQ, SOLO, HOSTIN, CCQ, PV, BAL, PC>.load(std::memory_order_acquire) & bit))
    return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);  // clusters of up to 16
  if (e != cudaSuccess) return e;
  if (bit) g_configured<BITS, D, DV, NT, WQ, SOLO, HOSTIN, CCQ, PV, BAL, PC>.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

template <int BITS, int D, int DV, int NT, int WQ, bool SOLO, int CCQ = 0, bool PV = false, bool BAL = false,
          bool PC = false>
cudaError_t launch_of(const PartialParams& p, const CUtensorMap& tk, const CUtensorMap& tv, dim3 grid,
                      cudaStream_t stream, int device) {
  using C = PartialCfg<BITS, D, DV, NT, WQ, SOLO, CCQ, BAL>;
  auto kern = pkv_partial_kernel<BITS, D, DV, NT, WQ, SOLO, false, CCQ, PV, BAL, PC>;
  cudaError_t e;
  // Grids launch as programmatic dependents (below). For a grid of one CTA per SM whose
  // length, query and block tables are all host memory of a host-driven step, the
  // variant that reads them before the dependency wait runs.
  constexpr int kAllHost = kHostSeqLens | kHostQuery | kHostTables;
  if constexpr (SOLO) {
    if (p.host_inputs == kAllHost) {
      kern = pkv_partial_kernel<BITS, D, DV, NT, WQ, SOLO, true, CCQ, PV>;
      e = configure_once<BITS, D, DV, NT, WQ, SOLO, true, CCQ, PV>(device);
    } else {
      e = configure_once<BITS, D, DV, NT, WQ, SOLO, false, CCQ, PV>(device);
    }
  } else {
    e = configure_once<BITS, D, DV, NT, WQ, SOLO, false, CCQ, PV, BAL, PC>(device);
  }
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (SOLO || p.mode != kModeCluster || p.host_inputs != 0) {
    // Programmatic dependent launch: the CTAs may be placed on SMs while the previous
    // kernel on the stream finishes, and wait for it (griddepcontrol.wait) before they
    // touch global memory. The launch latency then hides behind that kernel's tail:
    // host-driven steps of the batches took 2-4 us less, graph-replayed steps the same.
    // (Under graph replay the cluster grid of two CTAs per SM of the windowed workload
    // lost 2% this way: early CTAs take the slots the previous grid frees unevenly. A
    // host-driven step, launched one by one, gains more from the hidden launch.)
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
  if (p.mode == kModeCluster) {  // the partitions of one (sequence, KV head) form a cluster
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = grid.x;
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 1;
    ++cfg.numAttrs;
  }
  return cudaLaunchKernelEx(&cfg, kern, p, tk, tv);
}

// CTAs of the balanced-schedule instantiation that one SM of `device` (the current
// device) holds at once; 0 on an error.
template <int BITS, int D, int DV, int NT, int WQ, bool PV = false>
int bal_ctas_per_sm(int device) {
  using C = PartialCfg<BITS, D, DV, NT, WQ, false, 0, true>;
  static std::atomic<int> known[64];  // per device < 64, 0 until first asked
  const bool cache = device >= 0 && device < 64;
  if (cache) {
    const int n = known[device].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  if (configure_once<BITS, D, DV, NT, WQ, false, false, 0, PV, true>(device) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, pkv_partial_kernel<BITS, D, DV, NT, WQ, false, false, 0, PV, true>, C::kThreads, C::kSmemBytes) !=
      cudaSuccess)
    return 0;
  if (cache && n > 0) known[device].store(n, std::memory_order_relaxed);
  return n;
}

// Instantiation for `nq` query rows per KV head: NT n-tiles of 8 rows per warp and
// WQ warps per query group (NT * WQ * 8 >= nq), or (0, 0) when unsupported. A warp
// holds NT * (dv/4 + dk/8) registers of accumulators and query fragments; NT is the
// largest of 1, 2, 4 that keeps them within the 96 of a 256-dim head at NT = 1.
inline void tiles_for(int dk, int dv, int nq, int& nt, int& wq) {
  nt = wq = 0;
  if (nq < 1) return;
  const int per_tile = dv / 4 + dk / 8;
  const int nt_max = 96 / per_tile >= 4 ? 4 : 96 / per_tile >= 2 ? 2 : 1;
  const int ntiles = (nq + 7) / 8;
  if (ntiles <= nt_max) {
    nt = ntiles <= 1 ? 1 : ntiles <= 2 ? 2 : 4;
    wq = 1;
  } else if (ntiles <= 2 * nt_max) {
    nt = nt_max;
    wq = 2;
  } else if (ntiles <= 4 * nt_max && (dk >= 128 || dv >= 128)) {
    nt = nt_max;
    wq = 4;
  } else if (ntiles <= 8 && nt_max == 1) {  // 256-dim (or 192/128) heads: a CTA of 8 warps
    nt = 1;
    wq = 8;
  }
}

}  // namespace
}  // namespace pkv
