// C ABI of the paged decode attention library: argument checks, the partition
// plan, TMA descriptors and kernel launches. See include/pkv_decode.h.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "pkv_decode.h"
#include "pkv_launch.h"

namespace {

using pkv::PartialInfo;

thread_local char g_cuda_error[256] = "";

int cuda_fail(const char* what, cudaError_t e) {
  std::snprintf(g_cuda_error, sizeof(g_cuda_error), "%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
  return PKV_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// cc: the CUDA-core contraction (bf16 pages only), else the tensor-core one; bal: the
// balanced-schedule instantiation (tensor cores, several CTAs per SM).
PartialInfo partial_info(int bits, int dk, int dv, int nq, bool solo = false, bool cc = false, bool bal = false) {
  if (cc) return bits == 16 ? pkv::partial_info_bf16_cc(dk, dv, nq, solo) : PartialInfo{};
  if (bal) {
    if (solo) return PartialInfo{};
    if (bits == 16) return pkv::partial_info_bf16_bal(dk, dv, nq);
    if (bits == 4) return pkv::partial_info_u4_bal(dk, dv, nq);
    if (bits == 8) return pkv::partial_info_u8_bal(dk, dv, nq);
    return PartialInfo{};
  }
  if (bits == 16) return pkv::partial_info_bf16(dk, dv, nq, solo);
  if (bits == 4) return pkv::partial_info_u4(dk, dv, nq, solo);
  if (bits == 8) return pkv::partial_info_u8(dk, dv, nq, solo);
  return PartialInfo{};
}

// Value head dim of a layout (0 in the descriptor means the key head dim).
int v_dim(const pkv_pool_layout* L) { return L->v_head_dim > 0 ? L->v_head_dim : L->head_dim; }

// Balanced schedule: CTAs of instantiation `bi` one SM can hold, as far as its shared
// memory and threads tell (228 KB per SM, 1 KB of it reserved per CTA; 2048 threads).
// The grid launched holds at most this many per SM (the occupancy the registers allow
// may be lower), so the workspace sized from it suffices.
long long bal_ctas_per_sm_bound(const PartialInfo& bi) {
  const long long by_smem = (228ll * 1024) / (bi.smem_bytes + 1024);
  const long long by_threads = 2048 / bi.threads;
  return std::max(1ll, std::min(std::min(by_smem, by_threads), 32ll));
}

// Workspace of the balanced schedule with `runs` page groups: a state slot per (run,
// unit) pair that can occur, runs + units in all, each holding nq query rows: o
// [slot][nq][DV] floats, then (m, l) [slot][nq][2].
struct BalancedWorkspace {
  size_t o_bytes, bytes;
};
BalancedWorkspace balanced_workspace(long long runs, long long units, long long nq, int dv) {
  const size_t slots = static_cast<size_t>(runs + units) * static_cast<size_t>(nq);
  BalancedWorkspace w;
  w.o_bytes = (slots * dv * sizeof(float) + 255) / 256 * 256;
  w.bytes = w.o_bytes + slots * 2 * sizeof(float);
  return w;
}

// Stored bytes of one row of head dim `d`: bf16 values, or codes plus bf16 scale and bias.
long long stored_row_bytes(const pkv_pool_layout* L, int d) {
  return L->bits == 16 ? 2ll * d : static_cast<long long>(d) * L->bits / 8 + d / 64 * 4;
}

int chunk_rows_of(int bits) { return bits == 16 ? 16 : 32; }

int check_layout(const pkv_pool_layout* L) {
  if (!L) return PKV_ERR_NULL_POINTER;
  if (L->num_blocks <= 0 || L->num_kv_heads <= 0 || L->block_size <= 0) return PKV_ERR_BAD_LAYOUT;
  if (L->bits != 16 && L->bits != 4 && L->bits != 8) return PKV_ERR_BAD_LAYOUT;
  if (L->bits == 16) {
    if (L->head_dim != 64 && L->head_dim != 128 && L->head_dim != 192 && L->head_dim != 256) return PKV_ERR_BAD_LAYOUT;
    if (v_dim(L) != 64 && v_dim(L) != 128 && v_dim(L) != 256) return PKV_ERR_BAD_LAYOUT;
  } else {
    if (L->group_size != 64) return PKV_ERR_BAD_LAYOUT;
    if (L->head_dim != 128 && L->head_dim != 256) return PKV_ERR_BAD_LAYOUT;
    if (v_dim(L) != 128 && v_dim(L) != 256) return PKV_ERR_BAD_LAYOUT;
  }
  // Blocks of whole chunks, or smaller blocks of 8 or more rows that divide a chunk (a
  // chunk then spans several blocks and is copied block by block).
  const int ch = chunk_rows_of(L->bits);
  if (L->block_size % ch && (ch % L->block_size || L->block_size < 8)) return PKV_ERR_BAD_LAYOUT;
  const long long rows = static_cast<long long>(L->num_blocks) * L->num_kv_heads * L->block_size;
  if (rows >= (1ll << 31)) return PKV_ERR_BAD_LAYOUT;  // TMA row coordinates are int32
  if (L->num_kv_heads > 65535) return PKV_ERR_BAD_LAYOUT;
  return PKV_OK;
}

int check_params(const pkv_pool_layout* L, const pkv_decode_params* P) {
  if (!P) return PKV_ERR_NULL_POINTER;
  if (P->num_seqs <= 0 || P->num_seqs > 65535) return PKV_ERR_BAD_PARAMS;
  if (P->num_q_heads <= 0 || P->num_q_heads % L->num_kv_heads) return PKV_ERR_BAD_PARAMS;
  if (P->n_query < 1 || P->max_blocks_per_seq <= 0 || P->partition_tokens < 0 || P->window < 0)
    return PKV_ERR_BAD_PARAMS;
  if (static_cast<long long>(P->max_blocks_per_seq) * L->block_size >= (1ll << 31)) return PKV_ERR_BAD_PARAMS;
  if (P->contraction < PKV_CONTRACTION_AUTO || P->contraction > PKV_CONTRACTION_CUDA_CORE) return PKV_ERR_BAD_PARAMS;
  if (P->schedule < PKV_SCHEDULE_AUTO || P->schedule > PKV_SCHEDULE_BALANCED) return PKV_ERR_BAD_PARAMS;
  // output rows (and the merge grid) are counted in int
  if (static_cast<long long>(P->num_seqs) * P->num_q_heads * P->n_query >= (1ll << 31)) return PKV_ERR_BAD_PARAMS;
  const long long nq = static_cast<long long>(P->num_q_heads / L->num_kv_heads) * P->n_query;
  if (nq > 64) return PKV_ERR_UNSUPPORTED_SHAPE;
  const bool cc = P->contraction == PKV_CONTRACTION_CUDA_CORE;
  if (!partial_info(L->bits, L->head_dim, v_dim(L), static_cast<int>(nq), false, cc).exists)
    return PKV_ERR_UNSUPPORTED_SHAPE;
  return PKV_OK;
}

// Whether a call runs the CUDA-core contraction: when the caller asks for it, or, left to
// the library, for the shapes where it measured faster than the tensor cores.
bool use_cuda_cores(const pkv_pool_layout* L, const pkv_decode_params* P, long long ctas, int sm_count) {
  if (P->contraction == PKV_CONTRACTION_CUDA_CORE) return true;
  if (P->contraction == PKV_CONTRACTION_TENSOR) return false;
  (void)L;
  (void)ctas;
  (void)sm_count;
  return false;
}

long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

// Rows a step can read per sequence, counted from its partition base: the whole
// table, or with a window the span of W + N - 1 rows its queries see plus the
// alignment of the base to a chunk boundary below it.
long long window_rows(const pkv_decode_params* P, long long max_len) {
  if (P->window <= 0) return max_len;
  return std::min<long long>(max_len, static_cast<long long>(P->window) + P->n_query - 1 + (pkv::kWindowAlign - 1));
}

// `solo` (optional) receives whether the plan launches the variant for grids of at
// most one CTA per SM.
int plan_impl(const pkv_pool_layout* L, const pkv_decode_params* P, int sm_count, pkv_plan* out,
              bool* solo = nullptr) {
  const int ch = chunk_rows_of(L->bits);
  const long long max_len = static_cast<long long>(P->max_blocks_per_seq) * L->block_size;
  long long part;
  if (P->partition_tokens > 0) {
    // A caller's size past the table means one partition (INT_MAX included).
    part = round_up(std::min<long long>(P->partition_tokens, max_len), ch);
  } else {
    // Halve the partition until the grid covers the GPU about four times over (two
    // CTAs per SM) and no CTA gets more than 3 MB of K/V, never below 256 rows. Once
    // the grid fills a wave, stop before a CTA would get less than 512 KB: below that
    // its fixed costs (prologue, pipeline fill, epilogue) start to show (measured on the
    // windowed workload). The 3 MB cap keeps the last CTAs of a batch of mixed lengths
    // short: the 8-bit affine batch (8160-row partitions of 4.4 MB at four waves) went
    // from 717.2 to 697.9 us with 4080-row ones, while 2 MB CTAs (bf16 8 x 128K) were
    // 2% slower halved again.
    const long long slots = 2ll * (sm_count > 0 ? sm_count : 1);
    const long long target = 4 * slots;
    constexpr long long kMaxCtaBytes = 3ll << 20;
    const long long units = static_cast<long long>(P->num_seqs) * L->num_kv_heads;
    const long long kv_row = stored_row_bytes(L, L->head_dim) + stored_row_bytes(L, v_dim(L));  // K + V
    const long long floor_rows = 256;
    const long long rich_rows = std::max<long long>(floor_rows, (512ll << 10) / kv_row);
    const long long span = window_rows(P, max_len);
    part = round_up(span, ch);
    while (part > floor_rows) {
      const long long ctas = units * ((span + part - 1) / part);
      if (ctas >= target && part * kv_row <= kMaxCtaBytes) break;
      const long long half = std::max<long long>(floor_rows, round_up(part / 2, ch));
      if (half < rich_rows && ctas >= slots) break;
      part = half;
    }
    // With a window, every sequence longer than it reads the same span, so the
    // (sequence, KV head) units carry even work. When the grid above is at most two
    // waves (a short step, where the merge launch shows) and 2..16 partitions per unit
    // make a grid of one wave that fills at least three quarters of it, with CTAs of
    // at least 512 KB, take the most partitions that do (a wave of one CTA per SM
    // first, below): the partitions then merge inside their clusters, with no
    // workspace and no second launch.
    const long long nq_rows = static_cast<long long>(P->num_q_heads / L->num_kv_heads) * P->n_query;
    const PartialInfo two = partial_info(L->bits, L->head_dim, v_dim(L), static_cast<int>(nq_rows), false,
                                         P->contraction == PKV_CONTRACTION_CUDA_CORE);
    const long long default_ctas = units * ((span + part - 1) / part);
    if (P->window > 0 && default_ctas <= 2 * slots && two.exists && two.smem_bytes <= 114 * 1024) {
      // First a grid of one CTA per SM, where there is a variant for it: the most
      // partitions per unit (one included: no merge at all) that keep the grid within the
      // SMs and fill three quarters of them with CTAs of at least 1 MB. Its CTAs have
      // twice the warps, so the same rows stream from fewer, fuller SMs; on windowed
      // batches (4 to 16 sequences of 20000 rows, windows of 4096 and 8192 rows, HQ=32,
      // HK=8, N=4) that took 2-4% less time than two CTAs per SM, and host-driven steps
      // 6% less on 8 sequences. With CTAs of under 1 MB (2 sequences: 928 rows) the
      // per-CTA start and merge showed, and 496 short CTAs through the workspace were
      // 14% faster.
      const PartialInfo one = partial_info(L->bits, L->head_dim, v_dim(L), static_cast<int>(nq_rows), true,
                                           P->contraction == PKV_CONTRACTION_CUDA_CORE);
      const long long sms = sm_count > 0 ? sm_count : 1;
      bool placed = false;
      const bool whole_chunks = L->block_size >= two.chunk_rows;  // pools of smaller blocks have no such variant
      for (int k = pkv::kMaxClusterParts; one.exists && whole_chunks && k >= 1 && !placed; --k) {
        const long long pk = round_up((span + k - 1) / k, ch);
        const long long ctas = units * ((span + pk - 1) / pk);
        if (pk * kv_row >= (1ll << 20) && ctas <= sms && 4 * ctas >= 3 * sms) {
          part = pk;
          placed = true;
        }
      }
      for (int k = pkv::kMaxClusterParts; k >= 2 && !placed; --k) {
        const long long pk = round_up((span + k - 1) / k, ch);
        const long long ctas = units * ((span + pk - 1) / pk);
        if (pk >= rich_rows && ctas <= slots && 4 * ctas >= 3 * slots) {
          part = pk;
          placed = true;
        }
      }
    }
  }
  if (part >= max_len) part = round_up(max_len, ch);
  // Partitions per (sequence, KV head) in the grid and the workspace: all of the table,
  // or, with a window, enough to tile the rows from the aligned window base on.
  const int max_parts = ceil_div(window_rows(P, max_len), part);
  const long long nq = static_cast<long long>(P->num_q_heads / L->num_kv_heads) * P->n_query;
  // A grid of at most one CTA per SM takes the variant with more warps and stages
  // per CTA, where there is one for this shape.
  const long long sms = sm_count > 0 ? sm_count : 1;
  const long long ctas = static_cast<long long>(P->num_seqs) * L->num_kv_heads * max_parts;
  // Blocks smaller than the chunk the grids of several CTAs per SM stage: those grids'
  // instantiations for such pools (no CTA-alone variant, no balanced schedule, no
  // CUDA-core contraction).
  const bool pieces =
      L->block_size < partial_info(L->bits, L->head_dim, v_dim(L), static_cast<int>(nq), false, false).chunk_rows;
  if (pieces && P->contraction == PKV_CONTRACTION_CUDA_CORE) return PKV_ERR_UNSUPPORTED_SHAPE;
  const bool cc = use_cuda_cores(L, P, ctas, sm_count);
  const bool use_solo = !pieces && ctas <= sms &&
                        partial_info(L->bits, L->head_dim, v_dim(L), static_cast<int>(nq), true, cc).exists;
  if (solo) *solo = use_solo;
  const PartialInfo info = partial_info(L->bits, L->head_dim, v_dim(L), static_cast<int>(nq), use_solo, cc);
  out->contraction = cc ? PKV_CONTRACTION_CUDA_CORE : PKV_CONTRACTION_TENSOR;
  out->partition_tokens = static_cast<int32_t>(part);
  out->max_partitions = max_parts;
  out->chunk_rows = info.chunk_rows;
  out->sm_count = sm_count;
  out->threads_per_cta = info.threads;
  out->smem_bytes = info.smem_bytes;
  out->workspace_bytes = 0;
  // Merge inside a thread-block cluster when a (sequence, KV head) has 2..16
  // partitions and the grid is at most one wave: the CTAs of a cluster are then
  // resident together anyway, and the merge needs no workspace and no second launch.
  // A cluster of up to 16 CTAs fits 8 SMs at two CTAs per SM; at one CTA per SM it
  // takes 16 SMs of one GPC (GB300 GPCs hold more), which the one-CTA-per-SM variant
  // relies on, while the four-warp variant with large stages keeps to 8.
  const bool two_per_sm = !use_solo && info.smem_bytes <= 114 * 1024;
  out->merge_in_cluster = max_parts >= 2 && max_parts <= (two_per_sm || use_solo ? 16 : 8) &&
                          ctas <= sms * (two_per_sm ? 2 : 1);
  if (max_parts > 1 && !out->merge_in_cluster) {
    const size_t slots = static_cast<size_t>(P->num_seqs) * P->num_q_heads * P->n_query * max_parts;
    const size_t o_bytes = (slots * v_dim(L) * sizeof(float) + 255) / 256 * 256;
    out->workspace_bytes = o_bytes + slots * 2 * sizeof(float);
  }
  // Balanced schedule: with the library's choice of split, for 4-bit pages where the
  // partitions would go through the workspace (or wherever the caller asks for it), and
  // where there is an instantiation. The 4-bit kernels are bound by their arithmetic,
  // which runs at the same rate on every SM, so equal runs end together and the tail of
  // the partition waves goes away (4-bit batch layer 430.3 -> 392.7 us). The 8-bit and
  // bf16 kernels stream at the memory's pace, which differs from SM to SM by up to a
  // quarter; equal runs then end apart, while partition waves let the hardware hand the
  // faster SMs more CTAs (balanced: 8-bit layer 718.8 -> 748.1 us, bf16 8 x 128K rows
  // 609.6 -> 642.6 us). The chunk list must index in 32 bits: the longest unit reads at
  // most the table, or with a window W + N - 1 rows plus the alignment of its first chunk.
  out->balanced = 0;
  if (P->partition_tokens == 0 && P->schedule != PKV_SCHEDULE_PARTITIONS && !cc && !pieces &&
      P->num_seqs <= pkv::kMaxBalancedSeqs &&
      (P->schedule == PKV_SCHEDULE_BALANCED || (L->bits == 4 && max_parts > 1 && !out->merge_in_cluster))) {
    const PartialInfo bi = partial_info(L->bits, L->head_dim, v_dim(L), static_cast<int>(nq), false, false, true);
    const long long unit_chunks = (window_rows(P, max_len) + bi.chunk_rows - 1) / std::max(bi.chunk_rows, 1);
    const long long units = static_cast<long long>(P->num_seqs) * L->num_kv_heads;
    if (bi.exists && units * unit_chunks < (1ll << 31)) {
      const long long runs = sms * bal_ctas_per_sm_bound(bi) * bi.page_groups;
      out->balanced = 1;
      out->workspace_bytes = std::max(out->workspace_bytes, balanced_workspace(runs, units, nq, v_dim(L)).bytes);
    }
  }
  return PKV_OK;
}

constexpr int kMaxDevices = 256;
std::atomic<int> g_sm_count[kMaxDevices];  // 0 until first read

int device_sm_count(int* sms, int* device = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (device) *device = dev;
  if (dev >= 0 && dev < kMaxDevices) {
    const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
    if (cached > 0) {
      *sms = cached;
      return PKV_OK;
    }
  }
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail("cudaDeviceGetAttribute", e);
  if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(*sms, std::memory_order_relaxed);
  return PKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 3-D view of one pool plane: rows = num_blocks*HK*BS of `row_elems` elements, each
// row seen as row_bytes / box_row_bytes segments of `box_row_bytes` bytes, with the
// segment index outermost (dims: element in segment, row, segment; strides: the row
// pitch, then the segment width). One box takes `box_rows` rows of every segment and
// lands segment-major ([segment][row][box_row_bytes], swizzled to match), so a chunk
// of a plane is one TMA copy whatever its width.
// The box is box_rows rows of every segment of a row (one copy per chunk), or with
// one_segment, of a single segment (blocks smaller than a chunk: one copy per block piece
// and segment).
int encode_pool_tensor_map(CUtensorMap* map, const void* base, int elem_bytes, long long row_elems, long long rows,
                           int box_row_bytes, int box_rows, bool one_segment) {
  auto encode = tensor_map_encoder();
  if (!encode) {
    std::snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled entry point unavailable");
    return PKV_ERR_CUDA;
  }
  const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const long long row_bytes = row_elems * elem_bytes;
  const long long segments = row_bytes / box_row_bytes;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(box_row_bytes / elem_bytes), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(segments)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(box_row_bytes)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_row_bytes / elem_bytes), static_cast<cuuint32_t>(box_rows),
                       static_cast<cuuint32_t>(one_segment ? 1 : segments)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = box_row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = encode(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

// Descriptors of recently used pool planes: a decode loop calls with the same
// pools every step, so the encoding is done once per plane.
struct TensorMapEntry {
  const void* base;
  long long row_elems, rows;
  int elem_bytes, box_row_bytes, chunk_rows;
  bool one_segment;
  CUtensorMap map;
};
constexpr int kTensorMapCacheSize = 16;
std::mutex g_tmap_mutex;
TensorMapEntry g_tmap_cache[kTensorMapCacheSize];
int g_tmap_next = 0;

int pool_tensor_map(CUtensorMap* map, const void* base, int elem_bytes, long long row_elems, long long rows,
                    int box_row_bytes, int box_rows, bool one_segment) {
  {
    std::lock_guard<std::mutex> lock(g_tmap_mutex);
    for (const TensorMapEntry& e : g_tmap_cache) {
      if (e.base == base && e.row_elems == row_elems && e.rows == rows && e.elem_bytes == elem_bytes &&
          e.box_row_bytes == box_row_bytes && e.chunk_rows == box_rows && e.one_segment == one_segment) {
        *map = e.map;
        return PKV_OK;
      }
    }
  }
  int rc = encode_pool_tensor_map(map, base, elem_bytes, row_elems, rows, box_row_bytes, box_rows, one_segment);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_tmap_mutex);
  TensorMapEntry& e = g_tmap_cache[g_tmap_next];
  g_tmap_next = (g_tmap_next + 1) % kTensorMapCacheSize;
  e = TensorMapEntry{base, row_elems, rows, elem_bytes, box_row_bytes, box_rows, one_segment, *map};
  return PKV_OK;
}

}  // namespace

namespace {

// The device-space address of page-locked host memory at `p`, or nullptr when it is
// not mapped for the current device (pageable memory, say).
void* mapped_host_address(const void* p) {
  if (!p) return nullptr;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  return a.devicePointer;
}

}  // namespace

extern "C" {

int pkv_make_plan(const pkv_pool_layout* layout, const pkv_decode_params* params, int32_t sm_count,
                  pkv_plan* plan) {
  if (!plan) return PKV_ERR_NULL_POINTER;
  int rc = check_layout(layout);
  if (rc) return rc;
  rc = check_params(layout, params);
  if (rc) return rc;
  if (sm_count <= 0) return PKV_ERR_BAD_PARAMS;
  return plan_impl(layout, params, sm_count, plan);
}

int pkv_plan_for_current_device(const pkv_pool_layout* layout, const pkv_decode_params* params, pkv_plan* plan) {
  if (!plan) return PKV_ERR_NULL_POINTER;
  int rc = check_layout(layout);
  if (rc) return rc;
  rc = check_params(layout, params);
  if (rc) return rc;
  int sms = 0;
  rc = device_sm_count(&sms);
  if (rc) return rc;
  return plan_impl(layout, params, sms, plan);
}

}  // extern "C"

namespace {

pkv::AppendTarget append_target(bool quant, void* k_pool, void* v_pool, void* k_scales, void* k_biases,
                                void* v_scales, void* v_biases) {
  pkv::AppendTarget t{};
  t.k_pool_bf16 = quant ? nullptr : static_cast<__nv_bfloat16*>(k_pool);
  t.v_pool_bf16 = quant ? nullptr : static_cast<__nv_bfloat16*>(v_pool);
  t.k_pool_words = quant ? static_cast<uint32_t*>(k_pool) : nullptr;
  t.v_pool_words = quant ? static_cast<uint32_t*>(v_pool) : nullptr;
  t.k_scales = static_cast<__nv_bfloat16*>(k_scales);
  t.k_biases = static_cast<__nv_bfloat16*>(k_biases);
  t.v_scales = static_cast<__nv_bfloat16*>(v_scales);
  t.v_biases = static_cast<__nv_bfloat16*>(v_biases);
  return t;
}

constexpr int kPassPartial = 1;
constexpr int kPassMerge = 2;

// Bound of one main-loop pipeline wait in the partial kernels launched from now on
// (pkv_set_wait_limit_ns).
std::atomic<unsigned long long> g_wait_limit_ns{pkv::kWaitLimitNs};

// Everything one decode call launches, resolved from its arguments: the kernels'
// parameter blocks, the TMA descriptors of the pools and the launch shapes.
struct PreparedDecode {
  pkv::PartialParams p;
  pkv::MergeParams m;
  CUtensorMap tk, tv;
  dim3 grid;
  int bits, dk, dv, nq, device;
  bool solo, cc, bal, pc, partial, merge;
};

// Checks the arguments of a decode call (the passes in `passes`) and prepares its
// launches; no CUDA work is enqueued.
int prepare_decode(const pkv_pool_layout* layout, const pkv_decode_params* params, const void* q,
                   const void* k_pool, const void* v_pool, const void* k_scales, const void* k_biases,
                   const void* v_scales, const void* v_biases, const int32_t* block_tables,
                   const int32_t* seq_lens, float scale, void* out, void* workspace, size_t workspace_bytes,
                   int32_t* error_flag, int passes, const void* k_new, const void* v_new, PreparedDecode* pd) {
  int rc = check_layout(layout);
  if (rc) return rc;
  rc = check_params(layout, params);
  if (rc) return rc;
  const bool quant = layout->bits != 16;
  const bool partial = passes & kPassPartial;
  if (!seq_lens || !out) return PKV_ERR_NULL_POINTER;
  if (partial && (!q || !k_pool || !v_pool || !block_tables)) return PKV_ERR_NULL_POINTER;
  if (partial && quant && (!k_scales || !k_biases || !v_scales || !v_biases)) return PKV_ERR_NULL_POINTER;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(error_flag, 4) || !aligned(workspace, 16))
    return PKV_ERR_MISALIGNED;
  if (quant && (!aligned(k_scales, 16) || !aligned(k_biases, 16) || !aligned(v_scales, 16) || !aligned(v_biases, 16)))
    return PKV_ERR_MISALIGNED;
  if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_NULL_POINTER;
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return PKV_ERR_MISALIGNED;

  int sms = 0, dev = 0;
  rc = device_sm_count(&sms, &dev);
  if (rc) return rc;
  pkv_plan plan;
  bool solo = false;
  rc = plan_impl(layout, params, sms, &plan, &solo);
  if (rc) return rc;
  const bool bal = plan.balanced && k_new == nullptr;  // the fused call runs partitions
  const int mode = bal                       ? pkv::kModeBalanced
                   : plan.max_partitions == 1 ? pkv::kModeSingle
                   : plan.merge_in_cluster   ? pkv::kModeCluster
                                             : pkv::kModeWorkspace;
  const bool ws_mode = mode == pkv::kModeWorkspace || mode == pkv::kModeBalanced;
  if (ws_mode && (!workspace || workspace_bytes < plan.workspace_bytes)) return PKV_ERR_WORKSPACE_TOO_SMALL;
  if (bal) solo = false;

  const int D = layout->head_dim, DV = v_dim(layout), HK = layout->num_kv_heads;
  const int nq = (params->num_q_heads / HK) * params->n_query;
  const bool cc = plan.contraction == PKV_CONTRACTION_CUDA_CORE;
  const PartialInfo info = partial_info(layout->bits, D, DV, nq, solo, cc, bal);
  // Blocks smaller than the instantiation's chunk: a chunk spans 2^piece_log2 blocks. The
  // fused call writes a chunk's new rows into one block, so it needs whole chunks.
  int piece_log2 = 0;
  while ((info.chunk_rows >> piece_log2) > layout->block_size) ++piece_log2;
  const int piece_rows = info.chunk_rows >> piece_log2;
  if (piece_log2 > 0 && k_new) return PKV_ERR_UNSUPPORTED_SHAPE;
  // Balanced schedule: one wave of CTAs, as many per SM as the instantiation's occupancy
  // allows (within the bound the plan sized the workspace for).
  int bal_ctas = 0;
  if (bal) {
    const int occ = layout->bits == 16  ? pkv::partial_bal_ctas_per_sm_bf16(D, DV, nq, dev)
                    : layout->bits == 4 ? pkv::partial_bal_ctas_per_sm_u4(D, DV, nq, dev)
                                        : pkv::partial_bal_ctas_per_sm_u8(D, DV, nq, dev);
    if (occ <= 0) return cuda_fail("occupancy of the balanced partial kernel", cudaGetLastError());
    bal_ctas = sms * static_cast<int>(std::min<long long>(occ, bal_ctas_per_sm_bound(info)));
  }
  const long long rows = static_cast<long long>(layout->num_blocks) * HK * layout->block_size;
  const int elem = info.tensor_elem_bytes;
  const long long row_elems_k = quant ? static_cast<long long>(D) * layout->bits / 8 : D;
  const long long row_elems_v = quant ? static_cast<long long>(DV) * layout->bits / 8 : DV;

  *pd = PreparedDecode{};
  if (partial) {
    rc = pool_tensor_map(&pd->tk, k_pool, elem, row_elems_k, rows, info.box_row_bytes, piece_rows, piece_log2 > 0);
    if (rc) return rc;
    rc = pool_tensor_map(&pd->tv, v_pool, elem, row_elems_v, rows, info.box_row_bytes_v, piece_rows, piece_log2 > 0);
    if (rc) return rc;
  }

  pkv::PartialParams& p = pd->p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.k_scales = static_cast<const __nv_bfloat16*>(k_scales);
  p.k_biases = static_cast<const __nv_bfloat16*>(k_biases);
  p.v_scales = static_cast<const __nv_bfloat16*>(v_scales);
  p.v_biases = static_cast<const __nv_bfloat16*>(v_biases);
  p.out = static_cast<__nv_bfloat16*>(out);
  const size_t slots = static_cast<size_t>(params->num_seqs) * params->num_q_heads * params->n_query * plan.max_partitions;
  const size_t o_bytes = bal ? balanced_workspace(static_cast<long long>(bal_ctas) * info.page_groups,
                                                  static_cast<long long>(params->num_seqs) * HK, nq, DV)
                                   .o_bytes
                             : (slots * DV * sizeof(float) + 255) / 256 * 256;  // as plan_impl sizes it
  p.ws_o = ws_mode ? static_cast<float*>(workspace) : nullptr;
  p.ws_ml = ws_mode ? reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes) : nullptr;
  p.mode = mode;
  p.piece_log2 = piece_log2;
  p.num_seqs = params->num_seqs;
  p.window = params->window;
  p.host_inputs = 0;
  p.error_flag = error_flag;
  p.num_blocks = layout->num_blocks;
  p.num_kv_heads = HK;
  p.block_size = layout->block_size;
  p.max_blocks = params->max_blocks_per_seq;
  p.num_q_heads = params->num_q_heads;
  p.n_query = params->n_query;
  p.nq = nq;
  p.partition_tokens = plan.partition_tokens;
  p.max_partitions = plan.max_partitions;
  p.score_scale = scale * 1.4426950408889634f;  // log2(e): scores run in base 2
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  if (k_new) {  // the pools are the caller's writable planes (the fused entry takes them non-const)
    p.k_new = static_cast<const __nv_bfloat16*>(k_new);
    p.v_new = static_cast<const __nv_bfloat16*>(v_new);
    p.app = append_target(quant, const_cast<void*>(k_pool), const_cast<void*>(v_pool), const_cast<void*>(k_scales),
                          const_cast<void*>(k_biases), const_cast<void*>(v_scales), const_cast<void*>(v_biases));
  }

  pd->grid = bal ? dim3(bal_ctas) : dim3(plan.max_partitions, HK, params->num_seqs);
  pd->bits = layout->bits;
  pd->dk = D;
  pd->dv = DV;
  pd->nq = nq;
  pd->device = dev;
  pd->solo = solo;
  pd->cc = cc;
  pd->bal = bal;
  pd->pc = piece_log2 > 0;
  pd->partial = partial;
  pd->merge = (passes & kPassMerge) && ws_mode;
  if (pd->merge) {
    pkv::MergeParams& m = pd->m;
    m.ws_o = p.ws_o;
    m.ws_ml = p.ws_ml;
    m.seq_lens = seq_lens;
    m.out = p.out;
    m.error_flag = error_flag;
    m.rows_per_seq = params->num_q_heads * params->n_query;
    m.n_query = params->n_query;
    m.head_dim = DV;
    m.max_len = params->max_blocks_per_seq * layout->block_size;
    m.partition_tokens = plan.partition_tokens;
    m.max_partitions = plan.max_partitions;
    m.window = params->window;
    m.rows = params->num_seqs * params->num_q_heads * params->n_query;
    m.groups = pkv::merge_groups(DV, plan.max_partitions);
    if (bal) {
      // a unit's runs: about its share of the page groups plus one; two groups per row
      // take up to 8 in the first round of loads
      m.bal_runs = bal_ctas * info.page_groups;
      m.num_seqs = params->num_seqs;
      m.num_kv_heads = HK;
      m.nq = nq;
      m.chunk_rows = info.chunk_rows;
      m.groups = pkv::merge_groups(DV, 8);
    }
  }
  return PKV_OK;
}

// Enqueues the launches of a prepared decode call on `stream` (the device current
// when it was prepared must be current).
int launch_prepared(const PreparedDecode& pd, cudaStream_t st) {
  (void)cudaGetLastError();  // start from a clean error state
  cudaError_t e = cudaSuccess;
  if (pd.partial) {
    if (pd.pc)
      e = pd.bits == 16  ? pkv::launch_partial_bf16_pc(pd.dk, pd.dv, pd.nq, pd.p, pd.tk, pd.tv, pd.grid, st, pd.device)
          : pd.bits == 4 ? pkv::launch_partial_u4_pc(pd.dk, pd.dv, pd.nq, pd.p, pd.tk, pd.tv, pd.grid, st, pd.device)
                         : pkv::launch_partial_u8_pc(pd.dk, pd.dv, pd.nq, pd.p, pd.tk, pd.tv, pd.grid, st, pd.device);
    else if (pd.bal)
      e = pd.bits == 16  ? pkv::launch_partial_bf16_bal(pd.dk, pd.dv, pd.nq, pd.p, pd.tk, pd.tv, pd.grid, st, pd.device)
          : pd.bits == 4 ? pkv::launch_partial_u4_bal(pd.dk, pd.dv, pd.nq, pd.p, pd.tk, pd.tv, pd.grid, st, pd.device)
                         : pkv::launch_partial_u8_bal(pd.dk, pd.dv, pd.nq, pd.p, pd.tk, pd.tv, pd.grid, st, pd.device);
    else if (pd.cc)
      e = pkv::launch_partial_bf16_cc(pd.dk, pd.dv, pd.nq, pd.solo, pd.p, pd.tk, pd.tv, pd.grid, st, pd.device);
    else if (pd.bits == 16)
      e = pkv::launch_partial_bf16(pd.dk, pd.dv, pd.nq, pd.solo, pd.p, pd.tk, pd.tv, pd.grid, st, pd.device);
    else if (pd.bits == 4)
      e = pkv::launch_partial_u4(pd.dk, pd.dv, pd.nq, pd.solo, pd.p, pd.tk, pd.tv, pd.grid, st, pd.device);
    else
      e = pkv::launch_partial_u8(pd.dk, pd.dv, pd.nq, pd.solo, pd.p, pd.tk, pd.tv, pd.grid, st, pd.device);
    if (e != cudaSuccess) return cuda_fail("partial kernel launch", e);
  }
  if (pd.merge) {
    e = pkv::launch_merge(pd.m, st);
    if (e != cudaSuccess) return cuda_fail("merge kernel launch", e);
  }
  return PKV_OK;
}

int enqueue_decode(const pkv_pool_layout* layout, const pkv_decode_params* params, const void* q,
                   const void* k_pool, const void* v_pool, const void* k_scales, const void* k_biases,
                   const void* v_scales, const void* v_biases, const int32_t* block_tables,
                   const int32_t* seq_lens, float scale, void* out, void* workspace, size_t workspace_bytes,
                   int32_t* error_flag, void* stream, int passes, const void* k_new = nullptr,
                   const void* v_new = nullptr) {
  PreparedDecode pd;
  int rc = prepare_decode(layout, params, q, k_pool, v_pool, k_scales, k_biases, v_scales, v_biases, block_tables,
                          seq_lens, scale, out, workspace, workspace_bytes, error_flag, passes, k_new, v_new, &pd);
  if (rc) return rc;
  return launch_prepared(pd, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int pkv_paged_decode_attention(const pkv_pool_layout* layout, const pkv_decode_params* params, const void* q,
                               const void* k_pool, const void* v_pool, const void* k_scales,
                               const void* k_biases, const void* v_scales, const void* v_biases,
                               const int32_t* block_tables, const int32_t* seq_lens, float scale, void* out,
                               void* workspace, size_t workspace_bytes, int32_t* error_flag, void* stream) {
  return enqueue_decode(layout, params, q, k_pool, v_pool, k_scales, k_biases, v_scales, v_biases, block_tables,
                        seq_lens, scale, out, workspace, workspace_bytes, error_flag, stream,
                        kPassPartial | kPassMerge);
}

int pkv_paged_decode_partial(const pkv_pool_layout* layout, const pkv_decode_params* params, const void* q,
                             const void* k_pool, const void* v_pool, const void* k_scales, const void* k_biases,
                             const void* v_scales, const void* v_biases, const int32_t* block_tables,
                             const int32_t* seq_lens, float scale, void* out, void* workspace,
                             size_t workspace_bytes, int32_t* error_flag, void* stream) {
  return enqueue_decode(layout, params, q, k_pool, v_pool, k_scales, k_biases, v_scales, v_biases, block_tables,
                        seq_lens, scale, out, workspace, workspace_bytes, error_flag, stream, kPassPartial);
}

int pkv_merge_partitions(const pkv_pool_layout* layout, const pkv_decode_params* params, const int32_t* seq_lens,
                         const void* workspace, size_t workspace_bytes, void* out, int32_t* error_flag,
                         void* stream) {
  return enqueue_decode(layout, params, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                        seq_lens, 0.f, out, const_cast<void*>(workspace), workspace_bytes, error_flag, stream,
                        kPassMerge);
}

}  // extern "C"

struct pkv_step {
  PreparedDecode pd;
  const void* in_host;
  void* in_dev;
  size_t in_bytes;
  void* out_host;
  const void* out_dev;
  size_t out_bytes;
  cudaStream_t stream;
  bool copy_in;   // the inputs go through the copy engine (host memory the device cannot address)
  bool copy_out;  // likewise the output
};

namespace {

// Prepares a host-driven step into *s. Inputs inside [in_dev, in_dev + in_bytes) of
// mapped page-locked host memory are read by the kernels where they are; a mapped
// out_host is written by the kernels beside `out`; anything else is copied.
int build_step(const pkv_pool_layout* layout, const pkv_decode_params* params, const void* in_host, void* in_dev,
               size_t in_bytes, void* out_host, const void* q, const void* k_new, const void* v_new, void* k_pool,
               void* v_pool, void* k_scales, void* k_biases, void* v_scales, void* v_biases,
               const int32_t* block_tables, const int32_t* seq_lens, float scale, void* out, void* workspace,
               size_t workspace_bytes, int32_t* error_flag, void* stream, pkv_step* s) {
  if (in_bytes > 0 && (!in_host || !in_dev)) return PKV_ERR_NULL_POINTER;
  int rc = prepare_decode(layout, params, q, k_pool, v_pool, k_scales, k_biases, v_scales, v_biases, block_tables,
                          seq_lens, scale, out, workspace, workspace_bytes, error_flag, kPassPartial | kPassMerge,
                          k_new, v_new, &s->pd);
  if (rc) return rc;
  s->in_host = in_host;
  s->in_dev = in_dev;
  s->in_bytes = in_bytes;
  s->out_host = out_host;
  s->out_dev = out;
  s->out_bytes = static_cast<size_t>(params->num_seqs) * params->num_q_heads * params->n_query * v_dim(layout) * 2;
  s->stream = static_cast<cudaStream_t>(stream);
  const void* in_map =
      in_bytes > 0 && aligned(in_host, 16) && aligned(in_dev, 16) ? mapped_host_address(in_host) : nullptr;
  s->copy_in = in_bytes > 0 && !in_map;
  if (in_map) {
    const char* lo = static_cast<const char*>(in_dev);
    auto in_place = [&](const void* ptr) -> const void* {
      const char* c = static_cast<const char*>(ptr);
      return c && c >= lo && c < lo + in_bytes ? static_cast<const char*>(in_map) + (c - lo) : ptr;
    };
    pkv::PartialParams& p = s->pd.p;
    const void* q0 = p.q;
    const void* t0 = p.block_tables;
    const void* l0 = p.seq_lens;
    p.q = static_cast<const __nv_bfloat16*>(in_place(p.q));
    p.block_tables = static_cast<const int32_t*>(in_place(p.block_tables));
    p.seq_lens = static_cast<const int32_t*>(in_place(p.seq_lens));
    p.host_inputs = (p.seq_lens != l0 ? pkv::kHostSeqLens : 0) | (p.q != q0 ? pkv::kHostQuery : 0) |
                    (p.block_tables != t0 ? pkv::kHostTables : 0);
    p.k_new = static_cast<const __nv_bfloat16*>(in_place(p.k_new));
    p.v_new = static_cast<const __nv_bfloat16*>(in_place(p.v_new));
    s->pd.m.seq_lens = static_cast<const int32_t*>(in_place(s->pd.m.seq_lens));
  }
  void* out_map = out_host && aligned(out_host, 16) ? mapped_host_address(out_host) : nullptr;
  s->copy_out = out_host && !out_map;
  if (out_map) {
    s->pd.p.out_mirror = static_cast<__nv_bfloat16*>(out_map);
    s->pd.m.out_mirror = static_cast<__nv_bfloat16*>(out_map);
  }
  return PKV_OK;
}

int run_step(const pkv_step& s) {
  (void)cudaGetLastError();
  if (s.copy_in) {
    cudaError_t e = cudaMemcpyAsync(s.in_dev, s.in_host, s.in_bytes, cudaMemcpyHostToDevice, s.stream);
    if (e != cudaSuccess) return cuda_fail("input copy", e);
  }
  int rc = launch_prepared(s.pd, s.stream);
  if (rc) return rc;
  if (s.copy_out) {
    cudaError_t e = cudaMemcpyAsync(s.out_host, s.out_dev, s.out_bytes, cudaMemcpyDeviceToHost, s.stream);
    if (e != cudaSuccess) return cuda_fail("output copy", e);
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_paged_decode_attention_host(const pkv_pool_layout* layout, const pkv_decode_params* params,
                                    const void* in_host, void* in_dev, size_t in_bytes, void* out_host,
                                    const void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                    void* k_scales, void* k_biases, void* v_scales, void* v_biases,
                                    const int32_t* block_tables, const int32_t* seq_lens, float scale, void* out,
                                    void* workspace, size_t workspace_bytes, int32_t* error_flag, void* stream) {
  pkv_step s{};
  int rc = build_step(layout, params, in_host, in_dev, in_bytes, out_host, q, k_new, v_new, k_pool, v_pool, k_scales,
                      k_biases, v_scales, v_biases, block_tables, seq_lens, scale, out, workspace, workspace_bytes,
                      error_flag, stream, &s);
  if (rc) return rc;
  return run_step(s);
}

int pkv_step_create(const pkv_pool_layout* layout, const pkv_decode_params* params, const void* in_host, void* in_dev,
                    size_t in_bytes, void* out_host, const void* q, const void* k_new, const void* v_new,
                    void* k_pool, void* v_pool, void* k_scales, void* k_biases, void* v_scales, void* v_biases,
                    const int32_t* block_tables, const int32_t* seq_lens, float scale, void* out, void* workspace,
                    size_t workspace_bytes, int32_t* error_flag, void* stream, pkv_step** step) {
  if (!step) return PKV_ERR_NULL_POINTER;
  *step = nullptr;
  pkv_step* s = new (std::nothrow) pkv_step{};
  if (!s) return PKV_ERR_BAD_PARAMS;
  int rc = build_step(layout, params, in_host, in_dev, in_bytes, out_host, q, k_new, v_new, k_pool, v_pool, k_scales,
                      k_biases, v_scales, v_biases, block_tables, seq_lens, scale, out, workspace, workspace_bytes,
                      error_flag, stream, s);
  if (rc) {
    delete s;
    return rc;
  }
  *step = s;
  return PKV_OK;
}

int pkv_step_run(pkv_step* step) {
  if (!step) return PKV_ERR_NULL_POINTER;
  return run_step(*step);
}

void pkv_step_destroy(pkv_step* step) { delete step; }

int pkv_paged_decode_append_attention(const pkv_pool_layout* layout, const pkv_decode_params* params,
                                      const void* q, const void* k_new, const void* v_new, void* k_pool,
                                      void* v_pool, void* k_scales, void* k_biases, void* v_scales, void* v_biases,
                                      const int32_t* block_tables, const int32_t* seq_lens, float scale, void* out,
                                      void* workspace, size_t workspace_bytes, int32_t* error_flag, void* stream) {
  if (!k_new || !v_new) return PKV_ERR_NULL_POINTER;
  return enqueue_decode(layout, params, q, k_pool, v_pool, k_scales, k_biases, v_scales, v_biases, block_tables,
                        seq_lens, scale, out, workspace, workspace_bytes, error_flag, stream,
                        kPassPartial | kPassMerge, k_new, v_new);
}

int pkv_paged_append(const pkv_pool_layout* layout, int32_t num_seqs, int32_t max_blocks_per_seq, int32_t n_new,
                     const void* k_new, const void* v_new, const int32_t* block_tables, const int32_t* seq_lens,
                     void* k_pool, void* v_pool, void* k_scales, void* k_biases, void* v_scales, void* v_biases,
                     int32_t* error_flag, void* stream) {
  int rc = check_layout(layout);
  if (rc) return rc;
  if (!pkv::append_supported(layout->bits, layout->head_dim, v_dim(layout))) return PKV_ERR_BAD_LAYOUT;
  if (num_seqs <= 0 || num_seqs > 65535 || max_blocks_per_seq <= 0 || n_new < 0 || n_new > 65535)
    return PKV_ERR_BAD_PARAMS;
  if (static_cast<long long>(max_blocks_per_seq) * layout->block_size >= (1ll << 31)) return PKV_ERR_BAD_PARAMS;
  const bool quant = layout->bits != 16;
  if (!k_new || !v_new || !block_tables || !seq_lens || !k_pool || !v_pool) return PKV_ERR_NULL_POINTER;
  if (quant && (!k_scales || !k_biases || !v_scales || !v_biases)) return PKV_ERR_NULL_POINTER;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(error_flag, 4))
    return PKV_ERR_MISALIGNED;
  if (quant && (!aligned(k_scales, 4) || !aligned(k_biases, 4) || !aligned(v_scales, 4) || !aligned(v_biases, 4)))
    return PKV_ERR_MISALIGNED;
  pkv::AppendParams a{};
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.dst = append_target(quant, k_pool, v_pool, k_scales, k_biases, v_scales, v_biases);
  a.error_flag = error_flag;
  a.num_blocks = layout->num_blocks;
  a.num_kv_heads = layout->num_kv_heads;
  a.block_size = layout->block_size;
  a.max_blocks = max_blocks_per_seq;
  a.n_new = n_new;
  (void)cudaGetLastError();
  cudaError_t e = pkv::launch_append(a, layout->bits, layout->head_dim, v_dim(layout), num_seqs,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("append kernel launch", e);
  return PKV_OK;
}

int pkv_paged_gather(const void* pool, int32_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                     int32_t row_bytes, const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs,
                     int32_t max_blocks_per_seq, int32_t max_len, void* out, int32_t* error_flag, void* stream) {
  if (num_blocks <= 0 || num_kv_heads <= 0 || num_kv_heads > 65535 || block_size <= 0 || row_bytes <= 0 ||
      row_bytes % 4 || num_seqs <= 0 || num_seqs > 65535 || max_blocks_per_seq <= 0 || max_len < 0)
    return PKV_ERR_BAD_PARAMS;
  if (!pool || !block_tables || !seq_lens || !out) return PKV_ERR_NULL_POINTER;
  if (!aligned(pool, 16) || !aligned(out, 16) || !aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
      !aligned(error_flag, 4))
    return PKV_ERR_MISALIGNED;
  pkv::GatherParams g{};
  g.pool = static_cast<const uint8_t*>(pool);
  g.block_tables = block_tables;
  g.seq_lens = seq_lens;
  g.out = static_cast<uint8_t*>(out);
  g.error_flag = error_flag;
  g.num_blocks = num_blocks;
  g.num_kv_heads = num_kv_heads;
  g.block_size = block_size;
  g.row_words = row_bytes / 4;
  g.max_blocks = max_blocks_per_seq;
  g.max_len = max_len;
  (void)cudaGetLastError();
  cudaError_t e = pkv::launch_gather(g, num_seqs, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("gather kernel launch", e);
  return PKV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// The entry point that allocates nothing (pkv_paged_decode_attention_no_alloc)
// ---------------------------------------------------------------------------
namespace {

// Scratch for the partition states of the no-alloc entry point. Every GPU that
// loads this library holds it until the process exits; every call on a device
// shares it.
static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 256;
std::mutex g_scratch_mutex;
// Per device: the context the address was looked up in, and the address.
CUcontext g_scratch_context[kMaxScratchDevices] = {};
void* g_scratch_address[kMaxScratchDevices] = {};

// The driver's cuCtxGetCurrent, reached through the runtime (the library links no
// driver library).
PFN_cuCtxGetCurrent_v4000 current_context_getter() {
  static PFN_cuCtxGetCurrent_v4000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuCtxGetCurrent_v4000>(nullptr);
    return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }();
  return fn;
}

// Device address of g_static_scratch on the current device. Host code only has a
// host-side stand-in for the array's name, so the address is looked up with the
// device current and cached per device, keyed on the device's current context: a
// reset of the device (cudaDeviceReset) makes a new primary context, which loads the
// module again, so the address is looked up again there.
int static_scratch_address(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxScratchDevices) return PKV_ERR_BAD_PARAMS;
  auto get_ctx = current_context_getter();
  if (!get_ctx) {
    std::snprintf(g_cuda_error, sizeof(g_cuda_error), "cuCtxGetCurrent entry point unavailable");
    return PKV_ERR_CUDA;
  }
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  // No context current on this thread yet (the runtime makes it current on first
  // use), or another one than at the last look-up: look the address up again, which
  // also makes the device's primary context current.
  if (!ctx || !g_scratch_address[dev] || g_scratch_context[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress", e);
    if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    g_scratch_address[dev] = p;
    g_scratch_context[dev] = ctx;
  }
  *ptr = g_scratch_address[dev];
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_paged_decode_attention_no_alloc(const pkv_pool_layout* layout, const pkv_decode_params* params,
                                        const void* q, const void* k_pool, const void* v_pool,
                                        const void* k_scales, const void* k_biases, const void* v_scales,
                                        const void* v_biases, const int32_t* block_tables,
                                        const int32_t* seq_lens, float scale, void* out, int32_t* error_flag,
                                        void* stream) {
  int rc = check_layout(layout);
  if (rc) return rc;
  rc = check_params(layout, params);
  if (rc) return rc;
  const bool quant = layout->bits != 16;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return PKV_ERR_NULL_POINTER;
  if (quant && (!k_scales || !k_biases || !v_scales || !v_biases)) return PKV_ERR_NULL_POINTER;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(error_flag, 4))
    return PKV_ERR_MISALIGNED;
  if (quant && (!aligned(k_scales, 16) || !aligned(k_biases, 16) || !aligned(v_scales, 16) || !aligned(v_biases, 16)))
    return PKV_ERR_MISALIGNED;

  int sms = 0;
  rc = device_sm_count(&sms);
  if (rc) return rc;
  pkv_decode_params local = *params;
  pkv_plan plan;
  rc = plan_impl(layout, &local, sms, &plan);
  if (rc) return rc;
  if (plan.workspace_bytes > PKV_STATIC_SCRATCH_BYTES) {
    if (params->partition_tokens > 0) return PKV_ERR_SCRATCH_TOO_SMALL;  // the caller's partition size does not fit
    // A library-chosen plan coarsens its partitions until their states fit
    // (a single partition needs no scratch at all).
    // Doubling stops at the table's length, where one partition needs no scratch, so
    // the loop ends within 32 rounds; the bound on the rounds states it.
    const long long max_len = static_cast<long long>(params->max_blocks_per_seq) * layout->block_size;
    long long part = plan.partition_tokens;
    for (int round = 0; plan.workspace_bytes > PKV_STATIC_SCRATCH_BYTES; ++round) {
      if (round >= 40 || part >= max_len) return PKV_ERR_SCRATCH_TOO_SMALL;
      part = std::min(2 * part, max_len);
      local.partition_tokens = static_cast<int32_t>(part);
      rc = plan_impl(layout, &local, sms, &plan);
      if (rc) return rc;
    }
  }
  void* scratch = nullptr;
  rc = static_scratch_address(&scratch);
  if (rc) return rc;
  return pkv_paged_decode_attention(layout, &local, q, k_pool, v_pool, k_scales, k_biases, v_scales, v_biases,
                                    block_tables, seq_lens, scale, out, scratch, PKV_STATIC_SCRATCH_BYTES,
                                    error_flag, stream);
}

const char* pkv_strerror(int code) {
  switch (code) {
    case PKV_OK: return "success";
    case PKV_ERR_NULL_POINTER: return "a required pointer is NULL";
    case PKV_ERR_MISALIGNED: return "a pointer is not aligned (16 bytes for data planes, 4 for int32 arrays)";
    case PKV_ERR_BAD_LAYOUT: return "unsupported pool layout (bits, group_size, head dims or block_size)";
    case PKV_ERR_BAD_PARAMS: return "bad decode parameters (sequences, heads, n_query, table width or partition)";
    case PKV_ERR_UNSUPPORTED_SHAPE:
      return "no kernel for this pair of key/value head dims with this many query rows per KV head";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "workspace missing or smaller than the plan needs";
    case PKV_ERR_CUDA: return "a CUDA call failed (see pkv_last_cuda_error)";
    case PKV_ERR_SCRATCH_TOO_SMALL:
      return "the partition states exceed the static scratch of the no-alloc entry point (PKV_STATIC_SCRATCH_BYTES); "
             "use larger partition_tokens or 0";
    default: return "unknown error code";
  }
}

const char* pkv_last_cuda_error(void) { return g_cuda_error; }

uint64_t pkv_set_wait_limit_ns(uint64_t ns) {
  return g_wait_limit_ns.exchange(ns == 0 ? pkv::kWaitLimitNs : ns, std::memory_order_relaxed);
}

int pkv_version(void) { return 200; }

}  // extern "C"
