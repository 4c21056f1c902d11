// C ABI of the paged decode attention library: argument checks, the partition
// plan, TMA descriptors and kernel launches. See include/pkv_decode.h.
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

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

PartialInfo partial_info(int bits, int head_dim, int ntiles) {
  if (bits == 16) return pkv::partial_info_bf16(head_dim, ntiles);
  if (bits == 4) return pkv::partial_info_u4(head_dim, ntiles);
  if (bits == 8) return pkv::partial_info_u8(head_dim, ntiles);
  return PartialInfo{false, 0, 0, 0, 0, 0};
}

int chunk_rows_of(int bits) { return bits == 16 ? 16 : 32; }

int check_layout(const pkv_pool_layout* L) {
  if (!L) return PKV_ERR_NULL_POINTER;
  if (L->num_blocks <= 0 || L->num_kv_heads <= 0 || L->block_size <= 0) return PKV_ERR_BAD_LAYOUT;
  if (L->bits != 16 && L->bits != 4 && L->bits != 8) return PKV_ERR_BAD_LAYOUT;
  if (L->bits == 16) {
    if (L->head_dim != 64 && L->head_dim != 128 && L->head_dim != 256) return PKV_ERR_BAD_LAYOUT;
  } else {
    if (L->group_size != 64) return PKV_ERR_BAD_LAYOUT;
    if (L->head_dim != 128 && L->head_dim != 256) return PKV_ERR_BAD_LAYOUT;
  }
  if (L->block_size % chunk_rows_of(L->bits)) return PKV_ERR_BAD_LAYOUT;
  const long long rows = static_cast<long long>(L->num_blocks) * L->num_kv_heads * L->block_size;
  if (rows >= (1ll << 31)) return PKV_ERR_BAD_LAYOUT;  // TMA row coordinates are int32
  if (L->num_kv_heads > 65535) return PKV_ERR_BAD_LAYOUT;
  return PKV_OK;
}

int check_params(const pkv_pool_layout* L, const pkv_decode_params* P) {
  if (!P) return PKV_ERR_NULL_POINTER;
  if (P->num_seqs <= 0 || P->num_seqs > 65535) return PKV_ERR_BAD_PARAMS;
  if (P->num_q_heads <= 0 || P->num_q_heads % L->num_kv_heads) return PKV_ERR_BAD_PARAMS;
  if (P->n_query < 1 || P->max_blocks_per_seq <= 0 || P->partition_tokens < 0) return PKV_ERR_BAD_PARAMS;
  if (static_cast<long long>(P->max_blocks_per_seq) * L->block_size >= (1ll << 31)) return PKV_ERR_BAD_PARAMS;
  const long long nq = static_cast<long long>(P->num_q_heads / L->num_kv_heads) * P->n_query;
  if (nq > 64) return PKV_ERR_UNSUPPORTED_SHAPE;
  if (!partial_info(L->bits, L->head_dim, ceil_div(nq, 8)).exists) return PKV_ERR_UNSUPPORTED_SHAPE;
  return PKV_OK;
}

int round_up(long long x, int m) { return static_cast<int>((x + m - 1) / m * m); }

int plan_impl(const pkv_pool_layout* L, const pkv_decode_params* P, int sm_count, pkv_plan* out) {
  const int ch = chunk_rows_of(L->bits);
  const long long max_len = static_cast<long long>(P->max_blocks_per_seq) * L->block_size;
  long long part;
  if (P->partition_tokens > 0) {
    part = round_up(P->partition_tokens, ch);
  } else {
    // Enough partitions of the longest sequence that the grid covers the GPU a
    // few times over (2 CTAs fit per SM), but never below 256 rows a partition.
    const long long target = 4ll * (sm_count > 0 ? sm_count : 1) * 2;
    const long long units = static_cast<long long>(P->num_seqs) * L->num_kv_heads;
    const long long floor_rows = 256;
    part = round_up(max_len, ch);
    while (units * ((max_len + part - 1) / part) < target && part > floor_rows) {
      long long half = round_up(part / 2, ch);
      part = half < floor_rows ? floor_rows : half;
    }
  }
  if (part >= max_len) part = round_up(max_len, ch);
  const int max_parts = ceil_div(max_len, part);
  const long long nq = static_cast<long long>(P->num_q_heads / L->num_kv_heads) * P->n_query;
  const PartialInfo info = partial_info(L->bits, L->head_dim, ceil_div(nq, 8));
  out->partition_tokens = static_cast<int32_t>(part);
  out->max_partitions = max_parts;
  out->chunk_rows = info.chunk_rows;
  out->sm_count = sm_count;
  out->threads_per_cta = info.threads;
  out->smem_bytes = info.smem_bytes;
  out->workspace_bytes = 0;
  if (max_parts > 1) {
    const size_t slots = static_cast<size_t>(P->num_seqs) * P->num_q_heads * P->n_query * max_parts;
    const size_t o_bytes = (slots * L->head_dim * sizeof(float) + 255) / 256 * 256;
    out->workspace_bytes = o_bytes + slots * 2 * sizeof(float);
  }
  return PKV_OK;
}

int device_sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail("cudaDeviceGetAttribute", e);
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

// 2-D view of one pool plane: rows = num_blocks*HK*BS, `row_elems` elements per
// row; boxes of `box_rows` rows by `box_row_bytes` bytes with the matching swizzle.
int pool_tensor_map(CUtensorMap* map, const void* base, int elem_bytes, long long row_elems, long long rows,
                    const PartialInfo& info) {
  auto encode = tensor_map_encoder();
  if (!encode) {
    std::snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled entry point unavailable");
    return PKV_ERR_CUDA;
  }
  const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_elems), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_elems * elem_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(info.box_row_bytes / elem_bytes),
                       static_cast<cuuint32_t>(info.chunk_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = info.box_row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
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

constexpr int kPassPartial = 1;
constexpr int kPassMerge = 2;

int enqueue_decode(const pkv_pool_layout* layout, const pkv_decode_params* params, const void* q,
                   const void* k_pool, const void* v_pool, const void* k_scales, const void* k_biases,
                   const void* v_scales, const void* v_biases, const int32_t* block_tables,
                   const int32_t* seq_lens, float scale, void* out, void* workspace, size_t workspace_bytes,
                   int32_t* error_flag, void* stream, int passes) {
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

  int sms = 0;
  rc = device_sm_count(&sms);
  if (rc) return rc;
  pkv_plan plan;
  rc = plan_impl(layout, params, sms, &plan);
  if (rc) return rc;
  if (plan.workspace_bytes > 0 && (!workspace || workspace_bytes < plan.workspace_bytes))
    return PKV_ERR_WORKSPACE_TOO_SMALL;

  const int D = layout->head_dim, HK = layout->num_kv_heads;
  const int nq = (params->num_q_heads / HK) * params->n_query;
  const int ntiles = ceil_div(nq, 8);
  const PartialInfo info = partial_info(layout->bits, D, ntiles);
  const long long rows = static_cast<long long>(layout->num_blocks) * HK * layout->block_size;
  const int elem = info.tensor_elem_bytes;
  const long long row_elems = quant ? static_cast<long long>(D) * layout->bits / 8 : D;

  CUtensorMap tk, tv;
  if (partial) {
    rc = pool_tensor_map(&tk, k_pool, elem, row_elems, rows, info);
    if (rc) return rc;
    rc = pool_tensor_map(&tv, v_pool, elem, row_elems, rows, info);
    if (rc) return rc;
  }

  pkv::PartialParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.k_scales = static_cast<const __nv_bfloat16*>(k_scales);
  p.k_biases = static_cast<const __nv_bfloat16*>(k_biases);
  p.v_scales = static_cast<const __nv_bfloat16*>(v_scales);
  p.v_biases = static_cast<const __nv_bfloat16*>(v_biases);
  p.out = static_cast<__nv_bfloat16*>(out);
  const size_t slots = static_cast<size_t>(params->num_seqs) * params->num_q_heads * params->n_query * plan.max_partitions;
  const size_t o_bytes = (slots * D * sizeof(float) + 255) / 256 * 256;
  p.ws_o = plan.max_partitions > 1 ? static_cast<float*>(workspace) : nullptr;
  p.ws_ml = plan.max_partitions > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes) : nullptr;
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

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)cudaGetLastError();  // start from a clean error state
  const dim3 grid(plan.max_partitions, HK, params->num_seqs);
  cudaError_t e = cudaSuccess;
  if (partial) {
    if (layout->bits == 16)
      e = pkv::launch_partial_bf16(D, ntiles, p, tk, tv, grid, st);
    else if (layout->bits == 4)
      e = pkv::launch_partial_u4(D, ntiles, p, tk, tv, grid, st);
    else
      e = pkv::launch_partial_u8(D, ntiles, p, tk, tv, grid, st);
    if (e != cudaSuccess) return cuda_fail("partial kernel launch", e);
  }

  if ((passes & kPassMerge) && plan.max_partitions > 1) {
    pkv::MergeParams m{};
    m.ws_o = p.ws_o;
    m.ws_ml = p.ws_ml;
    m.seq_lens = seq_lens;
    m.out = p.out;
    m.error_flag = error_flag;
    m.rows_per_seq = params->num_q_heads * params->n_query;
    m.n_query = params->n_query;
    m.head_dim = D;
    m.max_len = params->max_blocks_per_seq * layout->block_size;
    m.partition_tokens = plan.partition_tokens;
    m.max_partitions = plan.max_partitions;
    e = pkv::launch_merge(m, params->num_seqs * params->num_q_heads * params->n_query, st);
    if (e != cudaSuccess) return cuda_fail("merge kernel launch", e);
  }
  return PKV_OK;
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
void* g_scratch_address[kMaxScratchDevices] = {};

// Device address of g_static_scratch on the current device. Host code only has a
// host-side stand-in for the array's name, so the address is looked up once per
// device, with that device current, and cached.
int static_scratch_address(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxScratchDevices) return PKV_ERR_BAD_PARAMS;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_address[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress", e);
    g_scratch_address[dev] = p;
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
    long long part = plan.partition_tokens;
    while (plan.workspace_bytes > PKV_STATIC_SCRATCH_BYTES) {
      part *= 2;
      local.partition_tokens = static_cast<int32_t>(part < (1ll << 30) ? part : (1ll << 30));
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
    case PKV_ERR_BAD_LAYOUT: return "unsupported pool layout (bits, group_size, head_dim or block_size)";
    case PKV_ERR_BAD_PARAMS: return "bad decode parameters (sequences, heads, n_query, table width or partition)";
    case PKV_ERR_UNSUPPORTED_SHAPE: return "too many query rows per KV head for this head_dim";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "workspace missing or smaller than the plan needs";
    case PKV_ERR_CUDA: return "a CUDA call failed (see pkv_last_cuda_error)";
    case PKV_ERR_SCRATCH_TOO_SMALL:
      return "the partition states exceed the static scratch of the no-alloc entry point (PKV_STATIC_SCRATCH_BYTES); "
             "use larger partition_tokens or 0";
    default: return "unknown error code";
  }
}

const char* pkv_last_cuda_error(void) { return g_cuda_error; }

int pkv_version(void) { return 100; }

}  // extern "C"
