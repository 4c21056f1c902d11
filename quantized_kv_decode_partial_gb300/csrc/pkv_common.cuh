// Device helpers shared by the paged decode kernels: inline PTX for mbarriers,
// TMA and cp.async copies, ldmatrix, warp-level MMA and movmatrix, cluster barriers
// and distributed shared memory, plus the kernel parameter blocks. sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

constexpr int kDevErrBadBlock = 1;
constexpr int kDevErrBadSeqLen = 2;
constexpr int kDevErrTimeout = 4;

// Default upper bound of one pipeline wait before the kernel gives up (nanoseconds).
// The main loop of the partial kernel takes its bound from PartialParams (the host
// may lower it); draining copies in flight after a give-up always uses this one.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Where appended rows are written: the pools and, for affine pages, the scale and
// bias planes (all [NB, HK, BS, ...]).
struct AppendTarget {
  __nv_bfloat16* k_pool_bf16;  // bf16 pages
  __nv_bfloat16* v_pool_bf16;
  uint32_t* k_pool_words;      // affine pages
  uint32_t* v_pool_words;
  __nv_bfloat16* k_scales;
  __nv_bfloat16* k_biases;
  __nv_bfloat16* v_scales;
  __nv_bfloat16* v_biases;
};

struct PartialParams {
  const __nv_bfloat16* q;     // [B, HQ, N, D]
  const int32_t* block_tables;  // [B, max_blocks]
  const int32_t* seq_lens;    // [B]
  const __nv_bfloat16* k_scales;  // [NB, HK, BS, D/64]   (affine pages)
  const __nv_bfloat16* k_biases;
  const __nv_bfloat16* v_scales;
  const __nv_bfloat16* v_biases;
  __nv_bfloat16* out;   // [B, HQ, N, DV], written directly with one partition or a cluster merge
  __nv_bfloat16* out_mirror;  // optional second destination of those writes (mapped host memory)
  float* ws_o;          // [B*HQ*N, max_partitions, D]
  float* ws_ml;         // [B*HQ*N, max_partitions, 2]  (running max in log2 units, normaliser)
  int32_t* error_flag;  // optional
  int num_blocks, num_kv_heads, block_size, max_blocks;
  int num_q_heads, n_query, nq;  // nq = (HQ/HK) * n_query rows served per KV head
  int partition_tokens, max_partitions;
  int mode;           // kModeSingle / kModeWorkspace / kModeCluster / kModeBalanced
  int piece_log2;     // blocks smaller than a chunk: a chunk spans 2^piece_log2 blocks (else 0)
  int num_seqs;       // B (read by the balanced schedule)
  int window;         // sliding window in rows (0: none)
  int host_inputs;    // kHost* bits: inputs a host-driven step keeps in host memory
  float score_scale;  // softmax scale * log2(e)
  unsigned long long wait_limit_ns;  // bound of one main-loop pipeline wait
  // Fused append (k_new != nullptr): the N new rows of every (sequence, KV head),
  // cache rows len-N .. len-1, are written into their pages by the CTA whose
  // partition holds them, before it reads that partition.
  const __nv_bfloat16* k_new;  // [B, HK, N, D]
  const __nv_bfloat16* v_new;
  AppendTarget app;
};

// Inputs of a host-driven step that live in (mapped) host memory, written by the host
// before the launch and by no kernel.
constexpr int kHostSeqLens = 1;
constexpr int kHostQuery = 2;
constexpr int kHostTables = 4;

// How the partial kernel finishes.
constexpr int kModeSingle = 0;     // one partition: the CTA writes bf16 output
constexpr int kModeWorkspace = 1;  // partition states go to the workspace; the merge kernel follows
constexpr int kModeCluster = 2;    // the partitions of a (sequence, KV head) form one thread-block
                                   // cluster and merge through distributed shared memory
constexpr int kModeBalanced = 3;   // equal runs of the flattened chunk list per page group; states to
                                   // the workspace, one per (page group, unit) run; the merge kernel follows
constexpr int kMaxClusterParts = 16;  // largest cluster (non-portable size)
constexpr int kMaxBalancedSeqs = 256;  // sequences a balanced schedule takes (its prefix lives in shared memory)

struct MergeParams {
  const float* ws_o;
  const float* ws_ml;
  const int32_t* seq_lens;
  __nv_bfloat16* out;
  __nv_bfloat16* out_mirror;  // optional second destination (mapped host memory)
  int32_t* error_flag;
  int rows_per_seq;  // HQ * N
  int n_query, head_dim, max_len, partition_tokens, max_partitions;
  int window;  // sliding window in rows (0: none)
  int rows;    // output rows (B * HQ * N)
  int groups;  // partition groups per output row (merge_groups)
  // Balanced schedule (bal_runs > 0): the states of a unit's runs sit in consecutive
  // workspace slots; the rest describes the partial pass's chunk list.
  int bal_runs;  // page groups of the partial grid (0: partitions)
  int num_seqs, num_kv_heads, nq, chunk_rows;
};

struct AppendParams {
  const __nv_bfloat16* k_new;  // [B, HK, n_new, D]
  const __nv_bfloat16* v_new;
  const int32_t* block_tables;
  const int32_t* seq_lens;     // rows before the append
  AppendTarget dst;
  int32_t* error_flag;
  int num_blocks, num_kv_heads, block_size, max_blocks, n_new;
};

struct GatherParams {
  const uint8_t* pool;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  uint8_t* out;
  int32_t* error_flag;
  int num_blocks, num_kv_heads, block_size, row_words, max_blocks, max_len;
};

// ---------------------------------------------------------------------------
// small PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy global writes before later async-proxy (TMA)
// reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// try_wait with an explicit bound on how long the thread may be suspended in it
// (suspendTimeHint, nanoseconds), instead of the system's own.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Bounds below this one (nanoseconds) also bound each suspension inside try_wait, which
// may otherwise outlast them.
constexpr unsigned long long kShortWaitLimitNs = 1000000ull;

// Waits, as a whole warp, for the phase of the mbarrier with the given parity. Gives
// up when `abort_flag` is set by another warp or after `limit_ns`, in which case it
// raises the abort flag and the timeout error bit; returns true when the phase
// completed. Every lane observes the phase, and the give-up decision is taken by lane
// 0 and shared, so the warp never splits.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               int32_t* error_flag, unsigned long long limit_ns) {
  const bool short_limit = limit_ns < kShortWaitLimitNs;  // warp-uniform (a kernel parameter)
  const uint32_t hint = static_cast<uint32_t>(short_limit ? limit_ns : 0ull);
  bool done = short_limit ? mbar_try_wait_hint(bar, parity, hint) : mbar_try_wait(bar, parity);
  if (__all_sync(0xffffffffu, done)) return true;
  const bool leader = (threadIdx.x & 31) == 0;
  const unsigned long long start = leader ? global_timer_ns() : 0ull;
  while (true) {
    if (!done) done = short_limit ? mbar_try_wait_hint(bar, parity, hint) : mbar_try_wait(bar, parity);
    int stop = 0;
    if (leader) {
      if (*abort_flag) {
        stop = 1;
      } else if (global_timer_ns() - start > limit_ns) {
        *abort_flag = 1;
        if (error_flag) atomicOr(error_flag, kDevErrTimeout);
        stop = 1;
      }
    }
    stop = __shfl_sync(0xffffffffu, stop, 0);
    if (__all_sync(0xffffffffu, done)) return true;
    if (stop) return false;
  }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

// Fetches a TMA descriptor (a __grid_constant__ kernel parameter) ahead of its first use.
// Starts fetching the 128-byte line holding `ptr` into L1 (and L2).
__device__ __forceinline__ void prefetch_l1(const void* ptr) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// 16-byte copy global -> shared through the load/store path (cp.async, L2 only), with
// an L2 policy hint. Addresses 16-byte aligned.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}

// Makes the current phase of the mbarrier also wait for this thread's earlier cp.async
// copies: its pending count is raised by one now and lowered when they have landed.
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// D = A * B + D, m16n8k16, bf16 inputs, f32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B + D, m16n8k16, fp16 inputs, f32 accumulators.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit elements held one row-pair per thread.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Thread-block cluster barrier: every thread of every CTA of the cluster arrives;
// writes before it (shared memory included) are visible to the cluster after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// First half of a cluster barrier without memory ordering, and the second half with
// acquire: together they tell that every member has started. Every thread of every
// member takes part, arrive before wait.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Stores at shared-memory address `addr` (this CTA's layout) in the shared memory of
// cluster CTA `rank`: one f32, or a 16-byte-aligned float4.
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_f32x4(uint32_t addr, uint32_t rank, float4 v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// Reads an f32 at shared-memory address `addr` (this CTA's layout) in the shared
// memory of cluster CTA `rank`.
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Reads the 16-byte-aligned float4 at `addr` (this CTA's layout) in the shared memory
// of cluster CTA `rank`.
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr, uint32_t rank) {
  uint32_t remote;
  float4 v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}

// Named CTA barrier over `count` threads that also ORs a predicate across them: every
// participant gets the same answer.
__device__ __forceinline__ bool group_barrier_any(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Programmatic dependent launch: let the next kernel on the stream be scheduled
// now (it still waits for this grid's completion before reading its results).
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the grids this kernel depends on have completed and their memory
// operations are visible (no-op when launched without a programmatic dependency).
__device__ __forceinline__ void wait_for_prerequisite_grids() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Read-only global loads kept in program order (volatile): a load issued before a
// branch is never moved past it, so its latency overlaps whatever the branch waits for.
__device__ __forceinline__ uint4 ld_nc_keep_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}
__device__ __forceinline__ uint2 ld_nc_keep_v2(const void* ptr) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(ptr));
  return v;
}
__device__ __forceinline__ uint32_t ld_nc_keep_u32(const void* ptr) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(ptr));
  return v;
}

// Alignment of the first partition of a windowed sequence: a multiple of every
// chunk size (16 or 32 rows), so partition starts stay on chunk boundaries.
constexpr int kWindowAlign = 32;

// Row at which partition 0 of a sequence starts. Without a window, row 0. With a
// window of W rows, the chunk boundary at or below the lowest row any of the N
// queries sees (len - N + 1 - W), so the partitions tile the visible span and
// nothing below it.
__host__ __device__ __forceinline__ int partition_base(int len, int n_query, int window) {
  if (window <= 0) return 0;
  const int lo = len - n_query + 1 - window;
  return lo > 0 ? lo / kWindowAlign * kWindowAlign : 0;
}

// ---- balanced schedule
// The partial pass reads, for every (sequence b, KV head) unit, the chunks of kCh rows
// from bal_first_row (0, or with a window the chunk boundary at or below the lowest
// row any query sees) up to the length. Units are listed sequence-major, KV heads
// within a sequence, chunks within a unit, giving T chunks in all; page group v of V
// takes the run [v T / V, (v + 1) T / V) of that list, split where it crosses units.
// The merge pass recomputes the same list from the lengths.
__host__ __device__ __forceinline__ int bal_first_row(int len, int n_query, int window, int ch) {
  const int lo = len - n_query + 1 - window;
  return window > 0 && lo > 0 ? lo / ch * ch : 0;
}

// Chunks of one unit of a sequence of length len; 0 for a length the partial pass rejects.
__host__ __device__ __forceinline__ int bal_unit_chunks(int len, int n_query, int window, int max_len, int ch) {
  if (len < n_query || len > max_len) return 0;
  return (len - bal_first_row(len, n_query, window, ch) + ch - 1) / ch;
}

// Fills S[0..B] with the index of each sequence's first chunk in the list (S[B] = T)
// and lens[0..B-1] with the lengths. Called by every thread of the block; B <=
// kMaxBalancedSeqs; ends with a block barrier.
__device__ __forceinline__ void bal_scan(const int32_t* seq_lens, int B, int HK, int n_query, int window, int max_len,
                                         int ch, int* S, int* lens) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int len = seq_lens[b];
    lens[b] = len;
    S[b + 1] = HK * bal_unit_chunks(len, n_query, window, max_len, ch);
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // one warp: lane l sums entries 8l .. 8l+7, then a warp scan
    constexpr int kPer = kMaxBalancedSeqs / 32;
    const int lane = threadIdx.x;
    int v[kPer];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = lane * kPer + j;
      v[j] = b < B ? S[b + 1] : 0;
      sum += v[j];
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += n;
    }
    __syncwarp();  // every lane has read its entries before any lane writes
    int run = incl - sum;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = lane * kPer + j;
      if (b < B) S[b] = run;
      run += v[j];
    }
    if (lane == 31) S[B] = incl;
  }
  __syncthreads();
}

// The sequence whose units hold chunk x (0 <= x < S[B]): the last b with S[b] <= x.
__device__ __forceinline__ int bal_seq_of(const int* S, int B, int x) {
  int lo = 0, hi = B;  // S[lo] <= x < S[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (S[mid] <= x) {
      lo = mid;
    } else {
      hi = mid;
    }
  }
  return lo;
}

// First chunk of page group v's run, and the page group whose run holds chunk x.
__host__ __device__ __forceinline__ int bal_run_start(int v, int T, int V) {
  return static_cast<int>(static_cast<long long>(v) * T / V);
}
__host__ __device__ __forceinline__ int bal_run_of(int x, int T, int V) {
  return static_cast<int>(((static_cast<long long>(x) + 1) * V - 1) / T);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packs (lo, hi) into a bf16x2 word, round to nearest even; lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packs (lo, hi) into an fp16x2 word, round to nearest even; lo in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Shared-memory address of 16-byte chunk `chunk` of row `row` inside a TMA box
// written with the 128-byte (rows of 128 B) or 64-byte (rows of 64 B) swizzle.
template <int RB>
__device__ __forceinline__ uint32_t swizzled(uint32_t box_base, int row, int chunk) {
  static_assert(RB == 128 || RB == 64, "box rows of 64 or 128 bytes");
  if constexpr (RB == 128) {
    return box_base + row * 128 + ((chunk ^ (row & 7)) << 4);
  } else {
    return box_base + row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
  }
}

}  // namespace pkv
