// Merge pass (log-sum-exp combination of partition states) and the bit-exact
// block-table gather.
#include "pkv_launch.h"

namespace pkv {

// A thread owns four consecutive head dims of one output row (sequence, query head,
// query index) and every groups-th of its partitions: a row takes `groups` groups of
// D/4 threads, a CTA 256 / (groups * D/4) rows. The partition states hold the running
// maximum in log2 units, the normaliser and the unnormalised output; partitions whose
// maximum is -inf saw no visible key and are skipped (kvq4-decode.ts and
// multi-query.ts merge kernels).
// Output = sum_p 2^(m_p-M) o_p / sum_p 2^(m_p-M) l_p.
// Each group merges its partitions online against its own running maximum; with more
// than one group per row the groups' states are combined once in shared memory. A
// thread's first kMergeUnroll partition slots are requested together with the sequence
// length (the slots exist for every row; those past the row's partition count are
// dropped once the length arrives), so a row with at most groups * kMergeUnroll
// partitions costs one memory round trip. The host takes the fewest groups that cover
// the partitions in that round trip, so that short rows pack several to a CTA and the
// grid stays within one wave.
constexpr int kMergeThreads = 256;
constexpr int kMergeUnroll = 4;

__device__ __forceinline__ void merge_one(float2 s, const float4& v, float& M, float& den, float4& acc) {
  if (s.x == -INFINITY) return;  // no visible key in this partition
  if (s.x > M) {                 // new running maximum: rescale what is summed so far
    const float c = fast_exp2(M - s.x);  // 0 while nothing is summed (M = -inf)
    den *= c;
    acc.x *= c;
    acc.y *= c;
    acc.z *= c;
    acc.w *= c;
    M = s.x;
  }
  const float w = fast_exp2(s.x - M);
  den = fmaf(w, s.y, den);
  acc.x = fmaf(w, v.x, acc.x);
  acc.y = fmaf(w, v.y, acc.y);
  acc.z = fmaf(w, v.z, acc.z);
  acc.w = fmaf(w, v.w, acc.w);
}

__global__ void __launch_bounds__(kMergeThreads) pkv_merge_kernel(const __grid_constant__ MergeParams p) {
  __shared__ float red_m[kMergeThreads];
  __shared__ float4 red_o[kMergeThreads];
  __shared__ float red_l[kMergeThreads];
  const int lanes = p.head_dim / 4;    // threads per group
  const int span = lanes * p.groups;  // threads per row
  const int row = blockIdx.x * (kMergeThreads / span) + threadIdx.x / span;
  const int grp = (threadIdx.x % span) / lanes, d = (threadIdx.x % lanes) * 4;
  const bool live = row < p.rows;  // the last CTA may hold fewer rows
  wait_for_prerequisite_grids();   // launched early behind the partial pass; its states are ready after this
  const int b = live ? row / p.rows_per_seq : 0;
  // The row's states: state i at ml[i * mstride] (m, l) and ob[i * ostride] (its four dims).
  const float2* ml;
  const float4* ob;
  int mstride, ostride, np;
  int run0 = 0, T = 0;  // balanced: the first run over the row's unit, and the list's length
  // Whether state i exists. A balanced run over fewer chunks than page groups may be
  // empty, and an empty run writes no state.
  auto has_state = [&](int i) {
    return i < np && (p.bal_runs == 0 ||
                      bal_run_start(run0 + i, T, p.bal_runs) < bal_run_start(run0 + i + 1, T, p.bal_runs));
  };
  float2 s[kMergeUnroll];
  float4 v[kMergeUnroll];
  if (p.bal_runs > 0) {
    // Balanced schedule: the runs that cover this row's unit, from the same chunk list
    // the partial pass split. Their states sit in consecutive slots, nq rows apart.
    __shared__ int bal_S[kMaxBalancedSeqs + 1], bal_len[kMaxBalancedSeqs];
    bal_scan(p.seq_lens, p.num_seqs, p.num_kv_heads, p.n_query, p.window, p.max_len, p.chunk_rows, bal_S, bal_len);
    const int in_seq = row - b * p.rows_per_seq;  // (query head, query index) within the sequence
    const int h = in_seq / p.n_query, rep = p.rows_per_seq / p.n_query / p.num_kv_heads;
    const int hk = h / rep, r = in_seq - hk * rep * p.n_query;  // KV head, row within its nq
    const int n = (bal_S[b + 1] - bal_S[b]) / p.num_kv_heads;  // 0 for a rejected length: zeroed
    const int first = bal_S[b] + hk * n;
    T = bal_S[p.num_seqs];
    run0 = n > 0 ? bal_run_of(first, T, p.bal_runs) : 0;
    np = live && n > 0 ? bal_run_of(first + n - 1, T, p.bal_runs) - run0 + 1 : 0;
    const size_t st = (static_cast<size_t>(run0) + static_cast<size_t>(b) * p.num_kv_heads + hk) * p.nq + r;
    ml = reinterpret_cast<const float2*>(p.ws_ml) + st;
    ob = reinterpret_cast<const float4*>(p.ws_o + st * p.head_dim + d);
    mstride = p.nq;
    ostride = p.nq * p.head_dim / 4;
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const int i = grp + u * p.groups;
      const bool has = has_state(i);
      s[u] = has ? ml[static_cast<size_t>(i) * mstride] : make_float2(-INFINITY, 0.f);
      v[u] = has ? ob[static_cast<size_t>(i) * ostride] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  } else {
    const int slots = live ? p.max_partitions : 0;
    ml = reinterpret_cast<const float2*>(p.ws_ml) + static_cast<size_t>(row) * p.max_partitions;
    ob = reinterpret_cast<const float4*>(p.ws_o + static_cast<size_t>(row) * p.max_partitions * p.head_dim + d);
    mstride = 1;
    ostride = p.head_dim / 4;
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const int i = grp + u * p.groups;
      s[u] = i < slots ? ml[i] : make_float2(-INFINITY, 0.f);
      v[u] = i < slots ? ob[static_cast<size_t>(i) * ostride] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int len = p.seq_lens[b];
    const bool bad = len < p.n_query || len > p.max_len;  // flagged by the partial pass; the row is zeroed
    // Slot i holds the partition of rows [base + i P, base + (i + 1) P).
    const int base = bad ? 0 : partition_base(len, p.n_query, p.window);
    np = live && !bad ? (len - base + p.partition_tokens - 1) / p.partition_tokens : 0;
  }

  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kMergeUnroll; ++u)
    if (grp + u * p.groups < np) merge_one(s[u], v[u], M, den, acc);
  for (int i0 = grp + kMergeUnroll * p.groups; i0 < np; i0 += p.groups * kMergeUnroll) {
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const int i = i0 + u * p.groups;
      const bool has = has_state(i);
      s[u] = has ? ml[static_cast<size_t>(i) * mstride] : make_float2(-INFINITY, 0.f);
      v[u] = has ? ob[static_cast<size_t>(i) * ostride] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) merge_one(s[u], v[u], M, den, acc);
  }
  if (p.groups > 1) {  // the same for the whole CTA
    red_m[threadIdx.x] = M;
    red_o[threadIdx.x] = acc;
    red_l[threadIdx.x] = den;
    __syncthreads();
    if (grp != 0) return;
    float Mall = M;
    for (int g = 1; g < p.groups; ++g) Mall = fmaxf(Mall, red_m[threadIdx.x + g * lanes]);
    den = 0.f;
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (Mall != -INFINITY) {
      for (int g = 0; g < p.groups; ++g) {
        const int k = threadIdx.x + g * lanes;
        const float mg = red_m[k];
        if (mg == -INFINITY) continue;
        const float w = fast_exp2(mg - Mall);
        const float4 o = red_o[k];
        den = fmaf(w, red_l[k], den);
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
      }
    }
  }
  if (!live) return;
  const size_t o_off = static_cast<size_t>(row) * p.head_dim + d;
  __nv_bfloat162* out = reinterpret_cast<__nv_bfloat162*>(p.out + o_off);
  __nv_bfloat162* mirror = p.out_mirror ? reinterpret_cast<__nv_bfloat162*>(p.out_mirror + o_off) : nullptr;
  // den is 0 for a bad length (no partition merged) and for a row that saw no key
  const __nv_bfloat162 v0 = den > 0.f ? __floats2bfloat162_rn(acc.x / den, acc.y / den) : __floats2bfloat162_rn(0.f, 0.f);
  const __nv_bfloat162 v1 = den > 0.f ? __floats2bfloat162_rn(acc.z / den, acc.w / den) : __floats2bfloat162_rn(0.f, 0.f);
  out[0] = v0;
  out[1] = v1;
  if (mirror) {
    mirror[0] = v0;
    mirror[1] = v1;
  }
}

// Partition groups per output row: the fewest (a power of two) whose first round of
// loads covers `max_partitions`, at most one group per thread of a row's dims.
int merge_groups(int head_dim, int max_partitions) {
  const int most = kMergeThreads / (head_dim / 4);
  int g = 1;
  while (g < most && g * kMergeUnroll < max_partitions) g *= 2;
  return g;
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  const int rows_per_cta = kMergeThreads / (p.head_dim / 4 * p.groups);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((p.rows + rows_per_cta - 1) / rows_per_cta);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap with the partial pass's tail
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pkv_merge_kernel, p);
}

// Grid (row blocks, KV head, sequence); one warp per logical row, lanes copy
// 32-bit words. Bytes are copied unchanged, so the result is bit-exact.
constexpr int kGatherRowsPerCta = 32;

__global__ void __launch_bounds__(256) pkv_gather_kernel(const __grid_constant__ GatherParams p) {
  const int b = blockIdx.z, h = blockIdx.y;
  const int len = p.seq_lens[b];
  if (len < 0 || len > p.max_len || len > p.max_blocks * p.block_size) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0 && p.error_flag) atomicOr(p.error_flag, kDevErrBadSeqLen);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_begin = blockIdx.x * kGatherRowsPerCta;
  const uint32_t* pool = reinterpret_cast<const uint32_t*>(p.pool);
  uint32_t* out = reinterpret_cast<uint32_t*>(p.out);
  for (int r = warp; r < kGatherRowsPerCta; r += blockDim.x >> 5) {
    const int tok = row_begin + r;
    if (tok >= len) break;
    const int phys = p.block_tables[static_cast<size_t>(b) * p.max_blocks + tok / p.block_size];
    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
      if (lane == 0 && p.error_flag) atomicOr(p.error_flag, kDevErrBadBlock);
      continue;
    }
    const uint32_t* src =
        pool + ((static_cast<size_t>(phys) * p.num_kv_heads + h) * p.block_size + tok % p.block_size) * p.row_words;
    uint32_t* dst = out + ((static_cast<size_t>(b) * p.num_kv_heads + h) * p.max_len + tok) * p.row_words;
    for (int w = lane; w < p.row_words; w += 32) dst[w] = src[w];
  }
}

cudaError_t launch_gather(const GatherParams& p, int num_seqs, cudaStream_t stream) {
  if (p.max_len == 0) return cudaSuccess;
  dim3 grid((p.max_len + kGatherRowsPerCta - 1) / kGatherRowsPerCta, p.num_kv_heads, num_seqs);
  pkv_gather_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
