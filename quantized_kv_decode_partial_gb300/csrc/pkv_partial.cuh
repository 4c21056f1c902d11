// Partial pass of paged decode attention (one CTA per sequence x KV head x
// partition) for bf16 pages and affine 4-/8-bit pages, sm_103a.
//
// What one CTA computes is the per-partition state of the pages' partial
// kernels ("@mlx-bun/inference 0.0.0-stage -> 1.0.0", kernels/attention/paged.ts
// ``paged_attention_partial`` / ``paged_attention_affine_partial``;
// kvq4-decode.ts partial kernel): for every query row served by its KV head, the
// running maximum of the scores, the normaliser and the unnormalised output over
// the partition's visible keys. With a single partition the CTA finishes the
// softmax itself and writes bf16 output. Under the balanced schedule (BAL) a CTA
// instead serves one wave's share of the list of all (sequence, KV head, chunk)
// triples: each of its page groups reads an equal run of that list and writes one
// such state per (sequence, KV head) the run crosses.
//
// Design (GB300):
//  * Four warps per CTA (six to eight for grids of at most one CTA per SM and for CTAs
//    whose stages fill more than half an SM anyway, eight for query groups of eight
//    warps); with W warps,
//    warp w takes chunks w, w+W, w+2W, ... of the partition (16 rows for bf16
//    pages, 32 or 16 for affine pages) and runs its own pipeline: lane 0 issues
//    the copies of its chunk `kStagesPerWarp` ahead into a private ring of
//    shared-memory stages guarded by mbarriers, so no warp waits on another.
//    (With more query rows than one warp holds, WQ warps share a ring and read
//    each chunk for their own rows.) The block table is read 32 entries per
//    coalesced load and resolved into TMA row coordinates once per 32 chunks. A
//    chunk of one page and KV head is contiguous in the pool, so it travels as
//    one 3-D TMA copy per plane (each row split into segments of 64 or 128 bytes,
//    segment-major in shared memory and hardware-swizzled so the ldmatrix reads
//    below are free of bank conflicts); the affine scale/bias rows come by
//    16-byte cp.async copies of the warp's lanes, tracked by the same mbarrier.
//    K and V rows may have different head dims.
//  * Each K/V row in shared memory is read once and multiplied against all
//    REP*N query rows of its KV head (GQA reuse) with warp-level tensor-core
//    MMA (m16n8k16, bf16 in, f32 out):
//    S^T = K Q^T puts 16 keys on the M side and 8 query rows on N, and the
//    probabilities are transposed in registers (movmatrix) into the B operand
//    of O^T += V^T P^T. The online softmax (running max, normaliser, rescale)
//    runs in f32 on the accumulators in base 2 (the softmax scale times log2 e
//    is applied to the f32 scores; q itself is never re-rounded).
//  * Affine pages never dequantise element by element. Both products run as
//    fp16 MMAs in which a code c enters as the fp16 value with bit pattern c,
//    i.e. the exact subnormal c * 2^-24 (a 4-bit field at bit 4 of a 16-bit
//    half reads as 16 c * 2^-24, compensated by q/16 on the K side and by a
//    1/16 m-tile factor on the V side). A pair of codes costs one LOP3 (4-bit)
//    or one PRMT (8-bit), with no offset to undo. Per 64-dim group g,
//        q.k = s_g * sum_d q_d c_d + b_g * sum_d q_d
//    (q converted to fp16 with an exact per-row power-of-two prescale), and with
//    P'_g = p * s_g rounded to fp16,
//        o_d = sum_t P'_g(t) c_td + sum_t p(t) b_g(t).
//    The scale terms cost a few FMAs per key and group instead of two per
//    element; the bias terms of the scores run as one extra bf16 MMA per tile.
//  * Rows at or past seq_len in the last page are masked before they can reach
//    an accumulator (scores set to -inf by select; their V operand or V scale
//    zeroed), so stale storage may hold anything, NaN included.
#pragma once

#include "pkv_append.cuh"
#include "pkv_common.cuh"
#include "pkv_partial_cc.cuh"

namespace pkv {

// SOLO: the variant for grids of at most one CTA per SM. Such a CTA has the SM to
// itself, so it takes 8 warps (two per scheduler, so one warp's dependent chain
// hides behind the other's) when two stages per warp fit in shared memory beside a
// receive area for the push-form cluster merge, else 7 without that area (pull-form
// merge), else 6, as many stages per warp (up to 4) as fit, and up to 255 registers
// per thread.
// D is the key (and query) head dim, DV the value head dim. Names without a V
// describe the K plane, names with one the V plane. CCQ = 0 takes the tensor-core
// contraction; CCQ = 2 or 4 the CUDA-core one (pkv_partial_cc.cuh) for bf16 pages
// with up to that many query rows per KV head (NT = WQ = 1).
template <int BITS, int D, int DV, int NT, int WQ, bool SOLO, int CCQ = 0, bool BAL = false>
struct PartialCfg {
  static constexpr bool kQuant = BITS != 16;
  static constexpr int kElemBytes = kQuant ? 1 : 2;                    // tensor-map element size
  static constexpr int kRowBytes = kQuant ? D * BITS / 8 : 2 * D;      // stored bytes of one K row
  static constexpr int kRowBytesV = kQuant ? DV * BITS / 8 : 2 * DV;   // ... and of one V row
  static constexpr int kGroups = D / 64;
  static constexpr int kGroupsV = DV / 64;
  // Rows per stage: 32 for affine pages when a stage stays within ~9.5 KB, else 16.
  static constexpr int kCh =
      (kQuant && 32 * (kRowBytes + kRowBytesV) + 2 * 32 * (kGroups + kGroupsV) * 2 <= 9728) ? 32 : 16;
  static constexpr int kRB = kRowBytes >= 128 ? 128 : kRowBytes;      // bytes of one box row
  static constexpr int kRBV = kRowBytesV >= 128 ? 128 : kRowBytesV;
  static constexpr int kBoxes = kRowBytes / kRB;
  static constexpr int kBoxesV = kRowBytesV / kRBV;
  static constexpr int kBoxBytes = kCh * kRB;
  static constexpr int kBoxBytesV = kCh * kRBV;
  static constexpr int kPlaneBytes = kBoxes * kBoxBytes;
  static constexpr int kPlaneBytesV = kBoxesV * kBoxBytesV;
  static constexpr int kSbBytes = kQuant ? kCh * kGroups * 2 : 0;     // one K scale or bias plane
  static constexpr int kSbBytesV = kQuant ? kCh * kGroupsV * 2 : 0;   // one V scale or bias plane
  // stage layout: K rows, V rows, K scales, K biases, V scales, V biases
  static constexpr int kOffV = kPlaneBytes;
  static constexpr int kOffKs = kPlaneBytes + kPlaneBytesV;
  static constexpr int kOffKb = kOffKs + kSbBytes;
  static constexpr int kOffVs = kOffKb + kSbBytes;
  static constexpr int kOffVb = kOffVs + kSbBytesV;
  static constexpr int kTxBytes = kOffVb + kSbBytesV;
  static constexpr int kTmaBytes = kPlaneBytes + kPlaneBytesV;  // the part the TMA copies bring
  static constexpr int kSbCopies = (2 * kSbBytes + 2 * kSbBytesV) / 16;  // 16-byte copies of scales and biases
  static constexpr int kStageBytes = (kTxBytes + 1023) / 1024 * 1024;
  static constexpr int kBarrierBytes = SOLO ? 512 : 256;
  static constexpr int kNqp = 8 * NT;       // query rows per warp (padded)
  static constexpr int kNqAll = WQ * kNqp;  // query rows per CTA (padded)
  // Push-form cluster merge: a receive area of the CTA's own, which the other members
  // write into (their (m, l) of every row, and their o runs of this CTA's share of the
  // outputs) while this CTA may still be streaming.
  static constexpr int kRecvNeedBytes = (2 * kMaxClusterParts * kNqAll + kNqAll * DV + 4 * kMaxClusterParts) * 4;
  // CUDA-core contraction: each warp's weights of one chunk (16 rows x 4 query rows of f32)
  static constexpr int kPBufBytes = CCQ ? 8 * 256 : 0;
  // balanced schedule: the chunk-list prefix over the sequences and their lengths
  static constexpr int kBalBytes = BAL ? (2 * kMaxBalancedSeqs + 4) * 4 : 0;
  // stage ring of a CTA alone on its SM, with the receive area of the push-form cluster
  // merge (kSoloBudget) or without it (kSoloBase)
  static constexpr int kSoloBase = 227 * 1024 - kBarrierBytes - 1024 - kPBufBytes - kBalBytes;
  static constexpr int kSoloBudget = kSoloBase - (SOLO ? kRecvNeedBytes : 0);
  // A CTA of a grid of several per SM whose four warps' two stages each already take more
  // than half the SM's shared memory (16 KB stages: bf16 D=256) has its SM to itself anyway.
  static constexpr bool kLone = !SOLO && 4 * 2 * kStageBytes > 114 * 1024;
  // A seventh warp where eight with two stages each do not fit beside the receive area
  // but seven fit without it (bf16 D=256: 7 x 2 x 16 KB), for a CTA alone on its SM; the
  // CTA then merges its cluster in the pull form. The single-CTA bf16 D=256 step went
  // from 12.89 to 11.97 us, its cluster grids moved by +0.3% to -3.6%, and bf16 D=256
  // batches of several CTAs per SM (four warps before) took 4-5% less time.
  static constexpr bool kSeven = (SOLO || kLone) && WQ == 1 && CCQ == 0 && 8 * 2 * kStageBytes > kSoloBudget &&
                                 7 * 2 * kStageBytes <= kSoloBase;
  // every warp computes: 8 when two stages per warp fit a CTA alone on its SM, else 7 as
  // above, else 6 (two of the four schedulers then hold two warps), else 4; a query group
  // of 8 warps (up to 64 query rows of 256-dim heads) is the whole CTA
  // A lone CTA of two-warp query groups (bf16 D=256 with 9-16 query rows per KV head)
  // takes three page groups, six warps, beside the receive area: its batches took 16-18%
  // less time than with four warps (0.64 -> 0.76 of the measured peak).
  static constexpr bool kSixLone = kLone && WQ == 2 && CCQ == 0 && 6 * 2 * kStageBytes + kRecvNeedBytes <= kSoloBase;
  // And one of four-warp query groups (bf16 D=256 with 17-32 query rows) takes two page
  // groups, eight warps, with a ring of four stages each: its batches took a third less
  // time than with one group and a ring of eight (0.35 -> 0.53 of the measured peak).
  static constexpr bool kEightLone = kLone && WQ == 4 && CCQ == 0 && 8 * kStageBytes + kRecvNeedBytes <= kSoloBase;
  static constexpr int kWarps = WQ == 8                              ? 8
                                : kSeven && !SOLO                    ? 7
                                : kSixLone                           ? 6
                                : kEightLone                         ? 8
                                : !SOLO                              ? 4
                                : 8 * 2 * kStageBytes <= kSoloBudget ? 8
                                : kSeven                             ? 7
                                : 6 * 2 * kStageBytes <= kSoloBudget ? 6
                                                                     : 4;
  static constexpr int kThreads = kWarps * 32;
  // The warps form kWP page groups of WQ warps. A page group takes every kWP-th chunk;
  // its WQ warps read each of its chunks, each for its own 8*NT query rows.
  static constexpr int kWP = kWarps / WQ;
  static constexpr int kSoloStages = (kSeven ? kSoloBase : kSixLone ? kSoloBase - kRecvNeedBytes : kSoloBudget) /
                                     (kWarps * kStageBytes);
  // (a query group of 8 warps shares one ring of 8 or 16 stages, within 144 KB)
  static constexpr int kStagesPerWarp = WQ == 8 ? (8 * 2 * kStageBytes <= 144 * 1024 ? 2 : 1)
                                        : kEightLone ? 1
                                        : SOLO || kSeven || kSixLone ? (kSoloStages < 4 ? kSoloStages : 4)
                                                : (kStageBytes <= 9 * 1024 ? 3 : 2);
  static constexpr int kStagesPerGroup = kStagesPerWarp * WQ;  // each page group's private ring
  static constexpr int kMt = DV / 16;       // 16-dim m-tiles of O^T
  static constexpr int kKs = D / 16;        // k16 steps of Q K^T
  static constexpr int kTiles = kCh / 16;   // 16-key tiles per stage
  // Row stride (floats) of the per-page-group outputs in the combine area: padded by 4 so
  // rows stay 16-byte aligned for vector access and a warp's stores spread over the banks.
  static constexpr int kCoStride = DV + 4;
  // per-page-group states (m, l, o) for the in-CTA combine, then the CTA's own state for a cluster merge
  static constexpr int kGroupStateFloats = kNqAll * (kCoStride + 2);
  static constexpr int kCtaStateFloats = kNqAll * (DV + 2);
  static constexpr int kCombineBytes = (kWP * kGroupStateFloats + kCtaStateFloats) * 4;
  static constexpr int kRingBytes = kWarps * kStagesPerWarp * kStageBytes;
  static constexpr int kGroupBytes = kStagesPerGroup * kStageBytes;  // one page group's ring
  // When a page group's state (and the CTA's, after the last group's) fits its own ring,
  // each group writes it there as soon as its chunks are done, with no CTA barrier first.
  static constexpr bool kOwnRegions = (kGroupStateFloats + kCtaStateFloats) * 4 <= kGroupBytes;
  static constexpr int kWorkBytes = kRingBytes > kCombineBytes ? kRingBytes : kCombineBytes;
  // The receive area (after the ring) is there when the CTA is alone on its SM, or when it
  // does not cost the second CTA per SM (or the CTA already has its SM to itself).
  static constexpr int kBaseSmem = kWorkBytes + kBarrierBytes + 1024;
  static constexpr bool kPush = !BAL && !kSeven && (SOLO || kBaseSmem + kRecvNeedBytes <= 114 * 1024 ||
                                         (kBaseSmem > 114 * 1024 && kBaseSmem + kRecvNeedBytes <= 227 * 1024));
  static constexpr int kRecvBytes = kPush ? kRecvNeedBytes : 0;
  static constexpr int kDataBytes = kWorkBytes + kRecvBytes;
  static constexpr int kSmemBytes = kDataBytes + kBarrierBytes + kPBufBytes + kBalBytes + 1024;  // + alignment slack
  static constexpr float kCodeUnit = 5.9604644775390625e-8f;  // 2^-24: value of fp16 bit pattern 1

  static_assert((kRB == 128 || kRB == 64) && (kRBV == 128 || kRBV == 64), "box rows of 64 or 128 bytes");
  static_assert(kRowBytes % kRB == 0 && kRowBytesV % kRBV == 0, "whole boxes per row");
  static_assert(kWarps * kStagesPerWarp * 12 + 4 <= kBarrierBytes, "barrier area");
  static_assert(!kQuant || (D % 64 == 0 && DV % 64 == 0), "affine head dims are whole 64-dim groups");
  static_assert(DV % 64 == 0, "value head dims are whole 4-m-tile groups");
  static_assert(WQ == 1 || WQ == 2 || WQ == 4 || WQ == 8, "query groups of 1, 2, 4 or 8 warps");
  static_assert(kWarps % WQ == 0, "whole query groups");
  static_assert(kStagesPerWarp >= 2 || WQ >= 4, "at least two stages per warp (a ring of 4 or 8 for 4- or 8-warp groups)");
  static_assert(!(WQ == 8 && SOLO), "a query group of 8 warps is its CTA already");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");
  static_assert(CCQ == 0 || (BITS == 16 && D == DV && NT == 1 && WQ == 1 && kCh == 16 && kRB == 128),
                "CUDA-core contraction: bf16 pages, equal head dims, 128-byte rows, one warp per query group");
  static_assert(!CCQ || kWarps <= 8, "weight buffers of at most 8 warps");
  static_assert(!BAL || (!SOLO && CCQ == 0), "balanced schedule: grids of several CTAs per SM, tensor cores");
};

// Physical head dim held by row `half` (0: g, 1: g + 8) of O^T m-tile `mt`.
template <int BITS>
__device__ __forceinline__ int out_dim(int mt, int half, int g) {
  if constexpr (BITS == 16) {
    return 16 * mt + 8 * half + g;
  } else if constexpr (BITS == 4) {
    return 64 * (mt >> 2) + 32 * half + 4 * g + (mt & 3);
  } else {
    return 64 * (mt >> 2) + 32 * ((mt >> 1) & 1) + 16 * half + 2 * g + (mt & 1);
  }
}

// Physical head dims feeding B-fragment register `reg` (0 or 1) of k-step kk for
// the thread with tid_in_group t: (low half, high half).
template <int BITS>
__device__ __forceinline__ void q_dims(int kk, int reg, int t, int& d_lo, int& d_hi) {
  if constexpr (BITS == 16) {
    d_lo = 16 * kk + 8 * reg + 2 * t;
    d_hi = d_lo + 1;
  } else if constexpr (BITS == 4) {
    // word t of 16-byte chunk (2 grp + cc) holds dims base..base+7, nibble n = dim base+n;
    // k-step s=0 takes nibbles (0,4) and (2,6), s=1 takes (1,5) and (3,7).
    const int grp = kk >> 2, cc = (kk >> 1) & 1, s = kk & 1;
    const int base = 64 * grp + 32 * cc + 8 * t + s + 2 * reg;
    d_lo = base;
    d_hi = base + 4;
  } else {
    const int grp = kk >> 2, c = kk & 3;
    const int base = 64 * grp + 16 * c + 4 * t + reg;
    d_lo = base;
    d_hi = base + 2;
  }
}

// Loads the query values one lane needs from row `qrow` (D bf16 values) as 2 * D/16
// words of bf16 pairs, with vector loads of the contiguous runs q_dims addresses
// (zeros when !valid): bf16 pages take a word per (k-step, register); 4-bit pages 16
// bytes per 32-dim half group; 8-bit pages 8 bytes per 16-dim quarter group.
template <int BITS, int D>
__device__ __forceinline__ void q_load_words(const __nv_bfloat16* qrow, int t, bool valid, uint32_t (&w)[D / 8]) {
  if constexpr (BITS == 16) {
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {  // i = 2 kk + reg: dims 16 kk + 8 reg + 2t, +1
      w[i] = valid ? ld_nc_keep_u32(qrow + 8 * i + 2 * t) : 0u;
    }
  } else if constexpr (BITS == 4) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {  // c = 2 grp + cc: dims 32 c + 8t .. + 7
      const uint4 v = valid ? ld_nc_keep_v4(qrow + 32 * c + 8 * t) : make_uint4(0, 0, 0, 0);
      w[4 * c] = v.x;
      w[4 * c + 1] = v.y;
      w[4 * c + 2] = v.z;
      w[4 * c + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {  // c = 4 grp + quarter: dims 16 c + 4t .. + 3
      const uint2 v = valid ? ld_nc_keep_v2(qrow + 16 * c + 4 * t) : make_uint2(0, 0);
      w[2 * c] = v.x;
      w[2 * c + 1] = v.y;
    }
  }
}

// The bf16 pair (dims d_lo, d_hi of q_dims(kk, reg)) from the words of q_load_words.
template <int BITS, int W>
__device__ __forceinline__ uint32_t q_pair(const uint32_t (&w)[W], int kk, int reg) {
  if constexpr (BITS == 16) {
    return w[2 * kk + reg];
  } else if constexpr (BITS == 4) {
    // 16-byte run c = kk/2 holds dims base..base+7 as words of pairs; the lane needs
    // elements j = (kk & 1) + 2 reg and j + 4
    const int c = kk >> 1, j = (kk & 1) + 2 * reg;
    return __byte_perm(w[4 * c + (j >> 1)], w[4 * c + 2 + (j >> 1)], (j & 1) ? 0x7632 : 0x5410);
  } else {
    // 8-byte run kk holds dims base..base+3; the lane needs elements reg and reg + 2
    return __byte_perm(w[2 * kk], w[2 * kk + 1], reg ? 0x7632 : 0x5410);
  }
}

// Final output element i (bf16), to `out` and to its mirror when there is one.
__device__ __forceinline__ void write_out(const PartialParams& p, size_t i, float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  p.out[i] = b;
  if (p.out_mirror) p.out_mirror[i] = b;
}

// Final output elements i .. i+3 (i a multiple of 4), one 8-byte store each.
__device__ __forceinline__ void write_out4(const PartialParams& p, size_t i, float4 v) {
  uint2 w;
  w.x = pack_bf16x2(v.x, v.y);
  w.y = pack_bf16x2(v.z, v.w);
  *reinterpret_cast<uint2*>(p.out + i) = w;
  if (p.out_mirror) *reinterpret_cast<uint2*>(p.out_mirror + i) = w;
}

// 4-bit k-steps with odd index read their codes at bit 4 of each half (16 c); their
// B fragments carry q / 16.
template <int BITS>
__device__ __forceinline__ bool q_over16(int kk) {
  return BITS == 4 && (kk & 1);
}

// Factor that brings O^T m-tile `mt` of the V-side MMA back to code units (4-bit
// m-tiles 4g+1 and 4g+3 read their nibble at bit 4: 16 c).
template <int BITS>
__device__ __forceinline__ float v_tile_factor(int mt) {
  return (BITS == 4 && (mt & 1)) ? 1.f / 16.f : 1.f;
}

// Two consecutive bf16 values (low half first) as floats.
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

// The G bf16 group values of one row of a scale/bias plane in shared memory.
template <int G>
__device__ __forceinline__ void load_group_row(uint32_t addr, float (&v)[G]) {
  static_assert(G == 2 || G == 4, "head dims 128 or 256");
  if constexpr (G == 4) {
    uint32_t w0, w1;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(addr) : "memory");
    bf16x2_to_f32(w0, v[0], v[1]);
    bf16x2_to_f32(w1, v[2], v[3]);
  } else {
    uint32_t w0;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(addr) : "memory");
    bf16x2_to_f32(w0, v[0], v[1]);
  }
}

// HOSTIN: a host-driven step whose length, query and block tables all live in host
// memory the host wrote before the launch (no kernel writes them): they are read before
// the wait for the previous kernel on the stream, so their NVLink-C2C latency overlaps it.
// PV: 4-bit pages with at most 4 query rows per KV head (NT = WQ = 1). The 8 columns of
// the MMAs then hold the query rows twice (columns 4-7 repeat rows 0-3), so the scores
// give every weight twice, and one transposed weight fragment serves a pair of 64-dim
// groups: columns 0-3 carry the weights scaled by the even group's value scales, columns
// 4-7 by the odd group's; each group's MMAs keep the columns of their own group.
template <int BITS, int D, int DV, int NT, int WQ, bool SOLO, bool HOSTIN, int CCQ = 0, bool PV = false,
          bool BAL = false, bool PC = false>
__global__ void __maxnreg__(255)
    pkv_partial_kernel(const __grid_constant__ PartialParams p, const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v) {
  using C = PartialCfg<BITS, D, DV, NT, WQ, SOLO, CCQ, BAL>;
  static_assert(!PV || (BITS == 4 && NT == 1 && WQ == 1 && CCQ == 0 && C::kGroupsV % 2 == 0),
                "paired value groups: 4-bit pages, one warp of 8 query columns, whole group pairs");
  static_assert(!PC || (!SOLO && !BAL && CCQ == 0), "blocks smaller than a chunk: partitions, tensor cores");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kDataBytes);  // [warp][stage]
  int* stage_ok = reinterpret_cast<int*>(full_bar + C::kWarps * C::kStagesPerWarp);
  volatile int* abort_flag = stage_ok + C::kWarps * C::kStagesPerWarp;

  // slot: rank in the cluster / workspace. Under the balanced schedule (b, hk) name the
  // unit the page group is working on, which changes along its run.
  const int slot = BAL ? 0 : blockIdx.x;
  int hk = BAL ? 0 : blockIdx.y, b = BAL ? 0 : blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int qg = warp % WQ, pg = warp / WQ;  // query group, page group
  const int rbase = qg * C::kNqp;            // first query row of this warp within the CTA
  const bool leader = qg == 0;               // issues its page group's copies
  const int N = p.n_query;
  const int rep = p.nq / N;
  size_t row0 = (static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(hk) * rep) * N;
  const bool single = p.mode == kModeSingle;
  const bool in_cluster = p.mode == kModeCluster;
  // When launched as a programmatic dependent (every grid but the clusters of several
  // CTAs per SM of device-input calls), everything the previous kernel on the stream
  // writes (inputs, pools, the output) is read or written only after it has completed;
  // otherwise the wait returns at once.
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmap_k);  // kernel parameters: no dependence
    prefetch_tensormap(&tmap_v);
  }
  if constexpr (!HOSTIN) wait_for_prerequisite_grids();
  int len = BAL ? 0 : p.seq_lens[b];
  // This lane's query values, fetched now so their latency overlaps the length's (under
  // the balanced schedule, at the start of each unit of the run):
  // 2 * kKs words of bf16 pairs per n-tile, in the order q_load_words reads them.
  uint32_t qw[NT][2 * C::kKs];
  uint4 qcw[CCQ ? CCQ : 1];  // CUDA-core contraction: this lane's 8 dims of each query row
  auto load_q = [&]() {
    if constexpr (CCQ) {
      const int d0 = (lane % (D / 8)) * 8;
#pragma unroll
      for (int qi = 0; qi < CCQ; ++qi)
        qcw[qi] = qi < p.nq ? ld_nc_keep_v4(p.q + (row0 + qi) * D + d0) : make_uint4(0u, 0u, 0u, 0u);
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = PV ? g & 3 : rbase + 8 * nt + g;  // PV: columns 4-7 repeat query rows 0-3
        const __nv_bfloat16* qrow = p.q + (row0 + (r < p.nq ? r : 0)) * D;
        q_load_words<BITS, D>(qrow, t, r < p.nq, qw[nt]);
      }
    }
  };
  if constexpr (!BAL) load_q();
  // Without a window the partition (and so this warp's first 32 chunks) does not
  // depend on len: fetch their block-table entries while len is still in flight.
  int tbl_pre = 0;
  if (!BAL && p.window == 0 && leader) {
    const int pl = PC ? p.piece_log2 : 0;
    const int lq = lane >> pl, lj = lane & ((1 << pl) - 1);  // piece `lane`: its chunk, and the piece in it
    const long long r =
        static_cast<long long>(slot) * p.partition_tokens + (pg + lq * C::kWP) * C::kCh + lj * (C::kCh >> pl);
    const long long blk = r / p.block_size < p.max_blocks ? r / p.block_size : p.max_blocks - 1;
    tbl_pre = static_cast<int>(ld_nc_keep_u32(p.block_tables + static_cast<size_t>(b) * p.max_blocks + blk));
  }
  if constexpr (HOSTIN) wait_for_prerequisite_grids();  // the host inputs are in flight; the rest may depend on it
  // Fused append: the step's new K/V rows of this (sequence, KV head) are read by the
  // warp whose chunk holds them just before it issues that chunk; fetch them now.
  if (!BAL && p.k_new != nullptr) {
    const size_t nrow = (static_cast<size_t>(b) * p.num_kv_heads + hk) * N;
    const int k_lines = (N * D * 2 + 127) / 128, v_lines = (N * DV * 2 + 127) / 128;
    const int i = threadIdx.x;
    if (i < k_lines) {
      prefetch_l1(reinterpret_cast<const char*>(p.k_new + nrow * D) + 128 * i);
    } else if (i < k_lines + v_lines) {
      prefetch_l1(reinterpret_cast<const char*>(p.v_new + nrow * DV) + 128 * (i - k_lines));
    }
  }
  // Balanced schedule: every sequence's first chunk in the list of (sequence, KV head,
  // chunk), and its length, in shared memory.
  int* const bal_S = reinterpret_cast<int*>(smem + C::kDataBytes + C::kBarrierBytes + C::kPBufBytes);
  int* const bal_len = bal_S + kMaxBalancedSeqs + 1;
  if constexpr (BAL) {
    bal_scan(p.seq_lens, p.num_seqs, p.num_kv_heads, N, p.window, p.max_blocks * p.block_size, C::kCh, bal_S,
             bal_len);
    if (blockIdx.x == 0 && p.error_flag) {  // lengths the list leaves out
      for (int i = threadIdx.x; i < p.num_seqs; i += C::kThreads)
        if (bal_len[i] < N || bal_len[i] > p.max_blocks * p.block_size) atomicOr(p.error_flag, kDevErrBadSeqLen);
    }
  }
  // The stage barriers do not depend on len either: set them up while it is in flight.
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kWarps * C::kStagesPerWarp; ++s) mbar_init(smem_addr(&full_bar[s]), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // In the push form a CTA stores its cluster-merge share into the other members' shared
  // memory; that needs every member running, which this first cluster phase tells.
  if constexpr (C::kPush) {
    if (in_cluster) cluster_arrive_relaxed();
  }

  if (!BAL && (len < N || len > p.max_blocks * p.block_size)) {
    // Every CTA of this sequence sees the same length and leaves here (before any
    // cluster barrier); the CTA of partition 0 zeroes the outputs unless the merge
    // pass does.
    if (threadIdx.x == 0 && slot == 0 && p.error_flag) atomicOr(p.error_flag, kDevErrBadSeqLen);
    if (single || (in_cluster && slot == 0)) {
      for (int i = threadIdx.x; i < p.nq * DV; i += C::kThreads) write_out(p, row0 * DV + i, 0.f);
    }
    return;
  }
  // With a sliding window only rows >= len - N + 1 - window are visible to any query;
  // the partitions then start at the chunk boundary below that row, so the grid
  // tiles the visible span evenly.
  const int win_lo = p.window > 0 ? max(0, len - N + 1 - p.window) : 0;
  const int t0 = partition_base(len, N, p.window) + slot * p.partition_tokens;
  const int t_end = min(len, t0 + p.partition_tokens);
  const bool empty = !BAL && t0 >= len;
  if (empty && !in_cluster) return;  // the merge pass never reads this partition
  // first row this CTA reads: the partition start, or the chunk holding the window's lowest row
  const int t_first = max(t0, win_lo / C::kCh * C::kCh);
  const int nchunks = empty ? 0 : (t_end - t_first + C::kCh - 1) / C::kCh;  // an empty cluster member still merges

  // Balanced schedule: page group bal_v's run [x0, x1) of the chunk list.
  int bal_v = 0, x0 = 0, x1 = 0;
  if constexpr (BAL) {
    const int T = bal_S[p.num_seqs];
    const int V = static_cast<int>(gridDim.x) * C::kWP;
    bal_v = static_cast<int>(blockIdx.x) * C::kWP + pg;
    x0 = bal_run_start(bal_v, T, V);
    x1 = bal_run_start(bal_v + 1, T, V);
  }

  // O^T accumulators and softmax state.
  float o[C::kMt][NT][4];
  float m_run[NT][2], l_run[NT][2];
  float corr_v[C::kQuant ? C::kGroupsV : 1][NT][2];
  // CUDA-core contraction: per query row, this lane's 8 dims of o, the running maximum
  // and this lane's share of the normaliser.
  constexpr int kCcq = CCQ ? CCQ : 1;
  float2 cco[kCcq][4];
  float ccm[kCcq], ccl[kCcq];

  {
    // ------------------------------------------------------------------ this warp's pipeline
    // Page group pg owns chunks pg, pg + kWP, pg + 2 kWP, ... of the partition and a
    // private ring of kStagesPerGroup stages; its leader warp issues the TMA copies
    // kStagesPerGroup chunks ahead, so no group waits on another group's progress.
    const int my_chunks = BAL ? x1 - x0 : nchunks > pg ? (nchunks - pg + C::kWP - 1) / C::kWP : 0;
    uint64_t* my_full = full_bar + pg * C::kStagesPerGroup;
    int* my_ok = stage_ok + pg * C::kStagesPerGroup;
    uint8_t* my_ring = smem + pg * C::kStagesPerGroup * C::kStageBytes;
    const int32_t* table = p.block_tables + static_cast<size_t>(b) * p.max_blocks;
    const uint64_t policy = l2_evict_first_policy();
    auto chunk_row = [&](int i) { return t_first + (pg + i * C::kWP) * C::kCh; };  // first cache row of local chunk i
    // Blocks smaller than a chunk: a chunk spans nb = 2^piece_log2 blocks, and is copied
    // as nb pieces of pb rows, one per block. Pieces are numbered chunk-major (piece q is
    // piece q mod nb of local chunk q / nb); with blocks of a chunk or more, piece q is
    // chunk q.
    const int nbl = PC ? p.piece_log2 : 0, nb = 1 << nbl, pb = C::kCh >> nbl;  // PC: instantiations for such pools
    auto piece_row = [&](int q) { return chunk_row(q >> nbl) + (q & (nb - 1)) * pb; };  // its first cache row
    // TMA row coordinate of local piece q in physical block ph (the block's rows of this
    // KV head plus the piece's offset in the block), -1 for a bad block id, or -2 for a
    // piece wholly at or past the length (a chunk's first piece never is): its block may
    // not exist, and its rows are masked like any stale row, so it is not copied. Each
    // lane of the leader warp holds the coordinate of one of the next 32 pieces to
    // issue, and the raw block ids of the 32 after those (0 for pieces past the length,
    // whose table entries are not read).
    auto coord_of = [&](int ph, int q) {
      return PC && piece_row(q) >= len ? -2
             : static_cast<unsigned>(ph) < static_cast<unsigned>(p.num_blocks)
                 ? (ph * p.num_kv_heads + hk) * p.block_size + piece_row(q) % p.block_size
                 : -1;
    };
    auto stored = [&](int q) { return !PC || piece_row(q) < len; };
    // Balanced schedule: the raw block id of local piece q (of a chunk < my_chunks), with
    // its KV head and row within the block packed into *pk as hk * block_size + row %
    // block_size, and the TMA row coordinate from the two.
    auto bal_entry = [&](int q, int* pk) {
      const int x = x0 + (q >> nbl);
      const int bb = bal_seq_of(bal_S, p.num_seqs, x);
      const int n = (bal_S[bb + 1] - bal_S[bb]) / p.num_kv_heads;
      const int rel = x - bal_S[bb];
      const int h = rel / n;
      const int row = bal_first_row(bal_len[bb], N, p.window, C::kCh) + (rel - h * n) * C::kCh + (q & (nb - 1)) * pb;
      if (PC && row >= bal_len[bb]) {  // a piece past the length: not copied (pk -1)
        *pk = -1;
        return 0;
      }
      *pk = h * p.block_size + row % p.block_size;
      return static_cast<int>(__ldg(p.block_tables + static_cast<size_t>(bb) * p.max_blocks + row / p.block_size));
    };
    auto bal_coord = [&](int ph, int pk) {
      return pk < 0 ? -2
             : static_cast<unsigned>(ph) < static_cast<unsigned>(p.num_blocks) ? ph * p.num_kv_heads * p.block_size + pk
                                                                                : -1;
    };
    const int my_pieces = my_chunks << nbl;
    int crd_cur = 0, tbl_next = 0, pk_next = 0;
    if (leader) {
      if constexpr (BAL) {
        int pk0 = 0;
        const int ph0 = lane < my_pieces ? bal_entry(lane, &pk0) : 0;
        tbl_next = 32 + lane < my_pieces ? bal_entry(32 + lane, &pk_next) : 0;
        crd_cur = bal_coord(ph0, pk0);
      } else {
        const int ph0 = p.window == 0 ? tbl_pre
                        : lane < my_pieces && stored(lane) ? __ldg(table + piece_row(lane) / p.block_size)
                                                           : 0;
        tbl_next = 32 + lane < my_pieces && stored(32 + lane) ? __ldg(table + piece_row(32 + lane) / p.block_size) : 0;
        crd_cur = coord_of(ph0, lane);
      }
    }
    int issued = 0;  // chunks issued so far

    // Affine pages: this lane's share of the 16-byte copies that bring a chunk's scale and
    // bias rows, fixed for the whole loop: copy j (lane + 32 j) belongs to piece
    // sb_piece[j] of the chunk, reads that piece's plane row `row` at sb_src[j] + row *
    // sb_pitch[j] bytes and lands at sb_dst[j] within the stage (a piece of at least 8
    // rows holds whole 16-byte copies).
    constexpr int kSbPerLane = C::kQuant ? (C::kSbCopies + 31) / 32 : 1;
    const char* sb_src[kSbPerLane];
    int sb_pitch[kSbPerLane], sb_dst[kSbPerLane];  // sb_dst: the piece in bits 16 and up
    if constexpr (C::kQuant) {
      constexpr int nk = C::kSbBytes / 16, nv = C::kSbBytesV / 16;
#pragma unroll
      for (int j = 0; j < kSbPerLane; ++j) {
        const int c = 32 * j + lane;
        const int cc = c < C::kSbCopies ? c : 0;
        const int plane = cc < 2 * nk ? cc / nk : 2 + (cc - 2 * nk) / nv;
        const int k = cc < 2 * nk ? cc % nk : (cc - 2 * nk) % nv;
        const __nv_bfloat16* src = plane == 0   ? p.k_scales
                                   : plane == 1 ? p.k_biases
                                   : plane == 2 ? p.v_scales
                                                : p.v_biases;
        sb_pitch[j] = 2 * (plane < 2 ? C::kGroups : C::kGroupsV);
        const int piece = 16 * k / (sb_pitch[j] * pb);
        sb_src[j] = reinterpret_cast<const char*>(src) + 16 * k - piece * pb * sb_pitch[j];
        sb_dst[j] = ((plane == 0 ? C::kOffKs : plane == 1 ? C::kOffKb : plane == 2 ? C::kOffVs : C::kOffVb) + 16 * k) |
                    (piece << 16);
      }
    }

    // Issues the next chunk into stage `is` (the one just consumed: with one stage per
    // chunk in flight, chunk i always lands in stage i mod kStagesPerGroup).
    auto issue_next = [&](int is) {  // the leader warp, warp-uniform
      if (issued >= my_chunks) return;
      const int ip = issued << nbl;  // the chunk's first piece
      if (ip > 0 && (ip & 31) == 0) {
        const int k = ip + 32 + lane;
        if constexpr (BAL) {
          crd_cur = bal_coord(tbl_next, pk_next);
          tbl_next = k < my_pieces ? bal_entry(k, &pk_next) : 0;
        } else {
          crd_cur = coord_of(tbl_next, ip + lane);
          tbl_next = k < my_pieces && stored(k) ? __ldg(table + piece_row(k) / p.block_size) : 0;
        }
      }
      // row: the first piece's coordinate, -1 when a stored piece has a bad block id
      int row = __shfl_sync(0xffffffffu, crd_cur, ip & 31);
      int pieces_in = 1;  // pieces copied
      if (nbl > 0) {
        const int mine = __shfl_sync(0xffffffffu, crd_cur, (ip + (lane & (nb - 1))) & 31);
        if (!__all_sync(0xffffffffu, mine >= 0 || mine == -2)) row = -1;
        pieces_in = __popc(__ballot_sync(0xffffffffu, lane < nb && mine >= 0));
      }
      if (!BAL && p.k_new != nullptr) {
        // Fused append: the step's new rows len-N .. len-1 that fall in this chunk are
        // written into its page first (the warp writes, fences its generic-proxy stores
        // against the async proxy, then lane 0 copies the chunk). Chunks lie inside one
        // partition and one block, so no other CTA or warp reads these rows.
        const int cr = chunk_row(issued);
        const int a0 = max(len - N, cr), a1 = min(len, cr + C::kCh);
        if (a0 < a1 && row >= 0) {
          for (int tr = a0; tr < a1; ++tr) {
            const size_t src = (static_cast<size_t>(b) * p.num_kv_heads + hk) * N + (tr - (len - N));
            append_row<BITS, D, DV>(p.k_new + src * D, p.v_new + src * DV, p.app, static_cast<size_t>(row) + (tr - cr),
                                    lane);
          }
          fence_proxy_async_global();
          __syncwarp();
        }
      }
      const uint32_t fb = smem_addr(&my_full[is]);
      const uint32_t st = smem_addr(my_ring + is * C::kStageBytes);
      if constexpr (C::kQuant) {
        // The chunk's scale and bias rows: 16-byte cp.async copies spread over the lanes,
        // which keeps the TMA unit to two copies per stage. Each lane makes the stage's
        // barrier wait for its copies before lane 0 arrives, so the phase cannot complete
        // without them.
        if (row >= 0) {
#pragma unroll
          for (int j = 0; j < kSbPerLane; ++j) {
            const int prow = nbl > 0 ? __shfl_sync(0xffffffffu, crd_cur, (ip + (sb_dst[j] >> 16)) & 31) : row;
            if (32 * j + lane < C::kSbCopies && prow >= 0)
              cp_async_16(st + (PC ? sb_dst[j] & 0xFFFF : sb_dst[j]), sb_src[j] + static_cast<size_t>(prow) * sb_pitch[j],
                          policy);
          }
          cp_async_mbar_arrive(fb);
        }
        __syncwarp();
      }
      if (nbl > 0 && row >= 0) {
        // one copy per piece and segment: the piece's rows land at their place in each
        // segment of the chunk (a multiple of 8 rows: whole swizzle atoms)
        if (lane == 0) {
          my_ok[is] = 1;
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(fb, pieces_in * (C::kTmaBytes >> nbl));
        }
        for (int j = 0; j < nb; ++j) {
          const int prow = __shfl_sync(0xffffffffu, crd_cur, (ip + j) & 31);
          if (lane == 0 && prow >= 0) {
#pragma unroll
            for (int sg = 0; sg < C::kBoxes; ++sg)
              tma_load_3d(st + (sg * C::kCh + j * pb) * C::kRB, &tmap_k, 0, prow, sg, fb, policy);
#pragma unroll
            for (int sg = 0; sg < C::kBoxesV; ++sg)
              tma_load_3d(st + C::kOffV + (sg * C::kCh + j * pb) * C::kRBV, &tmap_v, 0, prow, sg, fb, policy);
          }
        }
      } else if (lane == 0) {
        my_ok[is] = row >= 0 ? 1 : 0;
        if (row >= 0) {
          fence_proxy_async_smem();  // this warp's reads of the stage precede the copies into it
          mbar_arrive_expect_tx(fb, C::kTmaBytes);
          tma_load_3d(st, &tmap_k, 0, row, 0, fb, policy);  // all kBoxes segments of the K rows
          tma_load_3d(st + C::kOffV, &tmap_v, 0, row, 0, fb, policy);
        } else {
          if (p.error_flag) atomicOr(p.error_flag, kDevErrBadBlock);
          mbar_arrive(fb);
        }
      }
      ++issued;
    };

#pragma unroll 1
    for (int s = 0; s < C::kStagesPerGroup; ++s)
      if (leader) issue_next(s);

    int done = 0;             // local chunks consumed
    int cs = 0;               // its stage: done mod kStagesPerGroup
    uint32_t cs_parity = 0;   // the phase it waits for: (done / kStagesPerGroup) & 1
    int seg_end = my_chunks;  // local index past the current unit's chunks
    int seg_start = 0, seg_row = 0;  // balanced: local index and cache row of the unit's first chunk in the run
    // The units of this page group's run, one at a time: one unit (its partition),
    // except under the balanced schedule. The copies run on across units; at each
    // unit's start the warp loads that unit's query rows, and at its end it writes the
    // unit's state for this run to the workspace.
#pragma unroll 1
    for (;;) {
    if constexpr (BAL) {
      if (done >= my_chunks) break;
      const int x = x0 + done;
      b = bal_seq_of(bal_S, p.num_seqs, x);
      const int n = (bal_S[b + 1] - bal_S[b]) / p.num_kv_heads;
      const int rel = x - bal_S[b];
      hk = rel / n;
      const int off = rel - hk * n;
      len = bal_len[b];
      row0 = (static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(hk) * rep) * N;
      seg_start = done;
      seg_end = min(my_chunks, done + n - off);
      seg_row = bal_first_row(len, N, p.window, C::kCh) + off * C::kCh;
      load_q();
    }

    // B fragments of Q^T for every k-step, rows r = 8*nt + g of this KV head: bf16 as
    // stored for bf16 pages; for affine pages fp16, after an exact power-of-two
    // prescale per row that puts the row's largest |q| in [2^14, 2^15).
    uint32_t qf[C::kKs][NT][2];
    float colscale[NT][2];  // factor from accumulator to base-2 score, per query column 2t, 2t+1
    // affine: B fragment (k 0-7) of the K-bias MMA, per n-tile (k 8-15 are zero)
    uint32_t qsb[C::kQuant ? NT : 1];
    float2 ccq[kCcq][4];  // CUDA-core contraction: q as f32 pairs
    if constexpr (CCQ) {
#pragma unroll
      for (int qi = 0; qi < CCQ; ++qi) {
        ccq[qi][0] = bf16x2_pair(qcw[qi].x);
        ccq[qi][1] = bf16x2_pair(qcw[qi].y);
        ccq[qi][2] = bf16x2_pair(qcw[qi].z);
        ccq[qi][3] = bf16x2_pair(qcw[qi].w);
        ccm[qi] = -INFINITY;
        ccl[qi] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) cco[qi][i] = make_float2(0.f, 0.f);
      }
    } else {
      float qsum[C::kQuant ? C::kGroups : 1][NT][2];  // affine: 2^-24 * sum of prescaled q over each group
      float qv[C::kKs][NT][4];
#pragma unroll
      for (int kk = 0; kk < C::kKs; ++kk)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int reg = 0; reg < 2; ++reg)
            bf16x2_to_f32(q_pair<BITS>(qw[nt], kk, reg), qv[kk][nt][2 * reg], qv[kk][nt][2 * reg + 1]);
      if constexpr (!C::kQuant) {
#pragma unroll
        for (int kk = 0; kk < C::kKs; ++kk)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int reg = 0; reg < 2; ++reg)
              qf[kk][nt][reg] = pack_bf16x2(qv[kk][nt][2 * reg], qv[kk][nt][2 * reg + 1]);  // exact
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) colscale[nt][0] = colscale[nt][1] = p.score_scale;
      } else {
        int kexp[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float mx = 0.f;
#pragma unroll
          for (int kk = 0; kk < C::kKs; ++kk)
#pragma unroll
            for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fabsf(qv[kk][nt][i]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));  // the row's max over its 4 lanes
          const int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFF) - 127;
          kexp[nt] = mx > 0.f ? min(max(14 - e, -100), 126) : 0;  // |q| below 2^114 is assumed
          const float up = __uint_as_float(static_cast<uint32_t>(127 + kexp[nt]) << 23);  // 2^kexp
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < C::kKs; ++kk) {
            uint32_t fr[2];
#pragma unroll
            for (int reg = 0; reg < 2; ++reg)
              fr[reg] = pack_f16x2(qv[kk][nt][2 * reg] * up, qv[kk][nt][2 * reg + 1] * up);
            // Per-group sums of the prescaled q (columns 2t, 2t+1), through the MMA path.
            mma_f16(acc, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, fr[0], fr[1]);
            if ((kk & 3) == 3) {
              qsum[kk >> 2][nt][0] = acc[0] * C::kCodeUnit;
              qsum[kk >> 2][nt][1] = acc[1] * C::kCodeUnit;
              acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            }
            const float f = q_over16<BITS>(kk) ? up * (1.f / 16.f) : up;
#pragma unroll
            for (int reg = 0; reg < 2; ++reg)
              qf[kk][nt][reg] = pack_f16x2(qv[kk][nt][2 * reg] * f, qv[kk][nt][2 * reg + 1] * f);
          }
        }
        // Column c = 2t + e2 of n-tile nt is query row 8 nt + 2t + e2, prescaled by the
        // lanes whose g equals 2t + e2. Codes are counted in units of 2^-24.
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int k = __shfl_sync(0xffffffffu, kexp[nt], (2 * t + e2) * 4);
            colscale[nt][e2] = p.score_scale * __uint_as_float(static_cast<uint32_t>(127 + 24 - k) << 23);
          }
        // The bias part of the scores, sum_g b_g * sum_{d in g} q_d, runs as one bf16 MMA per
        // 16-key tile: A holds each key's G biases twice (k slots 0..G-1 and G..2G-1), B
        // holds query column g's group sums split into bf16 high parts (slots 0..G-1) and
        // the bf16 rounding of the remainders (slots G..2G-1), so the product keeps about
        // 16 significant bits of each sum. The lane with t = g/2 holds column g's sums.
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float cq[C::kGroups];
#pragma unroll
          for (int j = 0; j < C::kGroups; ++j) {
            const float v0 = __shfl_sync(0xffffffffu, qsum[j][nt][0], g >> 1);
            const float v1 = __shfl_sync(0xffffffffu, qsum[j][nt][1], g >> 1);
            cq[j] = (g & 1) ? v1 : v0;
          }
          float slot_val[2] = {0.f, 0.f};
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int slot = 2 * t + e;
#pragma unroll
            for (int j = 0; j < C::kGroups; ++j) {
              const float hi = __bfloat162float(__float2bfloat16_rn(cq[j]));
              const float lo = __bfloat162float(__float2bfloat16_rn(cq[j] - hi));
              slot_val[e] = slot == j ? hi : slot == C::kGroups + j ? lo : slot_val[e];
            }
          }
          qsb[nt] = pack_bf16x2(slot_val[0], slot_val[1]);  // exact: both are bf16 values
        }
      }
    }

#pragma unroll
    for (int mt = 0; mt < C::kMt; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        m_run[nt][e2] = -INFINITY;
        l_run[nt][e2] = 0.f;
#pragma unroll
        for (int grp = 0; grp < (C::kQuant ? C::kGroupsV : 1); ++grp) corr_v[grp][nt][e2] = 0.f;
      }
    }

    const int vis_base = len - N + 1;  // query row qi sees keys < vis_base + qi
    const int win = p.window;          // ... and, when win > 0, keys >= vis_base + qi - win
    // ldmatrix row/chunk of this lane: non-transposed (keys on M) and transposed (keys on K).
    const int lrow_n = (lane & 7) + ((lane >> 3) & 1) * 8, lch_n = lane >> 4;
    const int lrow_t = (lane & 7) + (lane >> 4) * 8, lch_t = (lane >> 3) & 1;
    // 4-bit pages: this lane's ldmatrix offsets within the K and V planes of a stage, per
    // 64-dim group, for the first 16-key tile (tile t adds 16 rows: the swizzle pattern
    // repeats every 8 rows), fixed for the whole loop.
    int k4ofs[BITS == 4 ? C::kGroups : 1], v4ofs[BITS == 4 ? C::kGroupsV : 1];
    if constexpr (BITS == 4) {
#pragma unroll
      for (int grp = 0; grp < C::kGroups; ++grp) k4ofs[grp] = swizzled<C::kRB>(0u, lrow_n, 2 * grp + lch_n);
#pragma unroll
      for (int grp = 0; grp < C::kGroupsV; ++grp) v4ofs[grp] = swizzled<C::kRBV>(0u, lrow_t, 2 * grp + lch_t);
    }

    // The tensor-core contraction of one staged chunk, in three parts. score_chunk: the
    // scores (keys on rows, base 2), the causal tail / window mask and the online-softmax
    // update of (m_run, l_run), giving the chunk's weights pr and, where a running maximum
    // grew, the factors corr (returns whether any did, warp-uniform). rescale: applies corr
    // to the value accumulators. value_chunk: O^T += V^T P^T over the chunk's value rows.
    auto score_chunk = [&](uint32_t kpl, uint32_t sbq, int kbase, bool full_vis, float (&pr)[C::kTiles][NT][4],
                           float (&corr)[NT][2]) -> bool {
      // ---- scores x = (K q) * scale * log2(e), keys on rows
      float x[C::kTiles][NT][4];
#pragma unroll
      for (int tile = 0; tile < C::kTiles; ++tile) {
        float sacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
        const int lrow = tile * 16 + lrow_n;
        if constexpr (BITS == 16) {
          // A CTA alone on its SM is bound by latency: two accumulators (even and odd
          // k-steps) halve its dependent MMA chain. Elsewhere one chain costs fewer
          // instructions.
          constexpr int kChains = SOLO ? 2 : 1;
          float sacc2[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc2[nt][e] = 0.f;
#pragma unroll
          for (int kk = 0; kk < C::kKs; ++kk) {
            uint32_t a[4];
            ldsm_x4(swizzled<C::kRB>(kpl + (kk >> 2) * C::kBoxBytes, lrow, (kk & 3) * 2 + lch_n), a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_bf16((kChains == 2 && (kk & 1)) ? sacc2[nt] : sacc[nt], a[0], a[1], a[2], a[3], qf[kk][nt][0],
                       qf[kk][nt][1]);
          }
          if constexpr (kChains == 2) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) sacc[nt][e] += sacc2[nt][e];
          }
        } else {
          // scales of keys g and g + 8 of this tile, all groups
          float ks0[C::kGroups], ks1[C::kGroups];
          load_group_row<C::kGroups>(sbq + (tile * 16 + g) * C::kGroups * 2, ks0);
          load_group_row<C::kGroups>(sbq + (tile * 16 + g + 8) * C::kGroups * 2, ks1);
          {
            // bias MMA: this lane's A words are the biases of k slots 2t, 2t+1 (groups
            // 2t mod G, 2t mod G + 1) of keys g and g + 8
            uint32_t ba0 = 0u, ba1 = 0u;
            const uint32_t kb = kpl + C::kOffKb + (tile * 16 + g) * C::kGroups * 2;
            if (C::kGroups == 4 || t < 2) {
              const uint32_t off = C::kGroups == 4 ? (t & 1) * 4 : 0;
              ba0 = ld_shared_u32(kb + off);
              ba1 = ld_shared_u32(kb + 8 * C::kGroups * 2 + off);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16(sacc[nt], ba0, ba1, 0u, 0u, qsb[nt], 0u);
          }
#pragma unroll
          for (int grp = 0; grp < C::kGroups; ++grp) {
            float sg[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) sg[nt][e] = 0.f;
            if constexpr (BITS == 4) {
              // words t of chunks 2 grp, 2 grp + 1 for rows g, g + 8
              uint32_t xk[4];
              ldsm_x4(kpl + k4ofs[grp] + tile * 16 * C::kRB, xk);  // rows g, g + 8 of the tile
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const uint32_t xg = xk[2 * cc], x8 = xk[2 * cc + 1];
                const uint32_t xg8 = xg >> 8, x88 = x8 >> 8;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  const int kk = 4 * grp + 2 * cc;
                  mma_f16(sg[nt], xg & 0x000F000Fu, x8 & 0x000F000Fu, xg8 & 0x000F000Fu, x88 & 0x000F000Fu,
                          qf[kk][nt][0], qf[kk][nt][1]);
                  mma_f16(sg[nt], xg & 0x00F000F0u, x8 & 0x00F000F0u, xg8 & 0x00F000F0u, x88 & 0x00F000F0u,
                          qf[kk + 1][nt][0], qf[kk + 1][nt][1]);
                }
              }
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t xk[4];
                ldsm_x4(swizzled<C::kRB>(kpl + (grp >> 1) * C::kBoxBytes, lrow, (grp & 1) * 4 + 2 * h + lch_n), xk);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                  const int kk = 4 * grp + 2 * h + cc;
                  const uint32_t xg = xk[2 * cc], x8 = xk[2 * cc + 1];
                  // bytes (0, 2) and (1, 3) of a word: dims (4t, 4t+2) and (4t+1, 4t+3)
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt)
                    mma_f16(sg[nt], __byte_perm(xg, 0u, 0x4240), __byte_perm(x8, 0u, 0x4240),
                            __byte_perm(xg, 0u, 0x4341), __byte_perm(x8, 0u, 0x4341), qf[kk][nt][0], qf[kk][nt][1]);
                }
              }
            }
            // fold the scale of group grp for keys g and g + 8 of this tile
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              sacc[nt][0] = fmaf(ks0[grp], sg[nt][0], sacc[nt][0]);
              sacc[nt][1] = fmaf(ks0[grp], sg[nt][1], sacc[nt][1]);
              sacc[nt][2] = fmaf(ks1[grp], sg[nt][2], sacc[nt][2]);
              sacc[nt][3] = fmaf(ks1[grp], sg[nt][3], sacc[nt][3]);
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) x[tile][nt][e] = sacc[nt][e] * colscale[nt][e & 1];
      }


      // ---- causal tail and stale rows
      if (!full_vis) {
#pragma unroll
        for (int tile = 0; tile < C::kTiles; ++tile)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = kbase + tile * 16 + g + 8 * (e >> 1);
              const int qi = (PV ? (2 * t + (e & 1)) & 3 : rbase + 8 * nt + 2 * t + (e & 1)) % N;
              const bool vis = key < vis_base + qi && (win == 0 || key >= vis_base + qi - win);
              x[tile][nt][e] = vis ? x[tile][nt][e] : -INFINITY;
            }
      }

      // ---- online softmax (base 2)
      bool grew = false;
      // This lane's maxima of the chunk. When no lane's exceeds the running maximum, the
      // chunk's maximum does not either: the running maximum stays and nothing is
      // rescaled, which is what the general path below computes too, without its
      // cross-lane reduction (so the results are the same bit for bit).
      float lmx[NT][2];
      bool below = true;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          float mx = -INFINITY;
#pragma unroll
          for (int tile = 0; tile < C::kTiles; ++tile) mx = fmaxf(mx, fmaxf(x[tile][nt][e2], x[tile][nt][e2 + 2]));
          lmx[nt][e2] = mx;
          below &= mx <= m_run[nt][e2];
        }
      if (__all_sync(0xffffffffu, below)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const float muse = m_run[nt][e2] == -INFINITY ? 0.f : m_run[nt][e2];
            float ls = 0.f;
#pragma unroll
            for (int tile = 0; tile < C::kTiles; ++tile) {
              pr[tile][nt][e2] = fast_exp2(x[tile][nt][e2] - muse);
              pr[tile][nt][e2 + 2] = fast_exp2(x[tile][nt][e2 + 2] - muse);
              ls += pr[tile][nt][e2] + pr[tile][nt][e2 + 2];
            }
            l_run[nt][e2] += ls;
          }
      } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            float mx = lmx[nt][e2];
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mnew = fmaxf(m_run[nt][e2], mx);
            const float muse = mnew == -INFINITY ? 0.f : mnew;
            const float c = fast_exp2(m_run[nt][e2] - muse);
            m_run[nt][e2] = mnew;
            float ls = 0.f;
#pragma unroll
            for (int tile = 0; tile < C::kTiles; ++tile) {
              pr[tile][nt][e2] = fast_exp2(x[tile][nt][e2] - muse);
              pr[tile][nt][e2 + 2] = fast_exp2(x[tile][nt][e2 + 2] - muse);
              ls += pr[tile][nt][e2] + pr[tile][nt][e2 + 2];
            }
            l_run[nt][e2] = fmaf(l_run[nt][e2], c, ls);
            corr[nt][e2] = c;
            grew |= c != 1.f;
          }
        }
        grew = __any_sync(0xffffffffu, grew);
      }
      return grew;

    };
    auto rescale = [&](const float (&corr)[NT][2]) {
#pragma unroll
      for (int mt = 0; mt < C::kMt; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[mt][nt][e] *= corr[nt][e & 1];
      if constexpr (C::kQuant) {
#pragma unroll
        for (int grp = 0; grp < C::kGroupsV; ++grp)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) corr_v[grp][nt][e2] *= corr[nt][e2];
      }
    };
    auto value_chunk = [&](uint32_t kpl, uint32_t vpl, int kbase, bool stale, const float (&pr)[C::kTiles][NT][4]) {
      // ---- O^T += V^T P^T
#pragma unroll
      for (int tile = 0; tile < C::kTiles; ++tile) {
        const int lrow = tile * 16 + lrow_t;
        if constexpr (BITS == 16) {
          uint32_t pb[NT][2];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            pb[nt][0] = movmatrix_trans(pack_bf16x2(pr[tile][nt][0], pr[tile][nt][1]));
            pb[nt][1] = movmatrix_trans(pack_bf16x2(pr[tile][nt][2], pr[tile][nt][3]));
          }
          uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
          if (stale) {
            const int k0 = kbase + tile * 16 + 2 * t;
            m01 = (k0 < len ? 0x0000ffffu : 0u) | (k0 + 1 < len ? 0xffff0000u : 0u);
            m23 = (k0 + 8 < len ? 0x0000ffffu : 0u) | (k0 + 9 < len ? 0xffff0000u : 0u);
          }
#pragma unroll
          for (int mt = 0; mt < C::kMt; ++mt) {
            uint32_t a[4];
            ldsm_x4_t(swizzled<C::kRBV>(vpl + (mt >> 2) * C::kBoxBytesV, lrow, (mt & 3) * 2 + lch_t), a);
            a[0] &= m01;
            a[1] &= m01;
            a[2] &= m23;
            a[3] &= m23;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16(o[mt][nt], a[0], a[1], a[2], a[3], pb[nt][0], pb[nt][1]);
          }
        } else {
          const int r_a = tile * 16 + g, r_b = r_a + 8;
          float vs0[C::kGroupsV], vs1[C::kGroupsV], vb0[C::kGroupsV], vb1[C::kGroupsV];
          load_group_row<C::kGroupsV>(kpl + C::kOffVs + r_a * C::kGroupsV * 2, vs0);
          load_group_row<C::kGroupsV>(kpl + C::kOffVs + r_b * C::kGroupsV * 2, vs1);
          load_group_row<C::kGroupsV>(kpl + C::kOffVb + r_a * C::kGroupsV * 2, vb0);
          load_group_row<C::kGroupsV>(kpl + C::kOffVb + r_b * C::kGroupsV * 2, vb1);
          if (stale) {  // rows at or past len may hold anything: keep them out of P' and the bias sums
            const bool va = kbase + r_a < len, vb = kbase + r_b < len;
#pragma unroll
            for (int grp = 0; grp < C::kGroupsV; ++grp) {
              vs0[grp] = va ? vs0[grp] : 0.f;
              vb0[grp] = va ? vb0[grp] : 0.f;
              vs1[grp] = vb ? vs1[grp] : 0.f;
              vb1[grp] = vb ? vb1[grp] : 0.f;
            }
          }
          if constexpr (PV) {
            // One weight fragment per group pair: columns 0-3 (lanes with t < 2) scaled by
            // the even group's value scales, columns 4-7 (t >= 2) by the odd group's; each
            // lane also sums the biases of its own group of the pair.
            const int odd = t >> 1;
#pragma unroll
            for (int pp = 0; pp < C::kGroupsV / 2; ++pp) {
              const float sa = odd ? vs0[2 * pp + 1] : vs0[2 * pp], sb = odd ? vs1[2 * pp + 1] : vs1[2 * pp];
              const float ba = odd ? vb0[2 * pp + 1] : vb0[2 * pp], bb = odd ? vb1[2 * pp + 1] : vb1[2 * pp];
              const uint32_t pb0 = movmatrix_trans(pack_f16x2(pr[tile][0][0] * sa, pr[tile][0][1] * sa));
              const uint32_t pb1 = movmatrix_trans(pack_f16x2(pr[tile][0][2] * sb, pr[tile][0][3] * sb));
              corr_v[pp][0][0] = fmaf(pr[tile][0][0], ba, fmaf(pr[tile][0][2], bb, corr_v[pp][0][0]));
              corr_v[pp][0][1] = fmaf(pr[tile][0][1], ba, fmaf(pr[tile][0][3], bb, corr_v[pp][0][1]));
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int grp = 2 * pp + h;
                uint32_t y[4];
                ldsm_x4_t(vpl + v4ofs[grp] + tile * 16 * C::kRBV, y);
                uint32_t y8[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) y8[i] = y[i] >> 8;
                mma_f16(o[4 * grp + 0][0], y[0] & 0x000F000Fu, y[1] & 0x000F000Fu, y[2] & 0x000F000Fu,
                        y[3] & 0x000F000Fu, pb0, pb1);
                mma_f16(o[4 * grp + 1][0], y[0] & 0x00F000F0u, y[1] & 0x00F000F0u, y[2] & 0x00F000F0u,
                        y[3] & 0x00F000F0u, pb0, pb1);
                mma_f16(o[4 * grp + 2][0], y8[0] & 0x000F000Fu, y8[1] & 0x000F000Fu, y8[2] & 0x000F000Fu,
                        y8[3] & 0x000F000Fu, pb0, pb1);
                mma_f16(o[4 * grp + 3][0], y8[0] & 0x00F000F0u, y8[1] & 0x00F000F0u, y8[2] & 0x00F000F0u,
                        y8[3] & 0x00F000F0u, pb0, pb1);
              }
            }
          } else {
#pragma unroll
          for (int grp = 0; grp < C::kGroupsV; ++grp) {
            uint32_t pb[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              pb[nt][0] = movmatrix_trans(pack_f16x2(pr[tile][nt][0] * vs0[grp], pr[tile][nt][1] * vs0[grp]));
              pb[nt][1] = movmatrix_trans(pack_f16x2(pr[tile][nt][2] * vs1[grp], pr[tile][nt][3] * vs1[grp]));
              corr_v[grp][nt][0] = fmaf(pr[tile][nt][0], vb0[grp], fmaf(pr[tile][nt][2], vb1[grp], corr_v[grp][nt][0]));
              corr_v[grp][nt][1] = fmaf(pr[tile][nt][1], vb0[grp], fmaf(pr[tile][nt][3], vb1[grp], corr_v[grp][nt][1]));
            }
            if constexpr (BITS == 4) {
              // y: unit g (dims 4g..4g+3) of keys 2t (low half) and 2t+1 (high half),
              // chunks 2 grp / 2 grp + 1, keys 0-7 / 8-15 of the tile
              uint32_t y[4];
              ldsm_x4_t(vpl + v4ofs[grp] + tile * 16 * C::kRBV, y);
              uint32_t y8[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) y8[i] = y[i] >> 8;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                mma_f16(o[4 * grp + 0][nt], y[0] & 0x000F000Fu, y[1] & 0x000F000Fu, y[2] & 0x000F000Fu,
                        y[3] & 0x000F000Fu, pb[nt][0], pb[nt][1]);
                mma_f16(o[4 * grp + 1][nt], y[0] & 0x00F000F0u, y[1] & 0x00F000F0u, y[2] & 0x00F000F0u,
                        y[3] & 0x00F000F0u, pb[nt][0], pb[nt][1]);
                mma_f16(o[4 * grp + 2][nt], y8[0] & 0x000F000Fu, y8[1] & 0x000F000Fu, y8[2] & 0x000F000Fu,
                        y8[3] & 0x000F000Fu, pb[nt][0], pb[nt][1]);
                mma_f16(o[4 * grp + 3][nt], y8[0] & 0x00F000F0u, y8[1] & 0x00F000F0u, y8[2] & 0x00F000F0u,
                        y8[3] & 0x00F000F0u, pb[nt][0], pb[nt][1]);
              }
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t y[4];
                ldsm_x4_t(swizzled<C::kRBV>(vpl + (grp >> 1) * C::kBoxBytesV, lrow, (grp & 1) * 4 + 2 * h + lch_t), y);
                // byte 0 / byte 2 of y: dim 2g of keys 2t / 2t+1; bytes 1 / 3: dim 2g + 1
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  mma_f16(o[4 * grp + 2 * h][nt], __byte_perm(y[0], 0u, 0x4240), __byte_perm(y[1], 0u, 0x4240),
                          __byte_perm(y[2], 0u, 0x4240), __byte_perm(y[3], 0u, 0x4240), pb[nt][0], pb[nt][1]);
                  mma_f16(o[4 * grp + 2 * h + 1][nt], __byte_perm(y[0], 0u, 0x4341), __byte_perm(y[1], 0u, 0x4341),
                          __byte_perm(y[2], 0u, 0x4341), __byte_perm(y[3], 0u, 0x4341), pb[nt][0], pb[nt][1]);
                }
              }
            }
          }
          }  // unpaired groups
        }
      }
    };

    for (; done < seg_end; ++done, cs_parity ^= (cs == C::kStagesPerGroup - 1), cs = cs == C::kStagesPerGroup - 1 ? 0 : cs + 1) {
      const bool landed = mbar_wait_warp(smem_addr(&my_full[cs]), cs_parity, abort_flag, p.error_flag, p.wait_limit_ns);
      if (landed && my_ok[cs]) {
        uint8_t* stage = my_ring + cs * C::kStageBytes;
        const uint32_t kpl = smem_addr(stage);
        const uint32_t vpl = kpl + C::kOffV;
        const uint32_t sbq = kpl + C::kOffKs;  // scale/bias planes (affine pages)
        const int kbase = BAL ? seg_row + (done - seg_start) * C::kCh : chunk_row(done);
        const bool full_vis = kbase + C::kCh <= vis_base && (win == 0 || kbase >= vis_base + N - 1 - win);
        const bool stale = kbase + C::kCh > len;
        if constexpr (CCQ) {
          float* pbuf = reinterpret_cast<float*>(smem + C::kDataBytes + C::kBarrierBytes) + warp * 64;
          cc_chunk<D, CCQ>(kpl, vpl, pbuf, ccq, cco, ccm, ccl, lane, kbase, len, vis_base, win, N, full_vis, stale,
                           p.score_scale);
        } else {
        float pr[C::kTiles][NT][4];
        float corr[NT][2];
        if (score_chunk(kpl, sbq, kbase, full_vis, pr, corr)) rescale(corr);
        value_chunk(kpl, vpl, kbase, stale, pr);
        }  // tensor-core contraction
      }
      if constexpr (WQ == 1) {
        if (!landed) break;
        __syncwarp();  // every lane is done with the stage before it is refilled
        issue_next(cs);
      } else {
        // every warp of the group is done with the stage; one give-up decision for all
        if (group_barrier_any(1 + pg, WQ * 32, !landed)) break;
        if (leader) issue_next(cs);
      }
    }
    if (leader && done < seg_end && done < issued && lane == 0) {
      // Aborted: let this group's copies still in flight land before the ring is reused.
      for (int c = done; c < issued; ++c) {
        const uint32_t bar = smem_addr(&my_full[c % C::kStagesPerGroup]);
        const unsigned long long start = global_timer_ns();
        while (!mbar_try_wait(bar, (c / C::kStagesPerGroup) & 1) && global_timer_ns() - start < kWaitLimitNs) {
        }
      }
    }

    if constexpr (CCQ) {
      // ---- per-warp totals: the normaliser over all lanes, o over the lanes that hold
      // the same dims of other rows
      using S = CcShape<D, CCQ>;
#pragma unroll
      for (int qi = 0; qi < CCQ; ++qi) {
        float l = ccl[qi];
#pragma unroll
        for (int delta = 1; delta < 32; delta <<= 1) l += __shfl_xor_sync(0xffffffffu, l, delta);
        ccl[qi] = l;
#pragma unroll
        for (int delta = S::kLanesPerRow; delta < 32; delta <<= 1)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            cco[qi][i].x += __shfl_xor_sync(0xffffffffu, cco[qi][i].x, delta);
            cco[qi][i].y += __shfl_xor_sync(0xffffffffu, cco[qi][i].y, delta);
          }
      }
    } else {
    // ---- per-warp totals: normaliser and value corrections summed over the 8 key lanes
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        float l = l_run[nt][e2];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        l_run[nt][e2] = l;
        if constexpr (C::kQuant) {
#pragma unroll
          for (int grp = 0; grp < C::kGroupsV; ++grp) {
            float cv = corr_v[grp][nt][e2];
            cv += __shfl_xor_sync(0xffffffffu, cv, 4);
            cv += __shfl_xor_sync(0xffffffffu, cv, 8);
            cv += __shfl_xor_sync(0xffffffffu, cv, 16);
            corr_v[grp][nt][e2] = cv;
          }
        }
      }
    }
    if constexpr (C::kQuant) {
#pragma unroll
      for (int mt = 0; mt < C::kMt; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[mt][nt][e] = fmaf(o[mt][nt][e], (1.f / C::kCodeUnit) * v_tile_factor<BITS>(mt),
                                corr_v[PV ? mt >> 3 : mt >> 2][nt][e & 1]);
    }
    }  // tensor-core contraction
    if constexpr (BAL) {
      // This run's state of the unit, into workspace slot bal_v + unit (the runs of one
      // unit take consecutive slots): (m, l) per query row, then o. After a wait gave up,
      // the unit and the rest of the run get a maximum of -inf (no state), which the
      // merge pass skips.
      const bool aborted = done < seg_end;
      float2* const wml = reinterpret_cast<float2*>(p.ws_ml);
      const size_t sbase = (static_cast<size_t>(bal_v) + static_cast<size_t>(b) * p.num_kv_heads + hk) * p.nq;
      if (g == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int r = PV ? 2 * t + e2 : rbase + 8 * nt + 2 * t + e2;
            if (r < p.nq && (!PV || t < 2))
              wml[sbase + r] = aborted ? make_float2(-INFINITY, 0.f) : make_float2(m_run[nt][e2], l_run[nt][e2]);
          }
      }
      if (aborted) {
        for (int i = seg_end; i < my_chunks;) {
          const int x = x0 + i;
          const int bb = bal_seq_of(bal_S, p.num_seqs, x);
          const int n = (bal_S[bb + 1] - bal_S[bb]) / p.num_kv_heads;
          const int h = (x - bal_S[bb]) / n;
          const size_t base = (static_cast<size_t>(bal_v) + static_cast<size_t>(bb) * p.num_kv_heads + h) * p.nq;
          for (int r = rbase + lane; r < rbase + C::kNqp && r < p.nq; r += 32) wml[base + r] = make_float2(-INFINITY, 0.f);
          i += n - (x - bal_S[bb] - h * n);
        }
        break;
      }
      // o: four (4-bit pages) or two (8-bit) consecutive head dims per store where the
      // accumulator layout puts them in one thread, as in the combine below
      constexpr int kRun = BITS == 4 ? 4 : BITS == 8 ? 2 : 1;
#pragma unroll
      for (int mt = 0; mt < C::kMt; mt += kRun)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (PV && ((mt >> 2) & 1) != (t >> 1)) continue;
            const int r = PV ? (2 * t + (e & 1)) & 3 : rbase + 8 * nt + 2 * t + (e & 1);
            if (r >= p.nq) continue;
            float* dst = p.ws_o + (sbase + r) * DV + out_dim<BITS>(mt, e >> 1, g);
            if constexpr (kRun == 4) {
              *reinterpret_cast<float4*>(dst) =
                  make_float4(o[mt][nt][e], o[mt + 1][nt][e], o[mt + 2][nt][e], o[mt + 3][nt][e]);
            } else if constexpr (kRun == 2) {
              *reinterpret_cast<float2*>(dst) = make_float2(o[mt][nt][e], o[mt + 1][nt][e]);
            } else {
              *dst = o[mt][nt][e];
            }
          }
      continue;
    }
    break;
    }  // units of the run
  }

  allow_dependent_launch();  // the merge pass may be scheduled while this epilogue runs
  if constexpr (BAL) return;  // every state went to the workspace
  // ---- combine the page groups' states and write out. Group w's state is m[kNqAll],
  // l[kNqAll], o[kNqAll][kCoStride] at gstate(w): in its own ring region when it fits
  // there (free once the group's chunks are consumed and its copies have landed), else
  // packed from the start of shared memory once every group is done.
  if constexpr (C::kOwnRegions) {
    if constexpr (WQ > 1) group_barrier_any(1 + pg, WQ * 32, false);  // the group's warps have left its ring
  } else {
    __syncthreads();  // every stage consumed, every copy landed: the stage ring is free
  }
  float* const sf = reinterpret_cast<float*>(smem);
  constexpr int kGS = C::kOwnRegions ? C::kGroupBytes / 4 : C::kGroupStateFloats;  // floats between group states
  auto gstate = [&](int w) { return sf + w * kGS; };
  float* const st_m = gstate(C::kWP - 1) + C::kGroupStateFloats;  // this CTA's merged state (cluster merge)
  float* const st_l = st_m + C::kNqAll;
  float* const st_o = st_l + C::kNqAll;
  {
    float* const cm = gstate(pg);
    float* const cl = cm + C::kNqAll;
    float* const co = cl + C::kNqAll;
    if constexpr (CCQ) {
      const int d0 = (lane % (D / 8)) * 8;
#pragma unroll
      for (int qi = 0; qi < CCQ; ++qi) {
        if (qi >= p.nq) continue;
        if (lane == 0) {
          cm[qi] = ccm[qi];
          cl[qi] = ccl[qi];
        }
        if (lane < D / 8) {
          float* dst = co + qi * C::kCoStride + d0;
          *reinterpret_cast<float4*>(dst) = make_float4(cco[qi][0].x, cco[qi][0].y, cco[qi][1].x, cco[qi][1].y);
          *reinterpret_cast<float4*>(dst + 4) = make_float4(cco[qi][2].x, cco[qi][2].y, cco[qi][3].x, cco[qi][3].y);
        }
      }
    } else {
    if (g == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int r = 8 * nt + 2 * t + e2;
          cm[rbase + r] = m_run[nt][e2];
          cl[rbase + r] = l_run[nt][e2];
        }
    }
    // o values, four (4-bit pages) or two (8-bit) consecutive head dims per store where
    // the accumulator layout puts them in one thread; padding rows of the last n-tile
    // are never read
    constexpr int kRun = BITS == 4 ? 4 : BITS == 8 ? 2 : 1;
#pragma unroll
    for (int mt = 0; mt < C::kMt; mt += kRun)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // PV: a lane holds the columns of one group of each pair (t < 2: even groups,
          // columns 0-3; t >= 2: odd groups, columns 4-7, query rows 0-3 again)
          if (PV && ((mt >> 2) & 1) != (t >> 1)) continue;
          const int r = PV ? (2 * t + (e & 1)) & 3 : 8 * nt + 2 * t + (e & 1);
          if (rbase + r >= p.nq) continue;
          float* dst = co + (rbase + r) * C::kCoStride + out_dim<BITS>(mt, e >> 1, g);
          if constexpr (kRun == 4) {
            *reinterpret_cast<float4*>(dst) = make_float4(o[mt][nt][e], o[mt + 1][nt][e], o[mt + 2][nt][e], o[mt + 3][nt][e]);
          } else if constexpr (kRun == 2) {
            *reinterpret_cast<float2*>(dst) = make_float2(o[mt][nt][e], o[mt + 1][nt][e]);
          } else {
            *dst = o[mt][nt][e];
          }
        }
    }  // tensor-core contraction
  }
  __syncthreads();

  // Each thread merges the page groups' states for four consecutive outputs of one query
  // row: M = max of the groups' maxima, weights 2^(m_w - M), L and O their weighted sums.
  constexpr int kQuads = DV / 4;  // four-dim runs per row
  const int cs = p.max_partitions;        // cluster size in cluster mode
  const int runs = p.nq * kQuads;
  const int per = (runs + cs - 1) / cs;  // runs each cluster CTA finishes
  float* const rm = reinterpret_cast<float*>(smem + C::kWorkBytes);  // receive area: [member][kNqAll]
  float* const rl = rm + kMaxClusterParts * C::kNqAll;
  float* const ro = rl + kMaxClusterParts * C::kNqAll;  // [member][per runs][4]
  if constexpr (C::kPush) {
    if (in_cluster) cluster_wait();  // every member is running: its receive area may be written
  }
  for (int i4 = threadIdx.x; i4 < runs; i4 += C::kThreads) {
    const int r = i4 / kQuads, d0 = 4 * (i4 % kQuads);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::kWP; ++w) M = fmaxf(M, gstate(w)[r]);
    float L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < C::kWP; ++w) {
      const float* gw = gstate(w);
      const float mw = gw[r];
      const float wt = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
      L = fmaf(wt, gw[C::kNqAll + r], L);
      const float4 v = *reinterpret_cast<const float4*>(gw + 2 * C::kNqAll + r * C::kCoStride + d0);
      O.x = fmaf(wt, v.x, O.x);
      O.y = fmaf(wt, v.y, O.y);
      O.z = fmaf(wt, v.z, O.z);
      O.w = fmaf(wt, v.w, O.w);
    }
    const size_t orow = row0 + r;
    if (single) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      write_out4(p, orow * DV + d0, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
    } else if (in_cluster) {
      if constexpr (C::kPush) {
        const int owner = i4 / per;
        st_cluster_f32x4(smem_addr(ro + 4 * (slot * per + (i4 - owner * per))), owner, O);
        if (d0 / 4 < cs) {  // the row's (m, l) to member d0 / 4
          st_cluster_f32(smem_addr(&rm[slot * C::kNqAll + r]), d0 / 4, M);
          st_cluster_f32(smem_addr(&rl[slot * C::kNqAll + r]), d0 / 4, L);
        }
      } else {
        *reinterpret_cast<float4*>(st_o + r * DV + d0) = O;
        if (d0 == 0) {
          st_m[r] = M;
          st_l[r] = L;
        }
      }
    } else {
      const size_t ws = orow * p.max_partitions + slot;
      *reinterpret_cast<float4*>(p.ws_o + ws * DV + d0) = O;
      if (d0 == 0) {
        p.ws_ml[ws * 2] = M;
        p.ws_ml[ws * 2 + 1] = L;
      }
    }
  }

  if (in_cluster && C::kPush) {
    // ---- cluster merge, push form: after one cluster barrier every member's (m, l) and
    // o runs for this CTA's share sit in its receive area; nothing reads this CTA's
    // shared memory afterwards, so it may leave when done.
    cluster_sync();
    const int end = min(runs, (slot + 1) * per);
    for (int i4 = slot * per + threadIdx.x; i4 < end; i4 += C::kThreads) {
      const int r = i4 / kQuads, d0 = 4 * (i4 % kQuads), e = i4 - slot * per;
      float M = -INFINITY;
      for (int j = 0; j < cs; ++j) M = fmaxf(M, rm[j * C::kNqAll + r]);
      float L = 0.f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
        for (int j = 0; j < cs; ++j) {
          const float mj = rm[j * C::kNqAll + r];
          if (mj == -INFINITY) continue;
          const float wt = fast_exp2(mj - M);
          const float4 v = *reinterpret_cast<const float4*>(ro + 4 * (j * per + e));
          L = fmaf(wt, rl[j * C::kNqAll + r], L);
          O.x = fmaf(wt, v.x, O.x);
          O.y = fmaf(wt, v.y, O.y);
          O.z = fmaf(wt, v.z, O.z);
          O.w = fmaf(wt, v.w, O.w);
        }
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      write_out4(p, (row0 + r) * DV + d0, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
    }
  } else if (in_cluster) {
    // ---- merge the cluster's partition states (log-sum-exp) through distributed
    // shared memory, pull form (where a receive area would cost the second CTA per SM);
    // cluster CTA j holds the state of slot j. Each CTA finishes one slice of the
    // four-dim output runs.
    cluster_sync();
    const int end = min(runs, (slot + 1) * per);
    for (int i4 = slot * per + threadIdx.x; i4 < end; i4 += C::kThreads) {
      const int r = i4 / kQuads, d0 = 4 * (i4 % kQuads);
      // every member's (m, l, o) for these outputs, all remote loads in flight together
      float mj[kMaxClusterParts], lj[kMaxClusterParts];
      float4 oj[kMaxClusterParts];
#pragma unroll
      for (int j = 0; j < kMaxClusterParts; ++j) {
        mj[j] = -INFINITY;
        lj[j] = 0.f;
        oj[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < cs) {
          mj[j] = ld_cluster_f32(smem_addr(&st_m[r]), j);
          lj[j] = ld_cluster_f32(smem_addr(&st_l[r]), j);
          oj[j] = ld_cluster_f32x4(smem_addr(&st_o[r * DV + d0]), j);
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int j = 0; j < kMaxClusterParts; ++j) M = fmaxf(M, mj[j]);
      float L = 0.f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
#pragma unroll
        for (int j = 0; j < kMaxClusterParts; ++j) {
          if (mj[j] == -INFINITY) continue;
          const float wt = fast_exp2(mj[j] - M);
          L = fmaf(wt, lj[j], L);
          O.x = fmaf(wt, oj[j].x, O.x);
          O.y = fmaf(wt, oj[j].y, O.y);
          O.z = fmaf(wt, oj[j].z, O.z);
          O.w = fmaf(wt, oj[j].w, O.w);
        }
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      write_out4(p, (row0 + r) * DV + d0, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
    }
    cluster_sync();  // no CTA leaves while another still reads its shared memory
  }
}

}  // namespace pkv
