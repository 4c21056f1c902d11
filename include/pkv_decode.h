/*
 * pkv_decode.h -- paged decode attention over a block-pool KV cache (GB300, sm_103a).
 *
 * What the library computes
 * -------------------------
 * Single-step and few-query decode attention over a paged KV cache, the read
 * described on the mlx-bun pages ("@mlx-bun/inference 0.0.0-stage -> 1.0.0",
 * package/src/kernels/attention/paged.ts: ``paged_attention_partial``,
 * ``paged_attention_affine_partial`` and ``paged_attention_merge`` behind
 * ``pagedAttentionView(...).attend(q, scale, mask)``; the 4-bit decode of
 * kernels/attention/kvq4-decode.ts; the few-query causal rule of
 * kernels/attention/multi-query.ts). For sequence b, query row i < N and query
 * head h:
 *
 *     kv    = h / (HQ / HK)                      consecutive heads share a KV head
 *     key t is visible iff t <= len_b - N + i    (len_b counts the N new rows)
 *                     and, with a sliding window W, t > len_b - N + i - W
 *     K[t]  = k_pool[block_tables[b][t / BS]][kv][t % BS][:]
 *     affine pages: K[t][d] = scale[t][d/64] * code[t][d] + bias[t][d/64]
 *     out[b][h][i] = softmax_t(scale * <q, K[t]>) . V[t]       rounded to bf16
 *
 * The work is split along the sequence into partitions; each partition keeps an
 * f32 online-softmax state (running max, normaliser, unnormalised output) and
 * a merge pass combines partitions by log-sum-exp. Each K/V row is read from
 * HBM once and serves every query head of its KV head (GQA reuse).
 *
 * Data layout (row-major, all device memory unless stated otherwise)
 * -----------------------------------------------------------------
 *   q             bf16  [num_seqs, num_q_heads, n_query, head_dim]
 *   k_pool,v_pool bits=16: bf16 [num_blocks, num_kv_heads, block_size, W]
 *                 bits=4/8: uint32 words [num_blocks, num_kv_heads, block_size,
 *                 W*bits/32]; code d of a row sits in word d/(32/bits) at
 *                 bit offset (d % (32/bits))*bits (lowest bits first).
 *                 W is head_dim for K and v_head_dim for V.
 *   k_scales, k_biases, v_scales, v_biases
 *                 bf16 [num_blocks, num_kv_heads, block_size, W/64]
 *                 (affine pages only; NULL for bf16 pages). Dim d uses group d/64.
 *                 These are the layouts of the pages' BlockPool
 *                 (state/paged/cache.ts): every plane [numBlocks, H, blockSize, width].
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]: logical page -> physical block.
 *   seq_lens      int32 [num_seqs]: cached rows per sequence, including the n_query
 *                 new ones.
 *   out           bf16  [num_seqs, num_q_heads, n_query, v_head_dim]
 *
 * Ownership: every pointer is borrowed; the library frees nothing and keeps no
 * pointer after a call returns (except a pkv_step handle, which keeps the pointers
 * it was created with until it is destroyed). Calls are asynchronous on the given stream
 * (a cudaStream_t passed as void*; NULL = the legacy default stream) and make
 * no allocation and no host synchronisation, so they can be captured in a
 * CUDA graph. Stream order holds as usual: the partial pass (unless its
 * partitions merge in clusters of several CTAs per SM outside a host-driven step
 * that reads its inputs from host memory) and the merge pass are launched as
 * programmatic dependents of the previous work on the stream (their CTAs may be
 * placed while that work finishes), and they touch no global memory before that
 * work has completed.
 *
 * Errors: host-side argument checks happen before any CUDA call and return a
 * negative PKV_ERR_* code without launching anything. Problems that only the
 * device can see (a block-table entry outside [0, num_blocks), a seq_len
 * below n_query or above max_blocks_per_seq*block_size) never trap: the
 * offending rows are skipped (bad block) or the sequence's outputs are written
 * as zeros (bad length), and a PKV_DEVERR_* bit is OR-ed into *error_flag when
 * error_flag is not NULL. Rows at or past seq_len in a sequence's last page
 * are never used, whatever they hold.
 */
#ifndef PKV_DECODE_H
#define PKV_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side return codes. */
#define PKV_OK 0
#define PKV_ERR_NULL_POINTER (-1)        /* a required pointer is NULL */
#define PKV_ERR_MISALIGNED (-2)          /* a device pointer is not 16-byte aligned */
#define PKV_ERR_BAD_LAYOUT (-3)          /* unsupported bits / group_size / head dims / block_size */
#define PKV_ERR_BAD_PARAMS (-4)          /* bad num_seqs, heads, n_query, table width or partition size */
#define PKV_ERR_UNSUPPORTED_SHAPE (-5)   /* no kernel for these head dims with (num_q_heads/num_kv_heads)*n_query rows */
#define PKV_ERR_WORKSPACE_TOO_SMALL (-6) /* workspace NULL or smaller than pkv_plan.workspace_bytes */
#define PKV_ERR_CUDA (-7)                /* a CUDA runtime or driver call failed */
#define PKV_ERR_SCRATCH_TOO_SMALL (-8)   /* no-alloc entry: partition states larger than its static scratch */

/* Size of the static device scratch behind pkv_paged_decode_attention_no_alloc. */
#define PKV_STATIC_SCRATCH_BYTES (16u << 20)

/* Device-side error bits, OR-ed into *error_flag. */
#define PKV_DEVERR_BAD_BLOCK 1   /* a referenced block id outside [0, num_blocks): its rows were skipped */
#define PKV_DEVERR_BAD_SEQ_LEN 2 /* seq_len < n_query or > max_blocks_per_seq*block_size: outputs zeroed */
#define PKV_DEVERR_TIMEOUT 4     /* an internal pipeline wait gave up (after about a second by
                                    default, see pkv_set_wait_limit_ns); the outputs of that call
                                    are then unspecified */

/* Pool layout descriptor (the pages' PagedAttentionStorage: blockSize, headDim,
 * vHeadDim, quantization {bits, groupSize}).
 * Head dims with a kernel (key/value; the host rejects the rest), each with up to 64
 * query rows per KV head ((num_q_heads / num_kv_heads) * n_query, the pages' limit for
 * the few-query kernel, kernels/attention/multi-query.ts):
 *   equal dims: 64, 128, 256 (bf16) and 128, 256 (affine);
 *   bf16 192/128, 256/128 and 128/256; affine 256/128 and 128/256. */
typedef struct pkv_pool_layout {
  int32_t num_blocks;   /* blocks in the pool, > 0 */
  int32_t num_kv_heads; /* HK, > 0 */
  int32_t block_size;   /* BS: rows per block; a multiple of the chunk the kernels stage (16 rows
                           bf16, 32 affine), or 8 (bf16) / 8 or 16 (affine) rows, a chunk then
                           spanning several blocks: such pools run partitions (not the balanced
                           schedule), and neither the CUDA-core contraction nor the fused
                           append-and-attend call takes them (PKV_ERR_UNSUPPORTED_SHAPE) */
  int32_t head_dim;     /* D: key (and query) head dim */
  int32_t bits;         /* 16 = bf16 pages; 4 or 8 = affine codes */
  int32_t group_size;   /* affine group; must be 64 (ignored for bf16) */
  int32_t v_head_dim;   /* Dv: value (and output) head dim; 0 = head_dim */
} pkv_pool_layout;

/* Per-call decode parameters. */
typedef struct pkv_decode_params {
  int32_t num_seqs;           /* B, > 0 */
  int32_t num_q_heads;        /* HQ, a multiple of num_kv_heads; num_seqs * HQ * n_query < 2^31 */
  int32_t n_query;            /* N >= 1 new query rows per sequence */
  int32_t max_blocks_per_seq; /* row stride of block_tables, > 0 */
  int32_t partition_tokens;   /* rows per partition: 0 = chosen from lengths and SM count;
                                 otherwise rounded up to the chunk rows (16 bf16, 32 affine).
                                 A value >= max_blocks_per_seq*block_size gives one partition. */
  int32_t window;             /* sliding window W in rows, 0 = none: query i then sees only keys
                                 t with len-N+i-W < t <= len-N+i (the W most recent positions,
                                 its own included), as the pages' causal mask with a window
                                 size (kernels/attention/masks.ts, createCausalMask). Reads
                                 start at the 32-row boundary at or below the lowest visible
                                 row, so up to 31 rows below the window are read and masked:
                                 their block-table entries must be valid and their values
                                 finite, as for any row below len; rows further below are
                                 never read */
  int32_t contraction;        /* how the dot products and the weighted value sums run:
                                 PKV_CONTRACTION_AUTO (0, the library's choice per shape),
                                 PKV_CONTRACTION_TENSOR (1, warp-level tensor-core MMA) or
                                 PKV_CONTRACTION_CUDA_CORE (2, per-lane f32 FMAs with warp-shuffle
                                 reductions, the form of the pages' direct paged kernel,
                                 kernels/attention/paged.ts; bf16 pages with equal key/value head
                                 dims and at most 4 query rows per KV head, else
                                 PKV_ERR_UNSUPPORTED_SHAPE) */
  int32_t schedule;           /* how the rows are split over the CTAs, when partition_tokens = 0:
                                 PKV_SCHEDULE_AUTO (0): balanced for 4-bit pages where the plan
                                 would otherwise write partition states to the workspace, else
                                 partitions;
                                 PKV_SCHEDULE_PARTITIONS (1): fixed-size partitions of every
                                 (sequence, KV head);
                                 PKV_SCHEDULE_BALANCED (2): balanced wherever it is available.
                                 Balanced: one wave of CTAs, each of whose page groups reads an
                                 equal run of the list of all (sequence, KV head, chunk)
                                 triples, whatever the lengths; a run's state per (sequence, KV
                                 head) goes to the workspace and the merge pass combines them.
                                 Available for up to 256 sequences, the tensor-core contraction
                                 and the unfused entry points (the fused append-and-attend call
                                 runs partitions). Ignored when partition_tokens > 0. */
} pkv_decode_params;

#define PKV_CONTRACTION_AUTO 0
#define PKV_CONTRACTION_TENSOR 1
#define PKV_CONTRACTION_CUDA_CORE 2

#define PKV_SCHEDULE_AUTO 0
#define PKV_SCHEDULE_PARTITIONS 1
#define PKV_SCHEDULE_BALANCED 2

/* How a call will be carried out. */
typedef struct pkv_plan {
  int32_t partition_tokens; /* resolved rows per partition */
  int32_t max_partitions;   /* partitions per (sequence, KV head) in the grid and the workspace: those
                               of the longest admissible sequence, or with a window those that tile
                               window + n_query - 1 rows from a base rounded down to a multiple of 32
                               rows (at most window + n_query + 30 rows) */
  int32_t chunk_rows;       /* rows staged per pipeline step */
  int32_t sm_count;         /* SM count the plan was made for */
  int32_t threads_per_cta;  /* partial-kernel CTA size */
  int32_t smem_bytes;       /* partial-kernel dynamic shared memory */
  int32_t merge_in_cluster; /* 1: the partitions of each (sequence, KV head) form one thread-block
                               cluster and merge through distributed shared memory inside the
                               partial kernel (2..16 partitions on a grid of at most one wave) */
  int32_t contraction;      /* the contraction the call runs: PKV_CONTRACTION_TENSOR or
                               PKV_CONTRACTION_CUDA_CORE */
  size_t workspace_bytes;   /* device scratch for the partition states; 0 with one partition
                               or with merge_in_cluster; with balanced = 1, enough for either
                               schedule (the fused call runs partitions) */
  int32_t balanced;         /* 1: the balanced schedule (pkv_decode_params.schedule); then
                               partition_tokens, max_partitions and merge_in_cluster describe the
                               partitions the fused call would run */
} pkv_plan;

/* Makes the plan for (layout, params) on a GPU with sm_count SMs. Pure host
 * code, no CUDA call. Returns PKV_OK or a PKV_ERR_* code. */
int pkv_make_plan(const pkv_pool_layout* layout, const pkv_decode_params* params, int32_t sm_count,
                  pkv_plan* plan);

/* pkv_make_plan for the current CUDA device (reads its SM count). */
int pkv_plan_for_current_device(const pkv_pool_layout* layout, const pkv_decode_params* params,
                                pkv_plan* plan);

/* Paged decode attention: partial pass (and merge pass when there is more than
 * one partition), asynchronous on `stream`.
 *   scale            softmax scale applied to <q, K> (e.g. 1/sqrt(head_dim))
 *   workspace        device scratch of at least plan.workspace_bytes (may be NULL
 *                    when that is 0); the caller owns it; its contents need no
 *                    initialisation and are overwritten.
 *   error_flag       optional device int32 that receives PKV_DEVERR_* bits; the
 *                    library only ORs into it, the caller clears it.
 * Returns PKV_OK once the kernels are enqueued, or a PKV_ERR_* code. */
int pkv_paged_decode_attention(const pkv_pool_layout* layout, const pkv_decode_params* params,
                               const void* q, const void* k_pool, const void* v_pool,
                               const void* k_scales, const void* k_biases, const void* v_scales,
                               const void* v_biases, const int32_t* block_tables,
                               const int32_t* seq_lens, float scale, void* out, void* workspace,
                               size_t workspace_bytes, int32_t* error_flag, void* stream);

/* The two passes of pkv_paged_decode_attention, for callers that schedule them
 * apart (for example to combine partition states computed elsewhere, or to time
 * the partial pass alone). pkv_paged_decode_partial takes the same arguments
 * and enqueues only the partial pass: with one partition, or when the plan merges
 * in a cluster, it writes the final `out`; otherwise it writes each partition's
 * state (running max in log2 units, normaliser, unnormalised output, all f32)
 * into `workspace`. pkv_merge_partitions then enqueues the log-sum-exp merge of
 * those states into `out` for the same layout and params (it does nothing when
 * the plan needs no merge pass).
 * Returns as pkv_paged_decode_attention. */
int pkv_paged_decode_partial(const pkv_pool_layout* layout, const pkv_decode_params* params, const void* q,
                             const void* k_pool, const void* v_pool, const void* k_scales,
                             const void* k_biases, const void* v_scales, const void* v_biases,
                             const int32_t* block_tables, const int32_t* seq_lens, float scale, void* out,
                             void* workspace, size_t workspace_bytes, int32_t* error_flag, void* stream);

int pkv_merge_partitions(const pkv_pool_layout* layout, const pkv_decode_params* params,
                         const int32_t* seq_lens, const void* workspace, size_t workspace_bytes, void* out,
                         int32_t* error_flag, void* stream);

/* One decode step driven from host memory, as a host-side serving loop runs it
 * (and what the end-to-end figure of bench.py times). The step's inputs (q,
 * seq_lens, changed block tables and, for the fused step, the new K/V rows) sit
 * packed in a host block in_host of in_bytes bytes, laid out as their device
 * counterparts in in_dev; the device pointers q, block_tables, seq_lens, k_new,
 * v_new may point into in_dev. On `stream` the call enqueues the decode
 * (pkv_paged_decode_append_attention when k_new and v_new are given, else
 * pkv_paged_decode_attention, the pools then only read) with the step's data
 * moving as follows:
 *   - in_host page-locked and mapped into the device's address space (the default
 *     for cudaHostAlloc / pinned memory on a GB300), with in_host and in_dev
 *     16-byte aligned: the kernels read every input that lies in in_dev's range
 *     directly from in_host, over NVLink-C2C, and in_dev is not written. The
 *     block must hold the step's final values when the call is made: a grid of
 *     one CTA per SM may read q, seq_lens and the block tables from it before the
 *     previous kernel on the stream has finished;
 *   - otherwise: one cudaMemcpyAsync of the block into in_dev first (synchronised
 *     by the runtime when in_host is pageable); in_bytes = 0 copies nothing;
 *   - out_host such mapped memory (16-byte aligned): the kernels write the bf16
 *     output to it as well as to `out`; other host memory gets a cudaMemcpyAsync
 *     of `out` after the decode; NULL: nothing.
 * The kernels reach mapped host memory with ordinary loads and stores; the
 * copy engine's start-up latency would be far larger than the transfer of a few
 * KB. All other arguments are those of the two decode calls; a failed copy
 * returns PKV_ERR_CUDA. */
int pkv_paged_decode_attention_host(const pkv_pool_layout* layout, const pkv_decode_params* params,
                                    const void* in_host, void* in_dev, size_t in_bytes, void* out_host,
                                    const void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                    void* k_scales, void* k_biases, void* v_scales, void* v_biases,
                                    const int32_t* block_tables, const int32_t* seq_lens, float scale, void* out,
                                    void* workspace, size_t workspace_bytes, int32_t* error_flag, void* stream);

/* A prepared host-driven step: the arguments of pkv_paged_decode_attention_host
 * checked, planned and resolved into kernel parameters and TMA descriptors once,
 * so that each step costs the host only its launches (and copies, if any). The step keeps
 * every pointer it is given: the buffers must outlive it and stay at their
 * addresses (a resized pool or workspace needs a new step), and the device that
 * was current at creation must be current when it runs. The handle lives in host
 * memory (the one host allocation of this library); no device memory is
 * allocated.
 *   pkv_step_create   arguments as pkv_paged_decode_attention_host, plus the
 *                     handle's address; returns PKV_OK or a PKV_ERR_* code
 *                     (nothing is created then)
 *   pkv_step_run      enqueues the step on the stream given at creation, moving
 *                     its data as pkv_paged_decode_attention_host does
 *   pkv_step_destroy  frees the handle (NULL is allowed); it does not wait for
 *                     work in flight, which keeps using the caller's buffers */
typedef struct pkv_step pkv_step;

int pkv_step_create(const pkv_pool_layout* layout, const pkv_decode_params* params, const void* in_host, void* in_dev,
                    size_t in_bytes, void* out_host, const void* q, const void* k_new, const void* v_new,
                    void* k_pool, void* v_pool, void* k_scales, void* k_biases, void* v_scales, void* v_biases,
                    const int32_t* block_tables, const int32_t* seq_lens, float scale, void* out, void* workspace,
                    size_t workspace_bytes, int32_t* error_flag, void* stream, pkv_step** step);
int pkv_step_run(pkv_step* step);
void pkv_step_destroy(pkv_step* step);

/* pkv_paged_decode_attention for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point.
 *
 * Some callers cannot call cudaMalloc: runtimes whose device memory is owned by
 * their own allocator, which reserves every byte up front and forbids other
 * allocations, and plugins that are handed only the tensors of one call. They
 * cannot provide the workspace the main entry point needs. This entry point
 * needs none. It keeps the f32 partition states in a file-scope static device
 * array of PKV_STATIC_SCRATCH_BYTES (16 MiB), which every GPU that loads the
 * library holds until the process exits. It calls no cudaMalloc, cudaFree or
 * allocating library routine. The caller still passes every input and `out`.
 *
 * Arguments and results are those of pkv_paged_decode_attention, without the
 * workspace. With partition_tokens = 0 the library picks the partition size as
 * usual and coarsens it until the states fit (one partition needs no scratch).
 * A caller-fixed partition_tokens whose states would exceed the scratch is
 * rejected with PKV_ERR_SCRATCH_TOO_SMALL.
 *
 * Set-up: the first call on each device looks up the scratch's device address
 * (cudaGetSymbolAddress, with that device current) and caches it, keyed on the
 * device's current context; a call after a device reset (which makes a new
 * context and loads the module again) looks it up anew. Make the first call on a
 * device, and the first after a reset, before any stream capture on it.
 *
 * Sharing: every call on a device uses the same scratch, which keeps the last
 * call's contents; nothing in it needs to start at zero. Calls whose kernels
 * overlap on the GPU (different streams, or concurrent host threads) race on
 * the scratch and must be ordered by the caller. */
int pkv_paged_decode_attention_no_alloc(const pkv_pool_layout* layout, const pkv_decode_params* params,
                                        const void* q, const void* k_pool, const void* v_pool,
                                        const void* k_scales, const void* k_biases, const void* v_scales,
                                        const void* v_biases, const int32_t* block_tables,
                                        const int32_t* seq_lens, float scale, void* out, int32_t* error_flag,
                                        void* stream);

/* Write side: appends each sequence's n_new new K and V rows into its pages at
 * cache positions seq_lens[b] .. seq_lens[b] + n_new - 1 (position t goes to block
 * block_tables[b][t / block_size], row t % block_size), the pages'
 * PagedKVCache.append / BlockPool.writeBlock (state/paged/cache.ts). Blocks must
 * already be in the tables; allocating them is the caller's.
 *   k_new, v_new  bf16 [num_seqs, num_kv_heads, n_new, head_dim / v_head_dim],
 *                 16-byte aligned
 *   seq_lens      rows held BEFORE the append (the caller then adds n_new)
 * bf16 pages are copied. Affine pages are quantised per row and 64-dim group
 * (the pages do not give the quantiser's formula; this is the min/max reading,
 * every step in f32):
 *     scale = bf16((max - min) / (2^bits - 1)), bias = bf16(min),
 *     code  = clamp(round_half_even((x - bias) / scale), 0, 2^bits - 1)
 *             (0 when the stored scale is 0),
 * codes packed lowest bits first. Bad block ids skip their row and set
 * PKV_DEVERR_BAD_BLOCK; seq_lens[b] + n_new above max_blocks_per_seq*block_size
 * sets PKV_DEVERR_BAD_SEQ_LEN and writes nothing for that sequence.
 * Layouts: every (bits, head dims) pair the decode has a kernel for.
 * Asynchronous on `stream`. */
int pkv_paged_append(const pkv_pool_layout* layout, int32_t num_seqs, int32_t max_blocks_per_seq, int32_t n_new,
                     const void* k_new, const void* v_new, const int32_t* block_tables, const int32_t* seq_lens,
                     void* k_pool, void* v_pool, void* k_scales, void* k_biases, void* v_scales, void* v_biases,
                     int32_t* error_flag, void* stream);

/* One decode step with its write: appends each sequence's N = n_query new K and
 * V rows into their pages, then attends over the cache that holds them, in the
 * same launches as pkv_paged_decode_attention. This is the pages' appendDecode
 * (PagedKVCache.appendDecode: append, then read the paged view of the grown
 * cache, "@mlx-bun/inference 0.0.0-stage -> 1.0.0", state/paged/cache.ts).
 *   k_new, v_new  bf16 [num_seqs, num_kv_heads, n_query, head_dim / v_head_dim], 16-byte
 *                 aligned: the K and V rows of the step's query tokens
 *   seq_lens      rows held AFTER the append, as for pkv_paged_decode_attention:
 *                 the new rows go to cache positions seq_lens[b] - n_query ..
 *                 seq_lens[b] - 1, whose blocks must already be in the tables
 * Every other argument is that of pkv_paged_decode_attention; k_pool, v_pool and,
 * for affine pages, the scale and bias planes are written. The rows written and
 * the output are bit for bit those of pkv_paged_append (with seq_lens - n_query)
 * followed by pkv_paged_decode_attention with the same plan. Each new row is
 * written by the CTA whose partition holds it, before that CTA reads the
 * partition, so no second launch and no re-read of the rows from another CTA is
 * needed. Blocks shared by several sequences must not receive new rows (the
 * caller copies them first). A row whose block id is bad is neither written nor
 * read and sets PKV_DEVERR_BAD_BLOCK. */
int pkv_paged_decode_append_attention(const pkv_pool_layout* layout, const pkv_decode_params* params,
                                      const void* q, const void* k_new, const void* v_new, void* k_pool,
                                      void* v_pool, void* k_scales, void* k_biases, void* v_scales,
                                      void* v_biases, const int32_t* block_tables, const int32_t* seq_lens,
                                      float scale, void* out, void* workspace, size_t workspace_bytes,
                                      int32_t* error_flag, void* stream);

/* Bit-exact gather of one pool plane into contiguous per-sequence rows, the
 * fetch copy of the pages' BlockPool.gather / pickBlocks (state/paged/cache.ts):
 *   out[b][h][t][:] = pool[block_tables[b][t / block_size]][h][t % block_size][:]
 * for t < seq_lens[b] (<= max_len); rows t >= seq_lens[b] of out are left as they
 * were. pool: [num_blocks, num_kv_heads, block_size, row_bytes] bytes;
 * out: [num_seqs, num_kv_heads, max_len, row_bytes] bytes. row_bytes must be a
 * positive multiple of 4; pool and out 16-byte aligned. Bad block ids skip the
 * row and set PKV_DEVERR_BAD_BLOCK; a seq_len outside [0, max_len] or above
 * max_blocks_per_seq*block_size sets PKV_DEVERR_BAD_SEQ_LEN and copies nothing
 * for that sequence. */
int pkv_paged_gather(const void* pool, int32_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                     int32_t row_bytes, const int32_t* block_tables, const int32_t* seq_lens,
                     int32_t num_seqs, int32_t max_blocks_per_seq, int32_t max_len, void* out,
                     int32_t* error_flag, void* stream);

/* Message for a PKV_ERR_* code (static storage). */
const char* pkv_strerror(int code);

/* Text of the last PKV_ERR_CUDA failure on this thread (static per-thread storage). */
const char* pkv_last_cuda_error(void);

/* Sets the bound, in nanoseconds, of one wait of the partial kernel's main loop for
 * the data of a pipeline stage, for every decode call prepared after it in this
 * process (a pkv_step keeps the bound it was created with), and returns the previous
 * bound; 0 restores the default of one second. The pages have no counterpart of it.
 * A wait that runs out gives up without a fault: the kernel sets PKV_DEVERR_TIMEOUT
 * in *error_flag, stops reading, lets every copy it has issued land (that drain waits
 * up to the default bound), finishes its epilogue and returns, so the stream and the
 * context stay usable and the output of that call is unspecified. It exists to check
 * this give-up path on a working GPU: a bound shorter than the time a stage takes
 * to arrive from HBM (a few microseconds) makes it run out on any input. Not
 * thread-safe against calls being prepared on other threads. */
uint64_t pkv_set_wait_limit_ns(uint64_t ns);

/* Library version, major*10000 + minor*100 + patch. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_DECODE_H */
