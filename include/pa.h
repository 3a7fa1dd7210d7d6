/*
 * pa.h -- C ABI of libpa: paged KV-cache write and paged decode attention on
 * one GB300 GPU (sm_103a), plus the untimed host block pool that builds the
 * block tables and slot mappings those two calls consume.
 *
 * Sources for what each call computes (page title, then section):
 *   [P2] the radix-tree prefix-cache fragmentation page (mhpq.cn) -- "Slotted Block 分槽与微块
 *        共享架构" (nodes packed as slots into shared blocks, (block_id, slot_offset, length)
 *        addressing, copy-on-write split-off on append, online defragmentation).
 *   [P1] "端侧 SLM 显存保活术：在 4GB 内存板卡上实现轻量 PagedAttention 与 KV 缓存分块"
 *        -- "注意力寻址：非连续物理块的间接寻址内核" (token t lives in logical block
 *        t / B at offset t % B; physical block = block_table[t / B]);
 *        "嵌入式轻量 Block 分配器设计" (free bitmap, lowest free block first,
 *        -1 when the pool is exhausted); "共享前缀块（Prefix Caching）" (shared,
 *        reference-counted prefix blocks).
 *   [P3] the KV Cache and BlockManager tutorial (hnwysp.cn) -- §3.4 (blocks swapped out to
 *        a pinned host buffer of 0.3 x the pool).
 *   [P4] "显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结"
 *        -- §三 sequence diagram (append a token: write at the next offset of the last
 *        block, or allocate and append a block when it is full; free all blocks at the end);
 *        §三.1 (two pool tensors, one fixed stride per physical block);
 *        §四 (copy-on-write of shared blocks, reference counts);
 *        FAQ on preemption (swap the blocks of a low-priority request to host memory);
 *        §五.1 (decode kernel: per sequence and head, loop over logical blocks through
 *        block_tables [num_seqs, max_blocks_per_seq] and context_lens [num_seqs],
 *        q.k, softmax with running rescale, weight V, normalise at the end).
 *
 * Conventions shared by every call:
 *   - Device pointers are owned by the caller; the library never frees them, never
 *     keeps them after the call returns and never allocates device memory for the
 *     caller's data.
 *   - Calls that take a `stream` are asynchronous on that stream (a cudaStream_t;
 *     NULL is the legacy default stream).  Their return value reports host-side
 *     argument checks and launch errors only.  Faults the kernels detect in the data
 *     (a block id outside the pool, a slot outside the pool, a context longer than
 *     the table) skip the offending access and set a bit in a per-device status word
 *     read by pa_read_device_status; no kernel traps.
 *   - Data layouts (row-major, element type pa_dtype, 16-byte aligned base pointers):
 *       q, out           [num_seqs][num_q_heads][head_dim]
 *       k, v (new rows)  [num_tokens][num_kv_heads][head_dim]
 *       k_cache, v_cache [num_blocks][num_kv_heads][block_size][head_dim]
 *                        (one (block, kv-head) tile is block_size*head_dim contiguous
 *                        elements)
 *       block_tables     int32 [num_seqs][max_blocks_per_seq]
 *       context_lens     int32 [num_seqs]; the length counts the newest token
 *       slot_mapping     int64 [num_tokens]; slot = physical_block * block_size + offset
 *   - Query head h attends with kv head h / (num_q_heads / num_kv_heads).
 *   - The library looks up, once per device, the device addresses of its own static
 *     device arrays (the status word, pa_decode_static's scratch) and keeps them for the
 *     life of the process: resetting a device (cudaDeviceReset, or any reset of its
 *     primary context) while the library is in use is not supported.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,     /* a null pointer, a negative size, a misaligned pointer */
    PA_ERR_UNSUPPORTED = -2,     /* a valid but unimplemented shape (head_dim, block size) */
    PA_ERR_CUDA = -3,            /* the CUDA runtime reported an error */
    PA_ERR_POOL_EXHAUSTED = -4,  /* the host pool has no free block */
    PA_ERR_DEVICE_TIMEOUT = -5,  /* reserved for waits that gave up (see status bits) */
    PA_ERR_BOUNDS = -6,          /* a host-side index outside its range */
    PA_ERR_WORKSPACE = -7,       /* workspace missing or smaller than required */
    PA_ERR_SCRATCH_LIMIT = -8    /* pa_decode_static: the problem needs more than its fixed scratch */
} pa_status;

/* Bits of the per-device status word (pa_read_device_status). */
#define PA_DEV_BAD_BLOCK_ID 0x1u /* a block-table entry outside [0, num_blocks) was skipped */
#define PA_DEV_BAD_CONTEXT  0x2u /* a context length < 0 or > max_blocks_per_seq*block_size was clamped */
#define PA_DEV_BAD_SLOT     0x4u /* a slot >= num_blocks*block_size was skipped */
#define PA_DEV_TIMEOUT      0x8u /* a copy pipeline wait gave up after about one second */
#define PA_DEV_BAD_PLAN     0x10u /* pa_decode_planned: the plan was built for another shape or grid */

/* Kernel choice of pa_decode_ex. */
typedef enum {
    PA_MATH_AUTO = 0,            /* the library's choice for the shape (PA_MATH_MMA when G <= 16) */
    PA_MATH_FMA = 1,             /* split grid, CUDA-core fp32 FMAs with warp-shuffle reductions,
                                    separate combine pass; G in {1, 2, 3, 4, 6, 8} */
    PA_MATH_MMA = 2,             /* tensor-core (mma.sync m16n8k16) QK^T and PV products in one
                                    persistent, load-balanced launch (num_seqs <= 1024; else the
                                    split grid below); G <= 16 */
    PA_MATH_MMA_SPLIT = 3        /* tensor-core products on the split grid with a combine pass */
} pa_math;

typedef struct {
    int tokens_per_split;        /* split grids: 0 = library's choice; else a multiple of
                                    max(block_size, 64), at most 1024 * block_size */
    int math;                    /* a pa_math value */
    int num_ctas;                /* persistent kernel: 0 = as many CTAs as fit on the GPU at once
                                    (16 fewer for the two-per-SM grid with PA_DECODE_EARLY_READS, so
                                    that a chained launch's last CTAs find free slots) */
    int flags;                   /* PA_DECODE_EARLY_READS: pa_decode_append / pa_multi_query_append may
                                    read lengths, tables and cached rows before the preceding kernel
                                    in the stream has finished (see pa_decode_append); off by
                                    default.  PA_PREFILL_MMA_SYNC: see pa_multi_query. */
    unsigned long long* timeline;/* persistent kernel trace, NULL = off; else device memory of
                                    num_ctas * 16 uint64 per CTA: global-timer ns at 0 entry,
                                    1 dependency wait passed, 2 prefix sums done, 3 first block ids
                                    read, 4 first copies issued, 5 first chunk landed, 6 last chunk
                                    landed, 7 last chunk consumed, 8 exit; then 9 ns consumers waited
                                    for chunks, 10 ns spent finishing segments, 11 ns the producer
                                    waited for a free stage, 12 cut segments merged, 13 segment
                                    pieces finished, 14 chunks streamed, 15 SM id.  Entries of CTAs
                                    that own no chunk stay as set. */
} pa_decode_options;

/* ------------------------------------------------------------------------------------
 * pa_cache_write  [P4 §三 sequence diagram; P1 address formula]
 * For every token i with slot_mapping[i] >= 0 and every kv head h, copy the rows
 *   k[i][h][:] -> k_cache[slot / block_size][h][slot % block_size][:]
 *   v[i][h][:] -> v_cache[slot / block_size][h][slot % block_size][:]
 * bit for bit.  A negative slot skips the token (padding).  A slot at or beyond
 * num_blocks*block_size is skipped and sets PA_DEV_BAD_SLOT.
 * head_dim must be a positive multiple of 8; all pointers 16-byte aligned.
 * Returns PA_OK, PA_ERR_INVALID_ARG or PA_ERR_CUDA.
 * ---------------------------------------------------------------------------------- */
int pa_cache_write(const void* k, const void* v, const int64_t* slot_mapping,
                   void* k_cache, void* v_cache,
                   int num_tokens, int num_kv_heads, int head_dim, int block_size,
                   int num_blocks, int dtype, void* stream);

/* ------------------------------------------------------------------------------------
 * pa_copy_blocks  [P4 §四 copy-on-write; P4 FAQ on preemption (swap); P3 §3.4 pinned
 *                  host swap buffer]
 * For i = 0..num_pairs-1 copy every kv head's rows of block src_ids[i] of the source pool
 * into block dst_ids[i] of the destination pool, bit for bit:
 *   dst_k[dst_ids[i]][h][:][:] = src_k[src_ids[i]][h][:][:] for every h, and the same for V.
 * Pools are [blocks][num_kv_heads][block_size][head_dim] (src_blocks, dst_blocks blocks).
 * Source and destination may be the same pool (copy-on-write inside the cache) or two pools
 * (swap out to, or in from, a pool in host memory).  Every pointer is device memory or
 * pinned host memory (cudaHostAlloc / cudaHostRegister), passed by the address the caller
 * holds; host memory that CUDA does not know as pinned is refused (PA_ERR_INVALID_ARG).
 * src_ids, dst_ids: int32 [num_pairs], device or pinned host memory.
 * A pair with an id outside its pool is skipped and sets PA_DEV_BAD_BLOCK_ID.  The
 * destination blocks must be distinct and no destination may be the source of another pair
 * (else which bytes land is unspecified).  Asynchronous on `stream`; pinned host memory
 * must stay allocated, and host code must not touch it, until the copy has completed.
 * A pa_decode_append launched right after it that reads the destination pool must not
 * ask for early reads (PA_DECODE_EARLY_READS), which could read the rows before they land.
 * head_dim a positive multiple of 8; pools 16-byte aligned.
 * Returns PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED or PA_ERR_CUDA.
 * ---------------------------------------------------------------------------------- */
int pa_copy_blocks(const void* src_k, const void* src_v, int src_blocks,
                   void* dst_k, void* dst_v, int dst_blocks,
                   const int32_t* src_ids, const int32_t* dst_ids, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int dtype, void* stream);

/* ------------------------------------------------------------------------------------
 * pa_decode  [P4 §五.1; P1 address formula]
 * For every sequence s and query head h (kv head hk = h / (num_q_heads/num_kv_heads)),
 * with L = context_lens[s] and the cached rows t = 0..L-1 found at
 *   (block_tables[s][t / block_size], t % block_size):
 *   out[s][h][:] = sum_t softmax_t(scale * q[s][h] . K[t]) * V[t][:]
 * accumulated in fp32 and rounded to nearest into the output dtype.  L == 0 gives
 * a zero row.  Supported: head_dim 128, block_size 16/32/64/128, num_q_heads a
 * multiple of num_kv_heads.
 *
 * All query heads of a GQA group share each K/V tile.  The default kernel is one
 * persistent launch in which every CTA streams an equal share of all 64-token
 * chunks of all (sequence, kv head) pairs; pairs cut by share boundaries leave
 * partial results in `workspace` that the last CTA to finish merges.
 * `workspace`: device memory of at least pa_decode_workspace_size(...) bytes,
 * owned by the caller, 16-byte aligned, ZERO-FILLED before its first use (see
 * pa_decode_workspace_init); every completed call leaves it ready for the next
 * one of any shape that runs the same kernel kind (pa_decode_kernel_kind) with the
 * same num_ctas option.  NULL is allowed when the size is 0.  Calls that share a
 * workspace must not overlap on the GPU.  After a call that set PA_DEV_TIMEOUT, or
 * before switching kernel kind or CTA count, zero it again.
 * Returns PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE or PA_ERR_CUDA.
 * ---------------------------------------------------------------------------------- */
int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens,
              float scale, int num_kv_heads,
              int num_seqs, int num_q_heads, int head_dim, int block_size, int num_blocks,
              int max_blocks_per_seq, int dtype,
              void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * pa_decode_static  [no counterpart on the pages: an allocation-free calling form]
 * pa_decode for callers that cannot allocate device memory: code that runs where it
 * does not own an allocator (a plugin or custom op inside a host framework whose
 * memory pool is reserved and managed by that framework), and real-time or
 * certified deployments that forbid device allocation after start-up.  Same inputs,
 * outputs and results as pa_decode; the scratch (partial results and arrival
 * counters) lives in one file-scope device array of PA_DECODE_STATIC_SCRATCH_BYTES
 * per GPU, held from the library's first use on that GPU until the process exits.
 * No call allocates or frees memory.
 *   - The first call on a device looks up that array's device address (once per
 *     device, with that device current); make that first call before any stream
 *     capture.
 *   - Problems whose scratch would not fit return PA_ERR_SCRATCH_LIMIT (see
 *     pa_decode_workspace_size for the requirement).
 *   - Every call shares the array and finds the previous call's contents; the call
 *     clears what has to start at zero.  Calls that may overlap on the GPU (other
 *     streams, other host threads) race on the array: serialise them.
 * Returns the codes of pa_decode, or PA_ERR_SCRATCH_LIMIT.
 * ---------------------------------------------------------------------------------- */
#define PA_DECODE_STATIC_SCRATCH_BYTES (16u << 20)
int pa_decode_static(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, const int32_t* context_lens,
                     float scale, int num_kv_heads,
                     int num_seqs, int num_q_heads, int head_dim, int block_size, int num_blocks,
                     int max_blocks_per_seq, int dtype, void* stream);

#define PA_DECODE_EARLY_READS 1
/* pa_multi_query beyond 16 query rows per (sequence, kv head): the mma.sync tiles of 64 rows
 * instead of the default tcgen05 tiles of 128 rows (same results within the parity tolerance). */
#define PA_PREFILL_MMA_SYNC 4
/* pa_decode_plan: shares of the decode launch's CTAs that follow their measured streaming rates
 * (see pa_decode_plan). */
#define PA_PLAN_ADAPTIVE 8
/* pa_decode_plan_size / pa_decode_plan_sections / pa_decode_planned: the plan is a runs plan
 * (pa_decode_plan_runs). */
#define PA_PLAN_RUNS 16

/* ------------------------------------------------------------------------------------
 * pa_decode_append  [P4 §三 sequence diagram + §五.1; P1 address formula]
 * One decode step of one layer in a single launch: the cache write of the newest token
 * followed by decode attention over the whole context, i.e. the effect of
 *   pa_cache_write(k_new, v_new, slot(s) = block_tables[s][(L-1)/B]*B + (L-1)%B, ...)
 *   pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, ...)
 * with L = context_lens[s] (sequences with L == 0 write nothing and get zero rows).
 * k_new, v_new: [num_seqs][num_kv_heads][head_dim].  Workspace as for pa_decode (same
 * size query, persistent kind).  Supported: the persistent kernel's shapes
 * (pa_decode_kernel_kind == PA_KERNEL_PERSISTENT_MMA); else PA_ERR_UNSUPPORTED.
 * Early reads (opt-in): with PA_DECODE_EARLY_READS in opts->flags the kernel may read
 * context_lens, block_tables and the cached rows of earlier tokens before the preceding
 * kernel in the stream has finished (so that, launched back to back, one layer's start
 * overlaps the previous layer's end); q, k_new and v_new are read, and out, the new slots
 * and the workspace written, only after it has finished.  The caller then guarantees that
 * the preceding kernel writes none of the caches, the tables or the lengths: a decode step
 * whose preceding kernel produces q and the new K/V qualifies; a pa_copy_blocks or
 * pa_gather_runs into the same pool (copy-on-write, defragmentation) does not.  Without the
 * flag nothing is read before the preceding kernel has finished.
 * ---------------------------------------------------------------------------------- */
int pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                     void* k_cache, void* v_cache,
                     const int32_t* block_tables, const int32_t* context_lens,
                     float scale, int num_kv_heads,
                     int num_seqs, int num_q_heads, int head_dim, int block_size, int num_blocks,
                     int max_blocks_per_seq, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream,
                     const pa_decode_options* opts);

/* ------------------------------------------------------------------------------------
 * pa_decode_plan / pa_decode_planned  [P4 §五.1 decode kernel; P1 address formula; P4 §三
 *                                     sequence diagram for the cache write of the new token]
 * A decode step runs the same attention over every layer with the same block tables and
 * lengths.  pa_decode_plan reads the tables and lengths once and writes a plan to device
 * memory: the 64-token chunks of every (sequence, kv head) with the physical ids of the blocks
 * each touches, and the share of the chunks each CTA of the decode launch streams.
 * pa_decode_planned then computes, per layer, exactly what pa_decode (k_new == NULL) or
 * pa_decode_append (k_new, v_new != NULL: the new token's rows written at position L - 1
 * first) computes, reading the plan instead of the tables and lengths.
 *   plan: device memory of pa_decode_plan_size(...) bytes, 16-byte aligned, caller-owned;
 *     plan_bytes (its size) must cover the call's shape (else PA_ERR_WORKSPACE).
 *     Valid while the tables' entries for positions < L and the lengths stay as they were
 *     when it was built, and only for the same shape and options (num_ctas).
 *   workspace: pa_decode_planned_workspace_size(opts) bytes, 16-byte aligned, caller-owned,
 *     FILLED WITH 0xFF BYTES before first use (pa_decode_planned_workspace_init); every
 *     completed call leaves it so for the next (after a call that set PA_DEV_TIMEOUT, fill it
 *     again).  Calls that share a workspace must not overlap on the GPU.
 *   opts: num_ctas (<= the SM count; 0 = one CTA per SM), flags (PA_DECODE_EARLY_READS: the
 *     plan and cached rows may be read before the preceding kernel ends; the preceding
 *     kernel must then write none of the plan, the caches or the tables -- in particular a
 *     pa_decode_planned right after pa_decode_plan must not ask for it), timeline.
 * Adaptive plans (PA_PLAN_ADAPTIVE in opts->flags, given alike to pa_decode_plan_size,
 * pa_decode_plan, pa_decode_plan_sections and every pa_decode_planned on the plan: the plan's
 * layout and the decode kernel depend on it; a mismatch makes the kernel set PA_DEV_BAD_PLAN
 * and write nothing): SMs stream at different
 * rates, so by default every CTA gets the same weight of chunks; an adaptive plan instead
 * gives CTA c a share proportional to its rate measured by earlier pa_decode_planned calls on
 * plans built into the same buffer (each such call folds one measurement per CTA into the
 * buffer's rates, an exponential average; the first adaptive build into a buffer, or one for
 * another CTA count, uses equal shares).  Such calls therefore write to the plan buffer, and
 * two of them on one buffer must not overlap on the GPU.  Outputs are the same function of
 * the inputs whatever the shares (within the parity tolerance: the split points move).  The
 * rates section is the one part of the plan that a pa_decode_planned with early reads may read
 * while the preceding pa_decode_planned on the same plan writes it: such a race only loses one
 * measurement.  Measured on GB300: one layer launched alone and repeated gains 3-8 % (configs 3
 * and 4 of the benchmark); in a chain of layers with early reads the CTAs' order on the SMs
 * changes from layer to layer, the rates follow the launch order rather than the SMs, and the
 * chain loses about 15 % -- leave adaptive plans off there.
 * A plan that does not match the call's shape or grid makes the kernel write nothing and
 * set PA_DEV_BAD_PLAN.  Supported: head_dim 128, block_size 16/32/64/128, num_q_heads /
 * num_kv_heads <= 8, num_seqs <= 1024; else PA_ERR_UNSUPPORTED.
 * Returns the codes of pa_decode.
 * ---------------------------------------------------------------------------------- */
size_t pa_decode_plan_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int max_blocks_per_seq, const pa_decode_options* opts);
int pa_decode_plan(void* plan, size_t plan_bytes, const int32_t* block_tables, const int32_t* context_lens,
                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                   int num_blocks, int max_blocks_per_seq, void* stream, const pa_decode_options* opts);
/* Where a plan of this shape keeps the two sections a caller may read back (for inspection):
 * *bounds_offset: int32 [2 * num_ctas + 1], the first chunk of each CTA's two groups in the
 * plan's chunk order (the last entry = the number of chunks); *rates_offset: float [num_ctas], the
 * CTAs' measured streaming rates of an adaptive plan (weight per SM cycle; 0 = no measurement;
 * meaningful only after a pa_decode_planned call on an adaptive plan).  *num_ctas: the grid the
 * plan is built for.  Returns PA_OK or the shape's error code. */
int pa_decode_plan_sections(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, const pa_decode_options* opts, int* num_ctas,
                            size_t* bounds_offset, size_t* rates_offset);
size_t pa_decode_planned_workspace_size(const pa_decode_options* opts);
/* ------------------------------------------------------------------------------------
 * pa_decode_plan_runs  [P2 "Slotted Block 分槽与微块共享架构": (block_id, slot_offset, length)
 *                       triples; P4 §五.1 attention]
 * The plan of a decode step whose contexts are given as runs (as pa_decode_runs: sequence s reads
 * runs seq_runs[s] .. seq_runs[s+1]-1 of `runs`, int32 [R][3]; a run that leaves its block or the
 * pool counts as empty and sets PA_DEV_BAD_BLOCK_ID; contexts longer than max_context are cut and
 * set PA_DEV_BAD_CONTEXT).  One warp per sequence writes its tokens' rows into a token table in
 * the plan, then the plan kernel cuts the chunks as pa_decode_plan does.  Two launches.
 *   plan: pa_decode_plan_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
 *     max_blocks_per_seq = ceil(max_context / block_size), opts with PA_PLAN_RUNS) bytes.
 * Then pa_decode_planned with PA_PLAN_RUNS in opts->flags, the same max_blocks_per_seq and no
 * new rows (k_new = v_new = NULL) decodes one layer: every token's K and V row is one bulk copy
 * into a padded shared-memory row.  Not adaptive.  Returns the codes of pa_decode_plan.
 * ---------------------------------------------------------------------------------- */
int pa_decode_plan_runs(void* plan, size_t plan_bytes, const int32_t* runs, const int32_t* seq_runs, int num_seqs,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                        int max_context, void* stream, const pa_decode_options* opts);
/* Fill `bytes` of a pa_decode_planned workspace with 0xFF on `stream` (cudaMemsetAsync). */
int pa_decode_planned_workspace_init(void* workspace, size_t bytes, void* stream);
int pa_decode_planned(void* out, const void* q, const void* k_new, const void* v_new,
                      void* k_cache, void* v_cache, void* plan, size_t plan_bytes, float scale,
                      int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int num_blocks, int max_blocks_per_seq, int dtype,
                      void* workspace, size_t workspace_bytes, void* stream,
                      const pa_decode_options* opts);

/* ------------------------------------------------------------------------------------
 * pa_multi_query  [P4 §五.1 attention over the paged cache; P4's closing section on
 *                  chunked prefill: several new tokens of a sequence at once]
 * Sequence s owns query rows query_start[s] .. query_start[s+1]-1 of q and out
 * ([num_q_tokens][num_q_heads][head_dim]): its n_s newest tokens, which are the last n_s of its
 * L = context_lens[s] cached tokens (their K/V already written, e.g. by pa_cache_write).
 * Query token i sits at position L - n_s + i and attends causally:
 *   out[row][h][:] = sum_{t <= L - n_s + i} softmax_t(scale * q[row][h] . K[t]) * V[t][:]
 * with row = query_start[s] + i and K/V of kv head h / (num_q_heads / num_kv_heads).
 * n_s = 1 everywhere is pa_decode.  query_start: int32 [num_seqs + 1], non-decreasing,
 * query_start[num_seqs] = num_q_tokens; max_q_per_seq bounds every n_s.  Counts outside
 * [0, min(L, max_q_per_seq)], and spans outside [0, num_q_tokens), are clamped and set
 * PA_DEV_BAD_CONTEXT.
 * Kernels: while max_q_per_seq x (num_q_heads / num_kv_heads) <= 16 (and num_seqs <= 1024)
 * the persistent kernel, with a workspace as for pa_decode (same size query, persistent kind;
 * opts: num_ctas and timeline apply); beyond that, tcgen05 tiles of
 * 128 query rows per (sequence, kv head) with accumulators in tensor memory, one CTA each, no
 * workspace (chunked prefill; at most 65535 sequences and kv heads); opts->flags with
 * PA_PREFILL_MMA_SYNC selects mma.sync tiles of 64 rows instead.
 * Returns the codes of pa_decode.
 * ---------------------------------------------------------------------------------- */
int pa_multi_query(void* out, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, const int32_t* context_lens, const int32_t* query_start,
                   float scale, int num_kv_heads,
                   int num_seqs, int num_q_tokens, int max_q_per_seq, int num_q_heads, int head_dim,
                   int block_size, int num_blocks, int max_blocks_per_seq, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream,
                   const pa_decode_options* opts);

/* ------------------------------------------------------------------------------------
 * pa_multi_query_append  [P4 §三 sequence diagram + §五.1; P4's closing section on chunked
 *                         prefill; P1 address formula]
 * The cache write of every sequence's n_s new tokens followed by pa_multi_query, in one
 * launch: the effect of
 *   pa_cache_write(k_new, v_new, slot(row) = block_tables[s][p / B] * B + p % B, ...)
 *   pa_multi_query(out, q, k_cache, v_cache, ...)
 * where row = query_start[s] + i holds the token at position p = L - n_s + i (after the
 * clamping of n_s that pa_multi_query describes; rows it drops write nothing).  k_new, v_new: [num_q_tokens][num_kv_heads][head_dim],
 * rows as q's.  A slot whose block id lies outside [0, num_blocks) is not written.
 * Supported: the persistent kernel's shapes (max_q_per_seq x (num_q_heads / num_kv_heads)
 * <= 16); beyond that PA_ERR_UNSUPPORTED (write the rows with pa_cache_write, then call
 * pa_multi_query).  Early reads as for pa_decode_append (opt-in, PA_DECODE_EARLY_READS):
 * context_lens, block_tables, query_start and the cached rows of earlier tokens may then be
 * read before the preceding kernel in the stream has finished; q, k_new and v_new are read,
 * and out, the new slots and the workspace written, only after it.
 * Returns the codes of pa_decode.
 * ---------------------------------------------------------------------------------- */
int pa_multi_query_append(void* out, const void* q, const void* k_new, const void* v_new,
                          void* k_cache, void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens,
                          const int32_t* query_start, float scale, int num_kv_heads,
                          int num_seqs, int num_q_tokens, int max_q_per_seq, int num_q_heads,
                          int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                          int dtype, void* workspace, size_t workspace_bytes, void* stream,
                          const pa_decode_options* opts);

/* ------------------------------------------------------------------------------------
 * pa_decode_runs  [P2 "Slotted Block 分槽与微块共享架构": nodes addressed by
 *                  (block_id, slot_offset, length) triples; P4 §五.1 attention]
 * One query token per sequence over a context given as runs instead of a block table:
 * sequence s reads runs seq_runs[s] .. seq_runs[s+1]-1 of `runs` (int32 [R][3]: block id,
 * slot offset, length) in order, so its token t is row slot_offset + (t - run start) of the
 * run's block, and its length L is the sum of its runs' lengths.  Otherwise as pa_decode:
 *   out[s][h][:] = sum_t softmax_t(scale * q[s][h] . K[t]) * V[t][:]   (L == 0: zero row).
 * max_context bounds every L (longer contexts are cut there and set PA_DEV_BAD_CONTEXT).  A run
 * that leaves its block or the pool counts as empty and sets PA_DEV_BAD_BLOCK_ID.
 * Up to 1024 sequences (and max_context up to 2^21): three launches on the stream -- one warp
 * per sequence lays its tokens' rows out in a token table, the decode plan kernel cuts the
 * 64-token chunks among the SMs, and the planned decode kernel copies every token's K and V row
 * (one bulk copy each) into padded shared-memory rows.  Beyond that the split CUDA-core kernel
 * runs (each run piece one bulk copy of contiguous rows).  num_q_heads / num_kv_heads in
 * {1, 2, 3, 4, 6, 8}, block_size 16/32/64/128, head_dim 128.
 * workspace: pa_decode_runs_workspace_size(...) bytes, 16-byte aligned (0: none needed), FILLED
 * WITH 0xFF BYTES before its first use (pa_decode_planned_workspace_init); every completed call
 * leaves it fit for the next (after a call that set PA_DEV_TIMEOUT, fill it again).  Calls that
 * share a workspace must not overlap on the GPU.
 * Returns PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE or PA_ERR_CUDA.
 * ---------------------------------------------------------------------------------- */
int pa_decode_runs(void* out, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* runs, const int32_t* seq_runs, float scale, int num_kv_heads,
                   int num_seqs, int num_q_heads, int head_dim, int block_size, int num_blocks,
                   int max_context, int dtype, void* workspace, size_t workspace_bytes, void* stream);
size_t pa_decode_runs_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                     int block_size, int max_context);

/* ------------------------------------------------------------------------------------
 * pa_gather_runs  [P2 online defragmentation: scattered read-only slots moved into
 *                  contiguous blocks; copy-on-write split-off of a shared slot]
 * For m = 0..num_moves-1, moves[m] = (src_block, src_off, length, dst_block, dst_off): every
 * kv head's rows src_off .. src_off+length-1 of src_block in (src_k, src_v) are copied bit
 * for bit to rows dst_off .. of dst_block in (dst_k, dst_v).  Pools [blocks][Hkv][B][D] on the
 * device (they may be the same pool).  A move that leaves a block or a pool is skipped and
 * sets PA_DEV_BAD_BLOCK_ID.  Destination rows of different moves must not overlap, nor any
 * move's source rows (else which bytes land is unspecified).  moves: int32 [num_moves][5],
 * device memory.  head_dim a positive multiple of 8; pools 16-byte aligned.
 * Returns PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED or PA_ERR_CUDA.
 * ---------------------------------------------------------------------------------- */
int pa_gather_runs(const void* src_k, const void* src_v, int src_blocks,
                   void* dst_k, void* dst_v, int dst_blocks,
                   const int32_t* moves, int num_moves,
                   int num_kv_heads, int head_dim, int block_size, int dtype, void* stream);

/* Bytes of workspace pa_decode needs for this shape on the current device. */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks_per_seq);

/* pa_decode with explicit options (opts may be NULL = defaults). */
int pa_decode_ex(void* out, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, const int32_t* context_lens,
                 float scale, int num_kv_heads,
                 int num_seqs, int num_q_heads, int head_dim, int block_size, int num_blocks,
                 int max_blocks_per_seq, int dtype,
                 void* workspace, size_t workspace_bytes, void* stream,
                 const pa_decode_options* opts);

size_t pa_decode_workspace_size_ex(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_blocks_per_seq,
                                   const pa_decode_options* opts);

/* Which kernel pa_decode_ex runs for this shape: PA_KERNEL_* below, or < 0 (a pa_status)
 * when no kernel serves it.  A workspace must stay with one kind: the persistent kernel
 * keeps arrival counters in it that split-grid partials would overwrite. */
#define PA_KERNEL_SPLIT_FMA 1
#define PA_KERNEL_PERSISTENT_MMA 2
#define PA_KERNEL_SPLIT_MMA 3
int pa_decode_kernel_kind(int num_seqs, int num_q_heads, int num_kv_heads, const pa_decode_options* opts);

/* Zero-fill `bytes` of workspace on `stream` (cudaMemsetAsync). */
int pa_decode_workspace_init(void* workspace, size_t bytes, void* stream);

/* The split length (tokens per split) pa_decode_ex would use; < 0 on invalid input. */
int pa_decode_plan_tokens_per_split(int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int max_blocks_per_seq,
                                    const pa_decode_options* opts);

/* Human-readable text of a pa_status value (static storage). */
const char* pa_status_string(int status);

/* Copy the current device's status word into *bits after all work on `stream`
 * has finished (this call synchronises the stream); clear it when `clear` != 0. */
int pa_read_device_status(void* stream, int clear, uint32_t* bits);

/* Number of kernels the library launched in this process (all devices). */
uint64_t pa_kernel_launch_count(void);

/* ------------------------------------------------------------------------------------
 * Host block pool  [P1 allocator section; P4 §三 lifecycle and §四 copy-on-write]
 * Not thread-safe; one owner.  Block ids are 0..num_blocks-1.
 * ---------------------------------------------------------------------------------- */
typedef struct pa_pool pa_pool;

/* A pool of num_blocks free blocks, or NULL if num_blocks <= 0 or memory is short. */
pa_pool* pa_pool_create(int num_blocks);
void pa_pool_destroy(pa_pool* pool);

/* The lowest-numbered free block, now with reference count 1, or PA_ERR_POOL_EXHAUSTED. */
int pa_pool_alloc(pa_pool* pool);
/* Add one reference to an allocated block; returns the new count or PA_ERR_BOUNDS. */
int pa_pool_incref(pa_pool* pool, int block_id);
/* Drop one reference; the block returns to the free set at 0.  Returns the new
 * count, or PA_ERR_BOUNDS for an id that is out of range or already free. */
int pa_pool_decref(pa_pool* pool, int block_id);
int pa_pool_refcount(const pa_pool* pool, int block_id);
int pa_pool_num_free(const pa_pool* pool);
int pa_pool_num_blocks(const pa_pool* pool);

/* Give a sequence of context_len tokens its ceil(context_len / block_size) blocks:
 * the first `shared_blocks` entries are copied from `shared_row` (each gains a
 * reference), the rest are allocated.  table_row has max_blocks entries; unused
 * ones are set to -1.  On PA_ERR_POOL_EXHAUSTED nothing stays allocated. */
int pa_pool_assign(pa_pool* pool, int32_t* table_row, int max_blocks, int context_len,
                   int block_size, const int32_t* shared_row, int shared_blocks);

/* Append one token to a sequence that holds context_len tokens (P4 §三): if its last
 * block is full (or it has none) allocate a block and append it to the table; if the
 * last block is shared (reference count > 1) and not full, copy-on-write: allocate a
 * new block, drop one reference of the old one and point the table at the new one,
 * reporting (*cow_src, *cow_dst) so that the caller copies the block's rows on the
 * GPU (both -1 when no copy is needed).  *slot receives the new token's slot.
 * Returns PA_OK, PA_ERR_POOL_EXHAUSTED or PA_ERR_BOUNDS (table full). */
int pa_pool_append_token(pa_pool* pool, int32_t* table_row, int max_blocks, int context_len,
                         int block_size, int64_t* slot, int32_t* cow_src, int32_t* cow_dst);

/* Drop one reference of each of the ceil(context_len / block_size) blocks of a
 * sequence (P4 §三, end of request) and set the entries to -1. */
int pa_pool_release(pa_pool* pool, int32_t* table_row, int max_blocks, int context_len,
                    int block_size);

/* Move the first n blocks of a sequence from pool `from` to pool `to` (swap out: device pool
 * to host pool; swap in: back), P4 FAQ on preemption: for each i < n allocate a block of
 * `to`, record the pair (src_ids[i], dst_ids[i]) = (table_row[i], new id), drop one reference
 * of the old block in `from` and point table_row[i] at the new one.  The caller then copies
 * the pairs with pa_copy_blocks before anything reuses a freed block.  On
 * PA_ERR_POOL_EXHAUSTED nothing has changed.  Returns n, PA_ERR_INVALID_ARG,
 * PA_ERR_BOUNDS (a table entry not allocated in `from`) or PA_ERR_POOL_EXHAUSTED. */
int pa_pool_move_blocks(pa_pool* from, pa_pool* to, int32_t* table_row, int n,
                        int32_t* src_ids, int32_t* dst_ids);

/* ---- Slotted blocks (host)  [P2 "Slotted Block 分槽与微块共享架构"] ----
 * Nodes of n <= block_size tokens packed into shared blocks.  A node goes to the
 * earliest-opened block whose free tail still holds n (offset = tokens already placed there),
 * else to a fresh block, the lowest free id.  A released slot's space is reused only once its
 * block has no live slot left and returns to the free set. */
typedef struct pa_slots pa_slots;
pa_slots* pa_slots_create(int num_blocks, int block_size);
void pa_slots_destroy(pa_slots* pool);
/* PA_OK with (*block, *offset), PA_ERR_POOL_EXHAUSTED or PA_ERR_INVALID_ARG. */
int pa_slots_alloc(pa_slots* pool, int n, int32_t* block, int32_t* offset);
/* Live slots left in the block, or PA_ERR_BOUNDS for a slot that is not placed there. */
int pa_slots_release(pa_slots* pool, int32_t block, int32_t offset, int n);
int pa_slots_tail(const pa_slots* pool, int32_t block);   /* tokens placed (next offset) */
int pa_slots_live(const pa_slots* pool, int32_t block);   /* live slots */
int pa_slots_num_free(const pa_slots* pool);

/* slots[s] = slot of token context_lens[s] - 1 (the newest one), or -1 when the
 * context is empty; host arrays.  Returns PA_OK or PA_ERR_BOUNDS if a length
 * exceeds max_blocks*block_size or a needed table entry is negative. */
int pa_build_slot_mapping(const int32_t* block_tables, int max_blocks,
                          const int32_t* context_lens, int num_seqs, int block_size,
                          int64_t* slots);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
