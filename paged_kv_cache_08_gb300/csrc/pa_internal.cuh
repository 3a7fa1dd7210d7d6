// Internal declarations shared by the libpa translation units (device side).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

constexpr int kHeadDim = 128;           // the only head size the pages use
constexpr int kStageTokens = 64;        // tokens of K (and of V) staged per pipeline step
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // give a copy wait ~1 s
constexpr int kMaxTableSlice = 1024;    // block-table entries of one split staged in shared memory
constexpr int kPersistMaxSeqs = 1024;   // sequences whose prefix sums the persistent kernel keeps on chip
constexpr int kPieceRows = 16;          // query rows per partial piece (the largest group), any G

// ---------------------------------------------------------------------------------------
// Arguments
// ---------------------------------------------------------------------------------------
struct CacheWriteArgs {
    const uint4* k;           // [T][Hkv][D] as 16-byte vectors
    const uint4* v;
    const int64_t* slots;     // [T]
    uint4* k_cache;           // [NB][Hkv][B][D]
    uint4* v_cache;
    unsigned int* status;
    long long total_vecs;     // T * Hkv * (D / 8)
    int num_kv_heads;
    int vecs_per_row;         // D / 8
    int block_size;
    long long pool_slots;     // NB * B
};

struct CopyBlocksArgs {
    const uint4* src_k;       // [src_blocks][Hkv][B][D] as 16-byte vectors (device or mapped host memory)
    const uint4* src_v;
    uint4* dst_k;             // [dst_blocks][Hkv][B][D]
    uint4* dst_v;
    const int32_t* src_ids;   // [num_pairs]
    const int32_t* dst_ids;   // [num_pairs]
    unsigned int* status;
    long long vecs_per_block; // Hkv * B * D / 8
    int num_pairs;
    int src_blocks;
    int dst_blocks;
};

struct DecodeArgs {
    void* out;                // [S][Hq][D]
    const void* q;            // [S][Hq][D]
    const void* k_cache;      // [NB][Hkv][B][D]
    const void* v_cache;
    const int32_t* block_tables;  // [S][max_blocks]
    const int32_t* context_lens;  // [S]
    float* part_o;            // [S][Hq][max_splits][D]       (unnormalised partial outputs)
    float2* part_ml;          // [S][Hq][max_splits] (m, l)   (running max in log2 units, sum)
    unsigned int* status;
    float scale_log2;         // scale * log2(e)
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int block_size;
    int num_blocks;
    int max_blocks_per_seq;
    int tokens_per_split;     // multiple of max(block_size, kStageTokens)
    int max_splits;
    int* seg_counters;        // persistent path: per-(sequence, kv head) arrival counters, zero between calls
    int num_ctas;             // persistent path: grid size
    unsigned long long* timeline;  // optional trace: [num_ctas][kTimelineSlots] (see pa.h); null = off
    const void* k_new;        // append mode: the new token's K and V rows [S][Hkv][D], written at
    const void* v_new;        //   position context_lens[s] - 1 before attention reads it; null = off
    int early;                // K/V of the first stages may be fetched before the preceding kernel ends
    int cut_unit, cut_seg;    // persistent path: weights of a chunk and of a segment end in the cut of the
                              // chunk list into CTA ranges (cut_seg == 0: equal chunk counts)
    const int32_t* q_start;   // several query tokens per sequence: rows q_start[s] .. q_start[s+1]-1 of q and
                              //   out (null: one query row per sequence, row s)
    int max_q;                // query tokens per sequence at most (1 without q_start)
    int q_rows;               // rows of q and out (several-token mode)
    const int32_t* runs;      // slotted mode (split CUDA-core kernel): [R][3] (block, slot_offset, length);
    const int32_t* seq_runs;  //   sequence s reads runs seq_runs[s] .. seq_runs[s+1]-1 in order; null = off
};

// Length of run r in slotted mode: 0 for a run that leaves its block or the pool.
__device__ __forceinline__ int run_len(const DecodeArgs& a, int r) {
    const int blk = a.runs[3 * r], off = a.runs[3 * r + 1], len = a.runs[3 * r + 2];
    const bool ok = blk >= 0 && blk < a.num_blocks && off >= 0 && len >= 0 && off + len <= a.block_size;
    return ok ? len : 0;
}

struct RowMoveArgs {
    const uint4* src_k;       // [src_blocks][Hkv][B][D] as 16-byte vectors
    const uint4* src_v;
    uint4* dst_k;             // [dst_blocks][Hkv][B][D]
    uint4* dst_v;
    const int32_t* moves;     // [M][5]: src_block, src_off, length, dst_block, dst_off
    unsigned int* status;
    int num_moves;
    int src_blocks;
    int dst_blocks;
    int num_kv_heads;
    int block_size;
    int vecs_per_row;         // D / 8
};

// New query tokens of sequence s (its newest ones, the last of its L cached tokens) and the
// first q / out row they occupy.  Out-of-range counts are clamped to [0, min(L, max_q)] (and to
// the rows of q) the same way wherever they are read.
struct QSpan {
    int row0;
    int n;
};

__device__ __forceinline__ QSpan q_span(const DecodeArgs& a, int s, int L) {
    if (!a.q_start) return QSpan{s, 1};
    const int r0 = max(0, min(a.q_start[s], a.q_rows));   // rows stay inside q and out
    const int n = a.q_start[s + 1] - a.q_start[s];
    return QSpan{r0, max(0, min(min(n, a.q_rows - r0), min(L, a.max_q)))};
}

// Element offset in q / out of row r of the segment (sequence s, kv head h): query token r / G
// of the span, group member r % G.
__device__ __forceinline__ size_t q_offset(const DecodeArgs& a, const QSpan& q, int h, int G, int r) {
    return ((size_t)(q.row0 + r / G) * a.num_q_heads + (size_t)h * G + r % G) * kHeadDim;
}

constexpr int kTimelineSlots = 16;

// ---------------------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<__half> {
    static __device__ __forceinline__ float2 to_float2(uint32_t u) {
        __half2 h = *reinterpret_cast<__half2*>(&u);
        return __half22float2(h);
    }
    static __device__ __forceinline__ float to_float(uint16_t u) {
        return __half2float(__ushort_as_half(u));
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
};

template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float2 to_float2(uint32_t u) {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
        return __bfloat1622float2(h);
    }
    static __device__ __forceinline__ float to_float(uint16_t u) {
        return __bfloat162float(__ushort_as_bfloat16(u));
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
};

template <typename T>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    float2 a = Elem<T>::to_float2(u.x), b = Elem<T>::to_float2(u.y);
    float2 c = Elem<T>::to_float2(u.z), d = Elem<T>::to_float2(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// ---------------------------------------------------------------------------------------
// Shared-memory barriers and bulk (TMA) copies, inline PTX
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// order this CTA's earlier generic-proxy shared-memory accesses before later async-proxy ones
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar`; false if it has not completed after ~kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// One contiguous global -> shared bulk copy completing on `bar` (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Programmatic dependent launch: wait for the preceding grid's results / let the next grid start.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Trace of the persistent kernel (slot layout documented with pa_decode_options in pa.h).
// trace: global time (ns) of an event of CTA `cta`; trace_put: any value.  Both no-ops when off.
__device__ __forceinline__ void trace_put(unsigned long long* tl, int cta, int slot, unsigned long long v) {
    if (tl) tl[(size_t)cta * kTimelineSlots + slot] = v;
}
__device__ __forceinline__ void trace(unsigned long long* tl, int cta, int slot) {
    if (tl) trace_put(tl, cta, slot, global_timer_ns());
}

__device__ __forceinline__ void flag_status(unsigned int* status, unsigned int bits) {
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---------------------------------------------------------------------------------------
// Host-side launch helpers (defined in the .cu files)
// ---------------------------------------------------------------------------------------
cudaError_t launch_cache_write(const CacheWriteArgs& a, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream);
cudaError_t launch_gather_runs(const RowMoveArgs& a, cudaStream_t stream);

// FMA (CUDA-core) split pass for group size G and element type; returns cudaErrorInvalidValue
// when G has no instantiation.
cudaError_t launch_decode_split_fma(const DecodeArgs& a, int dtype, int group, cudaStream_t stream);
cudaError_t launch_decode_combine(const DecodeArgs& a, int dtype, cudaStream_t stream);
bool fma_supports_group(int group);

// Persistent load-balanced tensor-core kernel (G <= 16, num_seqs <= kPersistMaxSeqs); one launch.
cudaError_t launch_decode_persist(const DecodeArgs& a, int dtype, cudaStream_t stream);
int persist_ctas_per_sm(int rows, int num_seqs);

// Several query tokens per sequence, any number: tiles of 64 query rows (prefill_mma.cu).
cudaError_t launch_prefill_mma(const DecodeArgs& a, int dtype, cudaStream_t stream);
// Several query tokens per sequence beyond 16 rows on tcgen05 tiles of 128 rows.
cudaError_t launch_prefill_tc(const DecodeArgs& a, int dtype, cudaStream_t stream);

// Planned decode (decode_planned.cu): the per-step plan and the per-layer launch that reads it.
constexpr int kPlanMaxSeqs = 1024;      // sequences the plan kernel keeps in shared memory
int planned_ctas(const pa_decode_options* opts);
size_t planned_plan_bytes(int num_seqs, int num_kv_heads, int block_size, int max_blocks_per_seq, int ctas,
                          bool adaptive);
size_t planned_workspace_bytes(int ctas);
size_t planned_runs_plan_bytes(int num_seqs, int num_kv_heads, int block_size, int max_blocks_per_seq, int ctas);
cudaError_t launch_decode_plan_runs(void* plan, const int32_t* runs, const int32_t* seq_runs, int num_seqs,
                                    int num_q_heads, int num_kv_heads, int block_size, int num_blocks,
                                    int max_blocks_per_seq, int max_context, int ctas, cudaStream_t stream);
cudaError_t launch_decode_planned_runs(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const void* plan, void* workspace, float scale, int num_seqs,
                                       int num_q_heads, int num_kv_heads, int block_size, int num_blocks,
                                       int max_blocks_per_seq, int dtype, int ctas, bool early,
                                       unsigned long long* timeline, cudaStream_t stream);
void planned_plan_offsets(int num_seqs, int num_kv_heads, int block_size, int max_blocks_per_seq, int ctas,
                          bool adaptive, size_t* bounds_offset, size_t* rates_offset);
cudaError_t launch_decode_plan(void* plan, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                               int num_q_heads, int num_kv_heads, int block_size, int num_blocks,
                               int max_blocks_per_seq, int ctas, bool adaptive, cudaStream_t stream);
cudaError_t launch_decode_planned(void* out, const void* q, const void* k_new, const void* v_new, const void* k_cache,
                                  const void* v_cache, void* plan, void* workspace, float scale, int num_seqs,
                                  int num_q_heads, int num_kv_heads, int block_size, int num_blocks,
                                  int max_blocks_per_seq, int dtype, int ctas, bool early, bool adaptive,
                                  unsigned long long* timeline, cudaStream_t stream);

// Tensor-core split pass (any G <= 16); builds the TMA tensor maps of the two caches.
cudaError_t launch_decode_split_mma(const DecodeArgs& a, int dtype, cudaStream_t stream);
bool mma_supports_group(int group);

// Where the persistent kernel keeps its arrival counters inside a workspace (api.cu).
bool persist_counter_region(int num_seqs, int num_kv_heads, int group, const pa_decode_options* opts,
                            size_t* offset, size_t* bytes);

// Launch-count bookkeeping (api.cu).
void note_launches(int n);

// SM count of the current device (api.cu; 152 when no device is visible).
int sm_count_current();

// Status word address on the current device (api.cu).
unsigned int* device_status_ptr();

}  // namespace pa
