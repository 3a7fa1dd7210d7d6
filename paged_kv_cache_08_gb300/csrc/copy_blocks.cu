// Whole-block copies between two pools: copy-on-write inside the cache, swap out to and back
// in from a pinned host pool.
//
// What it computes: "显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结", §四 -- when a
// sequence appends to a shared, unfilled last block, the block's contents are deep-copied into
// a freshly allocated block that the sequence then owns; its FAQ on preemption -- blocks of a
// low-priority request are moved to host memory and back.  "KV Cache 与 BlockManager" (§3.4)
// sizes that host buffer and asks for pinned memory.
//
// Design: a (block, pool) tile is num_kv_heads * block_size * head_dim contiguous elements,
// so a pair is two contiguous runs (K and V).  The grid strides over the 16-byte vectors of all
// pairs; each thread keeps four loads in flight before its stores.  A copy is bound by the
// slower side: HBM for device pools, the host link when one pool is in host memory.
#include "pa_internal.cuh"

namespace pa {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyBlocksArgs a) {
    grid_dependency_wait();   // the ids or the source rows may come from the preceding kernel
    const long long per_pair = 2 * a.vecs_per_block;   // K run, then V run
    const long long total = per_pair * a.num_pairs;
    const long long stride = (long long)gridDim.x * kCopyThreads;
    for (long long base = (long long)blockIdx.x * kCopyThreads + threadIdx.x; base < total;
         base += stride * kCopyUnroll) {
        uint4 val[kCopyUnroll];
        uint4* dst[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            dst[u] = nullptr;
            const long long i = base + u * stride;
            if (i >= total) continue;
            const int pair = (int)(i / per_pair);
            const long long r = i - (long long)pair * per_pair;
            const bool is_v = r >= a.vecs_per_block;
            const long long e = is_v ? r - a.vecs_per_block : r;
            const int s = a.src_ids[pair], d = a.dst_ids[pair];
            if (s < 0 || s >= a.src_blocks || d < 0 || d >= a.dst_blocks) {
                if (r == 0) flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
                continue;
            }
            const uint4* src = (is_v ? a.src_v : a.src_k) + (long long)s * a.vecs_per_block + e;
            val[u] = *src;
            dst[u] = (is_v ? a.dst_v : a.dst_k) + (long long)d * a.vecs_per_block + e;
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u)
            if (dst[u]) *dst[u] = val[u];
    }
    grid_launch_dependents();
}

// Row-run moves (online defragmentation of slotted blocks, "Slotted Block 分槽与微块共享架构" on
// the radix-tree fragmentation page): one CTA per move; its threads stride over the 16-byte
// vectors of the run's rows in every kv head.  A move that leaves a block or a pool is skipped
// and flagged.
__global__ void __launch_bounds__(kCopyThreads) gather_runs_kernel(const RowMoveArgs a) {
    grid_dependency_wait();
    const int m = blockIdx.x;
    const int sb = a.moves[5 * m], so = a.moves[5 * m + 1], len = a.moves[5 * m + 2];
    const int db = a.moves[5 * m + 3], dof = a.moves[5 * m + 4];
    const int B = a.block_size;
    if (sb < 0 || sb >= a.src_blocks || db < 0 || db >= a.dst_blocks || len < 0 || so < 0 || dof < 0 ||
        so + len > B || dof + len > B) {
        if (threadIdx.x == 0) flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
        return;
    }
    const int per_head = len * a.vecs_per_row;
    const int total = per_head * a.num_kv_heads;
    for (int e0 = threadIdx.x; e0 < total; e0 += kCopyThreads * kCopyUnroll) {
        uint4 kv[kCopyUnroll], vv[kCopyUnroll];
        long long dst[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int e = e0 + u * kCopyThreads;
            dst[u] = -1;
            if (e >= total) continue;
            const int h = e / per_head;
            const int w = e - h * per_head;   // vector within the head's run
            const long long s_vec = (((long long)sb * a.num_kv_heads + h) * B + so) * a.vecs_per_row + w;
            dst[u] = (((long long)db * a.num_kv_heads + h) * B + dof) * a.vecs_per_row + w;
            kv[u] = a.src_k[s_vec];
            vv[u] = a.src_v[s_vec];
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u)
            if (dst[u] >= 0) {
                a.dst_k[dst[u]] = kv[u];
                a.dst_v[dst[u]] = vv[u];
            }
    }
    grid_launch_dependents();
}

}  // namespace

cudaError_t launch_gather_runs(const RowMoveArgs& a, cudaStream_t stream) {
    if (a.num_moves == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.num_moves);
    cfg.blockDim = dim3(kCopyThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gather_runs_kernel, a);
    if (e == cudaSuccess) note_launches(1);
    return e;
}

cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream) {
    const long long total = 2 * a.vecs_per_block * a.num_pairs;
    if (total == 0) return cudaSuccess;
    // enough CTAs for every SM to hold several, no more than the work needs
    const long long need = (total + (long long)kCopyThreads * kCopyUnroll - 1) / ((long long)kCopyThreads * kCopyUnroll);
    const long long cap = (long long)sm_count_current() * 8;
    const unsigned blocks = (unsigned)(need < cap ? need : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kCopyThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, copy_blocks_kernel, a);
    if (e == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace pa
