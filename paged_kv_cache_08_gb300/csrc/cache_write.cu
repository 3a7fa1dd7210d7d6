// Paged cache write: scatter each new (token, kv-head) K/V row into its slot.
//
// What it computes: "显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结", §三 sequence
// diagram -- the new token lands at the next offset of the sequence's current block (or at
// offset 0 of a freshly appended one); the slot is physical_block * B + offset, the address
// rule of "端侧 SLM 显存保活术：在 4GB 内存板卡上实现轻量 PagedAttention 与 KV 缓存分块",
// section "注意力寻址：非连续物理块的间接寻址内核".
//
// Design: one thread per 16-byte vector of a row; 16 consecutive threads cover one
// 256-byte (token, head) row, so every warp moves two whole rows with full 128-byte
// transactions on both sides.  The same thread copies the K vector and the V vector.
// The work is a pure copy bound by HBM (or by launch latency for small batches).
#include "pa_internal.cuh"

namespace pa {

namespace {

__device__ __forceinline__ uint4 load_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__global__ void __launch_bounds__(256) cache_write_kernel(const CacheWriteArgs a) {
    grid_dependency_wait();  // inputs may come from the preceding kernel
    grid_launch_dependents();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.total_vecs) return;
    const int vec = (int)(i % a.vecs_per_row);
    const long long row = i / a.vecs_per_row;  // token * Hkv + head
    const int head = (int)(row % a.num_kv_heads);
    const long long token = row / a.num_kv_heads;
    const long long slot = a.slots[token];
    if (slot < 0) return;  // padding token
    if (slot >= a.pool_slots) {
        if (vec == 0 && head == 0) flag_status(a.status, PA_DEV_BAD_SLOT);
        return;
    }
    const long long blk = slot / a.block_size;
    const long long off = slot - blk * a.block_size;
    const long long dst = ((blk * a.num_kv_heads + head) * a.block_size + off) * a.vecs_per_row + vec;
    const uint4 kv = load_stream(a.k + i);
    const uint4 vv = load_stream(a.v + i);
    a.k_cache[dst] = kv;
    a.v_cache[dst] = vv;
}

}  // namespace

cudaError_t launch_cache_write(const CacheWriteArgs& a, cudaStream_t stream) {
    if (a.total_vecs == 0) return cudaSuccess;
    const int threads = 256;
    const long long blocks = (a.total_vecs + threads - 1) / threads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, cache_write_kernel, a);
    if (e == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace pa
