// pa_decode_static: paged decode attention for callers that cannot allocate device memory.
//
// The scratch that pa_decode takes from the caller (partial results of sequences cut between
// CTAs, and their arrival counters) lives here in one file-scope device array.  Host code must
// not pass the array's name to a kernel: on the host it is only a stand-in symbol.  Its device
// address is looked up once per device with cudaGetSymbolAddress and cached.
#include <atomic>
#include <cstdint>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = PA_DECODE_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of this device's scratch array (nullptr when the lookup fails).
void* scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    void* p = g_scratch_addr[dev].load();
    if (p) return p;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return nullptr;
    }
    g_scratch_addr[dev].store(p);
    return p;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int pa_decode_static(void* out, const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens, float scale,
                                int num_kv_heads, int num_seqs, int num_q_heads, int head_dim, int block_size,
                                int num_blocks, int max_blocks_per_seq, int dtype, void* stream) {
    pa_decode_options opts = {0, PA_MATH_AUTO, 0, 0, nullptr};
    const int kind = pa_decode_kernel_kind(num_seqs, num_q_heads, num_kv_heads, &opts);
    if (kind < 0) return kind;
    const size_t need = pa_decode_workspace_size_ex(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                                    max_blocks_per_seq, &opts);
    if (need > kStaticScratchBytes) return PA_ERR_SCRATCH_LIMIT;
    void* scratch = scratch_address();
    if (!scratch) return PA_ERR_CUDA;
    if (kind == PA_KERNEL_PERSISTENT_MMA && num_seqs > 0) {
        // the arrival counters start at zero (a call that gave up may have left them dirty)
        size_t off = 0, bytes = 0;
        persist_counter_region(num_seqs, num_kv_heads, num_q_heads / num_kv_heads, &opts, &off, &bytes);
        if (bytes && cudaMemsetAsync(static_cast<char*>(scratch) + off, 0, bytes,
                                     static_cast<cudaStream_t>(stream)) != cudaSuccess) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
    }
    return pa_decode_ex(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads, num_seqs,
                        num_q_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, dtype, scratch,
                        kStaticScratchBytes, stream, &opts);
}
