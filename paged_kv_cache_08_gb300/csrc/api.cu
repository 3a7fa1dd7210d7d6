// libpa C ABI: argument checks, split planning, kernel dispatch, device status word.
#include <atomic>
#include <cstdint>
#include <cstring>

#include "pa_internal.cuh"

namespace pa {

// Per-device status word (static device memory, no allocation).  Kernels atomicOr
// PA_DEV_* bits into it when they skip an out-of-range access or give up a wait.
__device__ unsigned int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_launches{0};
std::atomic<unsigned int*> g_status_ptr[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return -1;
    }
    return dev;
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 152;  // no device visible: size plans for a GB300
    int n = g_sm_count[dev].load();
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    g_sm_count[dev].store(n);
    return n;
}

bool supported_block_size(int b) { return b == 16 || b == 32 || b == 64 || b == 128; }

// Split plan.  Sequences are split into runs of `tps` tokens (a multiple of the stage and of
// the block) so that about four CTAs per SM are available even when the batch is small; the
// floor of 256 tokens keeps the fp32 partials a few percent of the K/V bytes they summarise.
int plan_tps(int num_seqs, int num_kv_heads, int block_size, int max_blocks_per_seq,
             const pa_decode_options* opts) {
    const int unit = block_size > kStageTokens ? block_size : kStageTokens;
    const long long cap = (long long)max_blocks_per_seq * block_size;
    const long long cap_units = ((cap + unit - 1) / unit) * unit;
    const long long max_tps = (long long)kMaxTableSlice * block_size;  // table slice held in shared memory
    if (opts && opts->tokens_per_split > 0) {
        if (opts->tokens_per_split % unit || opts->tokens_per_split > max_tps) return PA_ERR_INVALID_ARG;
        return opts->tokens_per_split;
    }
    if (cap_units == 0) return unit;
    const long long pairs = (long long)num_seqs * num_kv_heads;
    const long long target = 4LL * sm_count();
    long long splits = pairs > 0 ? (target + pairs - 1) / pairs : 1;
    if (splits < 1) splits = 1;
    long long tps = (cap + splits - 1) / splits;
    if (tps < 256) tps = 256;
    tps = ((tps + unit - 1) / unit) * unit;
    if (tps > cap_units) tps = cap_units;
    if (tps > max_tps) tps = max_tps;
    return (int)tps;
}

int check_decode_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       int max_blocks_per_seq) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq < 0 || block_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
    if (head_dim != kHeadDim || !supported_block_size(block_size)) return PA_ERR_UNSUPPORTED;
    if ((long long)max_blocks_per_seq * block_size > (1LL << 30)) return PA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_kv_heads > 65535 || num_q_heads > 65535) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

size_t workspace_bytes_for(int num_seqs, int num_q_heads, int max_splits) {
    if (max_splits <= 1) return 0;
    const size_t n = (size_t)num_seqs * num_q_heads * max_splits;
    return n * (kHeadDim * sizeof(float) + sizeof(float2));
}

enum Path { kPathFma, kPathMmaSplit, kPathPersist };

// Which kernel serves (num_seqs, group, math); PA_ERR_UNSUPPORTED when none does.
int choose_path(int num_seqs, int group, int math, Path* path) {
    if (math == PA_MATH_AUTO) math = mma_supports_group(group) ? PA_MATH_MMA : PA_MATH_FMA;
    switch (math) {
        case PA_MATH_FMA:
            if (!fma_supports_group(group)) return PA_ERR_UNSUPPORTED;
            *path = kPathFma;
            return PA_OK;
        case PA_MATH_MMA:
            if (!mma_supports_group(group)) return PA_ERR_UNSUPPORTED;
            *path = num_seqs <= kPersistMaxSeqs ? kPathPersist : kPathMmaSplit;
            return PA_OK;
        case PA_MATH_MMA_SPLIT:
            if (!mma_supports_group(group)) return PA_ERR_UNSUPPORTED;
            *path = kPathMmaSplit;
            return PA_OK;
        default:
            return PA_ERR_INVALID_ARG;
    }
}

inline size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// Launches with early reads run back to back, and the block scheduler hands a launch's CTAs
// the slots of the previous launch's CTAs as they exit, in index order: with every slot of the
// two-per-SM grid taken, the last CTAs start only as the previous launch's slowest ones finish,
// with no time left to fill their ring before the dependency wait, and set the next launch's
// end.  Leaving a few slots free lets them start earlier (measured on the 24-layer chain of 64
// sequences: 304 CTAs 17.6 us per layer, 300 16.3, 288 16.1, 272 16.4; one launch alone changes
// by about 1 %).
constexpr int kEarlySpareSlots = 16;

int persist_ctas(int rows, int num_seqs, bool early, const pa_decode_options* opts) {
    if (opts && opts->num_ctas > 0) return opts->num_ctas;
    const int per_sm = persist_ctas_per_sm(rows, num_seqs);
    const int n = per_sm * sm_count();
    return (early && per_sm == 2 && n > 4 * kEarlySpareSlots) ? n - kEarlySpareSlots : n;
}

// CTA count the workspace layout is sized for: the requested count, or the largest default
// grid (two CTAs per SM) whatever the group size, so that one workspace serves every shape.
int persist_layout_ctas(const pa_decode_options* opts) {
    if (opts && opts->num_ctas > 0) return opts->num_ctas;
    return 2 * sm_count();
}

// Persistent-path workspace: [C][2][16][D] fp32 partial outputs, [C][2][16] (m, l), then one
// arrival counter per (sequence, kv head).  Pieces are sized for the largest group so that the
// counters start at an offset that depends on the CTA count alone: a workspace keeps its zeroed
// counters across calls of any shape that use the same CTA count.
// Pieces of the persistent kernel: at most two per CTA (its first and its last sequence).
inline size_t persist_pieces(int ctas) { return (size_t)ctas * 2 * kPieceRows; }

size_t persist_workspace_bytes(int num_seqs, int num_kv_heads, int group, int ctas) {
    (void)group;
    const size_t pieces = persist_pieces(ctas);
    return align256(pieces * kHeadDim * sizeof(float)) + align256(pieces * sizeof(float2)) +
           align256((size_t)num_seqs * num_kv_heads * sizeof(int));
}

int max_splits_for(int block_size, int max_blocks_per_seq, int tps) {
    const long long cap = (long long)max_blocks_per_seq * block_size;
    long long n = (cap + tps - 1) / tps;
    return n < 1 ? 1 : (int)n;
}

}  // namespace

void note_launches(int n) { g_launches.fetch_add((uint64_t)n); }

int sm_count_current() { return sm_count(); }

bool persist_counter_region(int num_seqs, int num_kv_heads, int group, const pa_decode_options* opts,
                            size_t* offset, size_t* bytes) {
    (void)group;
    const size_t pieces = persist_pieces(persist_layout_ctas(opts));
    *offset = align256(pieces * kHeadDim * sizeof(float)) + align256(pieces * sizeof(float2));
    *bytes = (size_t)num_seqs * num_kv_heads * sizeof(int);
    return true;
}

unsigned int* device_status_ptr() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    unsigned int* p = g_status_ptr[dev].load();
    if (p) return p;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    p = static_cast<unsigned int*>(addr);
    g_status_ptr[dev].store(p);
    return p;
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_POOL_EXHAUSTED: return "block pool exhausted";
        case PA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case PA_ERR_BOUNDS: return "index out of bounds";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than pa_decode_static's fixed array holds";
        default: return "unknown status";
    }
}

uint64_t pa_kernel_launch_count(void) { return g_launches.load(); }

int pa_read_device_status(void* stream, int clear, uint32_t* bits) {
    if (!bits) return PA_ERR_INVALID_ARG;
    unsigned int* p = device_status_ptr();
    if (!p) return PA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int v = 0;
    if (cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return PA_ERR_CUDA;
    if (clear && cudaMemsetAsync(p, 0, sizeof(unsigned int), st) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
    *bits = v;
    return PA_OK;
}

int pa_cache_write(const void* k, const void* v, const int64_t* slot_mapping, void* k_cache, void* v_cache,
                   int num_tokens, int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype,
                   void* stream) {
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 || block_size <= 0 ||
        num_blocks < 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    CacheWriteArgs a;
    a.k = static_cast<const uint4*>(k);
    a.v = static_cast<const uint4*>(v);
    a.slots = slot_mapping;
    a.k_cache = static_cast<uint4*>(k_cache);
    a.v_cache = static_cast<uint4*>(v_cache);
    a.status = device_status_ptr();
    a.vecs_per_row = head_dim / 8;
    a.total_vecs = (long long)num_tokens * num_kv_heads * a.vecs_per_row;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.pool_slots = (long long)num_blocks * block_size;
    if ((a.total_vecs + 255) / 256 > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    cudaError_t e = launch_cache_write(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

// Device address of memory the kernels may touch: device memory as it is, pinned (page-locked,
// mapped) host memory translated to its device view; nullptr for pageable host memory.
static const void* device_view(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    switch (at.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            return p;
        case cudaMemoryTypeHost:
            return at.devicePointer;
        default:
            return nullptr;
    }
}

int pa_gather_runs(const void* src_k, const void* src_v, int src_blocks, void* dst_k, void* dst_v, int dst_blocks,
                   const int32_t* moves, int num_moves, int num_kv_heads, int head_dim, int block_size, int dtype,
                   void* stream) {
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (num_moves < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 || block_size <= 0 || src_blocks < 0 ||
        dst_blocks < 0)
        return PA_ERR_INVALID_ARG;
    if (num_moves == 0) return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !moves) return PA_ERR_INVALID_ARG;
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v) || !aligned4(moves))
        return PA_ERR_INVALID_ARG;
    if ((long long)num_kv_heads * block_size * (head_dim / 8) > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    RowMoveArgs a;
    a.src_k = static_cast<const uint4*>(src_k);
    a.src_v = static_cast<const uint4*>(src_v);
    a.dst_k = static_cast<uint4*>(dst_k);
    a.dst_v = static_cast<uint4*>(dst_v);
    a.moves = moves;
    a.status = device_status_ptr();
    a.num_moves = num_moves;
    a.src_blocks = src_blocks;
    a.dst_blocks = dst_blocks;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.vecs_per_row = head_dim / 8;
    cudaError_t e = launch_gather_runs(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

// Slotted decode: the split CUDA-core kernel with its copies driven by runs.
static int runs_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_context,
                     int* tps, int* maxb, int* max_splits) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads || max_context < 0)
        return PA_ERR_INVALID_ARG;
    if (head_dim != kHeadDim || !supported_block_size(block_size)) return PA_ERR_UNSUPPORTED;
    if (!fma_supports_group(num_q_heads / num_kv_heads)) return PA_ERR_UNSUPPORTED;
    *maxb = (max_context + block_size - 1) / block_size;
    if ((long long)*maxb * block_size > (1LL << 30)) return PA_ERR_UNSUPPORTED;
    *tps = plan_tps(num_seqs, num_kv_heads, block_size, *maxb, nullptr);
    if (*tps <= 0) return PA_ERR_INVALID_ARG;
    *max_splits = max_splits_for(block_size, *maxb, *tps);
    return PA_OK;
}

static int planned_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int max_blocks_per_seq);

// A runs plan: the block-table plan's shapes, and a token table of num_seqs x max_context rows.
static int runs_planned_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              int max_blocks_per_seq) {
    int rc = planned_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq);
    if (rc != PA_OK) return rc;
    const long long stride = ((long long)max_blocks_per_seq * block_size + kStageTokens - 1) / kStageTokens * kStageTokens;
    if ((long long)num_seqs * stride > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// The one-shot pa_decode_runs on the planned kernel: its workspace holds the runs plan and the
// decode's partial slots.
static bool runs_one_shot(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int max_context, size_t* plan_bytes, size_t* total) {
    if (num_seqs <= 0 || max_context <= 0) return false;
    const int maxb = (max_context + block_size - 1) / block_size;
    if (runs_planned_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, maxb) != PA_OK) return false;
    const int ctas = planned_ctas(nullptr);
    *plan_bytes = planned_runs_plan_bytes(num_seqs, num_kv_heads, block_size, maxb, ctas);
    *total = ((*plan_bytes + 255) & ~size_t(255)) + planned_workspace_bytes(ctas);
    return true;
}

size_t pa_decode_runs_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                     int max_context) {
    int tps, maxb, ms;
    if (runs_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context, &tps, &maxb, &ms) != PA_OK)
        return 0;
    size_t pb, total;
    if (runs_one_shot(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context, &pb, &total))
        return total;
    return ms > 1 ? workspace_bytes_for(num_seqs, num_q_heads, ms) : 0;
}

int pa_decode_runs(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* runs,
                   const int32_t* seq_runs, float scale, int num_kv_heads, int num_seqs, int num_q_heads,
                   int head_dim, int block_size, int num_blocks, int max_context, int dtype, void* workspace,
                   size_t workspace_bytes, void* stream) {
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    int tps, maxb, ms;
    int rc = runs_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context, &tps, &maxb, &ms);
    if (rc != PA_OK) return rc;
    if (num_seqs == 0) return PA_OK;
    if (num_blocks <= 0 || !out || !q || !k_cache || !v_cache || !runs || !seq_runs) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned4(runs) ||
        !aligned4(seq_runs))
        return PA_ERR_INVALID_ARG;
    if ((long long)num_blocks * num_kv_heads * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    size_t pb, total;
    if (runs_one_shot(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context, &pb, &total)) {
        if (!workspace || workspace_bytes < total || !aligned16(workspace)) return PA_ERR_WORKSPACE;
        const int ctas = planned_ctas(nullptr);
        const int maxb = (max_context + block_size - 1) / block_size;
        void* plan = workspace;
        void* ws = static_cast<char*>(workspace) + ((pb + 255) & ~size_t(255));
        cudaError_t e = launch_decode_plan_runs(plan, runs, seq_runs, num_seqs, num_q_heads, num_kv_heads, block_size,
                                                num_blocks, maxb, max_context, ctas, st);
        if (e == cudaSuccess)
            e = launch_decode_planned_runs(out, q, k_cache, v_cache, plan, ws, scale, num_seqs, num_q_heads,
                                           num_kv_heads, block_size, num_blocks, maxb, dtype, ctas, false, nullptr, st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
        return PA_OK;
    }
    const size_t need = ms > 1 ? workspace_bytes_for(num_seqs, num_q_heads, ms) : 0;
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return PA_ERR_WORKSPACE;
    DecodeArgs a;
    std::memset(&a, 0, sizeof(a));
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.runs = runs;
    a.seq_runs = seq_runs;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.max_blocks_per_seq = maxb;
    a.tokens_per_split = tps;
    a.max_splits = ms;
    const size_t n_part = (size_t)num_seqs * num_q_heads * ms;
    a.part_o = need ? static_cast<float*>(workspace) : nullptr;
    a.part_ml = need ? reinterpret_cast<float2*>(static_cast<char*>(workspace) + n_part * kHeadDim * sizeof(float))
                     : nullptr;
    a.status = device_status_ptr();
    cudaError_t e = launch_decode_split_fma(a, dtype, num_q_heads / num_kv_heads, st);
    if (e == cudaSuccess && ms > 1) e = launch_decode_combine(a, dtype, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

int pa_copy_blocks(const void* src_k, const void* src_v, int src_blocks, void* dst_k, void* dst_v, int dst_blocks,
                   const int32_t* src_ids, const int32_t* dst_ids, int num_pairs, int num_kv_heads, int head_dim,
                   int block_size, int dtype, void* stream) {
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 || block_size <= 0 || src_blocks < 0 ||
        dst_blocks < 0)
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !src_ids || !dst_ids) return PA_ERR_INVALID_ARG;
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v) || !aligned4(src_ids) ||
        !aligned4(dst_ids))
        return PA_ERR_INVALID_ARG;
    CopyBlocksArgs a;
    a.src_k = static_cast<const uint4*>(device_view(src_k));
    a.src_v = static_cast<const uint4*>(device_view(src_v));
    a.dst_k = static_cast<uint4*>(const_cast<void*>(device_view(dst_k)));
    a.dst_v = static_cast<uint4*>(const_cast<void*>(device_view(dst_v)));
    a.src_ids = static_cast<const int32_t*>(device_view(src_ids));
    a.dst_ids = static_cast<const int32_t*>(device_view(dst_ids));
    if (!a.src_k || !a.src_v || !a.dst_k || !a.dst_v || !a.src_ids || !a.dst_ids) return PA_ERR_INVALID_ARG;
    a.status = device_status_ptr();
    a.vecs_per_block = (long long)num_kv_heads * block_size * (head_dim / 8);
    a.num_pairs = num_pairs;
    a.src_blocks = src_blocks;
    a.dst_blocks = dst_blocks;
    if (a.vecs_per_block > (1LL << 40) / num_pairs) return PA_ERR_UNSUPPORTED;
    cudaError_t e = launch_copy_blocks(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

int pa_decode_plan_tokens_per_split(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, int max_blocks_per_seq, const pa_decode_options* opts) {
    int rc = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq);
    if (rc != PA_OK) return rc;
    return plan_tps(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, opts);
}

size_t pa_decode_workspace_size_ex(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                   int max_blocks_per_seq, const pa_decode_options* opts) {
    if (check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq) != PA_OK)
        return 0;
    const int group = num_q_heads / num_kv_heads;
    Path path;
    if (choose_path(num_seqs, group, opts ? opts->math : PA_MATH_AUTO, &path) != PA_OK) return 0;
    if (path == kPathPersist)
        return persist_workspace_bytes(num_seqs, num_kv_heads, group, persist_layout_ctas(opts));
    int tps = plan_tps(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, opts);
    if (tps <= 0) return 0;
    return workspace_bytes_for(num_seqs, num_q_heads, max_splits_for(block_size, max_blocks_per_seq, tps));
}

int pa_decode_kernel_kind(int num_seqs, int num_q_heads, int num_kv_heads, const pa_decode_options* opts) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
    Path path;
    int rc = choose_path(num_seqs, num_q_heads / num_kv_heads, opts ? opts->math : PA_MATH_AUTO, &path);
    if (rc != PA_OK) return rc;
    return path == kPathFma ? PA_KERNEL_SPLIT_FMA : (path == kPathPersist ? PA_KERNEL_PERSISTENT_MMA
                                                                          : PA_KERNEL_SPLIT_MMA);
}

int pa_decode_workspace_init(void* workspace, size_t bytes, void* stream) {
    if (bytes == 0) return PA_OK;
    if (!workspace) return PA_ERR_INVALID_ARG;
    if (cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int max_blocks_per_seq) {
    return pa_decode_workspace_size_ex(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                       max_blocks_per_seq, nullptr);
}

static int decode_impl(void* out, const void* q, const void* k_new, const void* v_new, const void* k_cache,
                       const void* v_cache, const int32_t* block_tables, const int32_t* context_lens, float scale,
                       int num_kv_heads, int num_seqs, int num_q_heads, int head_dim, int block_size, int num_blocks,
                       int max_blocks_per_seq, int dtype, void* workspace, size_t workspace_bytes, void* stream,
                       const pa_decode_options* opts, const int32_t* q_start = nullptr, int max_q = 1,
                       int q_rows = 0) {
    const bool append = k_new != nullptr;
    const bool multi = q_start != nullptr;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    int rc = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq);
    if (rc != PA_OK) return rc;
    if (num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (opts && (opts->math < PA_MATH_AUTO || opts->math > PA_MATH_MMA_SPLIT || opts->num_ctas < 0))
        return PA_ERR_INVALID_ARG;
    if ((long long)num_blocks * num_kv_heads * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !block_tables || !context_lens || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned4(block_tables) || !aligned4(context_lens))
        return PA_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    Path path;
    rc = choose_path(num_seqs, group, opts ? opts->math : PA_MATH_AUTO, &path);
    if (rc != PA_OK) return rc;
    if (multi) {
        // several query tokens per sequence: the persistent kernel while a (sequence, kv head)
        // has at most 16 query rows, else tcgen05 tiles of 128 rows (or mma.sync tiles of 64 rows
        // on request), no workspace
        if (max_q < 1 || !aligned4(q_start)) return PA_ERR_INVALID_ARG;
        if ((long long)max_q * group > kPieceRows) {
            if (append) return PA_ERR_UNSUPPORTED;   // the tiles kernel writes no cache rows
            if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
            DecodeArgs a;
            std::memset(&a, 0, sizeof(a));
            a.out = out;
            a.q = q;
            a.k_cache = k_cache;
            a.v_cache = v_cache;
            a.block_tables = block_tables;
            a.context_lens = context_lens;
            a.scale_log2 = scale * 1.4426950408889634f;
            a.num_seqs = num_seqs;
            a.num_q_heads = num_q_heads;
            a.num_kv_heads = num_kv_heads;
            a.block_size = block_size;
            a.num_blocks = num_blocks;
            a.max_blocks_per_seq = max_blocks_per_seq;
            a.status = device_status_ptr();
            a.q_start = q_start;
            a.max_q = max_q;
            a.q_rows = q_rows;
            const bool mma_sync_tiles = opts && (opts->flags & PA_PREFILL_MMA_SYNC);
            const cudaError_t pe = mma_sync_tiles ? launch_prefill_mma(a, dtype, static_cast<cudaStream_t>(stream))
                                                  : launch_prefill_tc(a, dtype, static_cast<cudaStream_t>(stream));
            if (pe != cudaSuccess) {
                cudaGetLastError();
                return PA_ERR_CUDA;
            }
            return PA_OK;
        }
        if (path != kPathPersist) return PA_ERR_UNSUPPORTED;
    }
    if (append) {
        if (path != kPathPersist) return PA_ERR_UNSUPPORTED;
        if (!v_new || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_INVALID_ARG;
    }

    DecodeArgs a;
    std::memset(&a, 0, sizeof(a));
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;

    if (path == kPathPersist) {
        const bool early = append && opts && (opts->flags & PA_DECODE_EARLY_READS);
        const int ctas = persist_ctas(multi ? max_q * group : group, num_seqs, early, opts);
        const size_t need = persist_workspace_bytes(num_seqs, num_kv_heads, group, persist_layout_ctas(opts));
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_WORKSPACE;
        const size_t pieces = persist_pieces(persist_layout_ctas(opts));
        char* w = static_cast<char*>(workspace);
        a.part_o = reinterpret_cast<float*>(w);
        a.part_ml = reinterpret_cast<float2*>(w + align256(pieces * kHeadDim * sizeof(float)));
        a.seg_counters = reinterpret_cast<int*>(w + align256(pieces * kHeadDim * sizeof(float)) +
                                                align256(pieces * sizeof(float2)));
        a.num_ctas = ctas;
        a.timeline = opts ? opts->timeline : nullptr;
        a.k_new = k_new;
        a.v_new = v_new;
        a.early = early ? 1 : 0;
        a.q_start = q_start;
        a.max_q = multi ? max_q : 1;
        a.q_rows = q_rows;
        a.tokens_per_split = 0;
        a.max_splits = 1;
        a.status = device_status_ptr();
        e = launch_decode_persist(a, dtype, st);
    } else {
        const int tps = plan_tps(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, opts);
        if (tps <= 0) return PA_ERR_INVALID_ARG;
        const int max_splits = max_splits_for(block_size, max_blocks_per_seq, tps);
        const size_t need = workspace_bytes_for(num_seqs, num_q_heads, max_splits);
        if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return PA_ERR_WORKSPACE;
        const size_t n_part = (size_t)num_seqs * num_q_heads * max_splits;
        a.part_o = need ? static_cast<float*>(workspace) : nullptr;
        a.part_ml = need ? reinterpret_cast<float2*>(static_cast<char*>(workspace) +
                                                     n_part * kHeadDim * sizeof(float))
                         : nullptr;
        a.tokens_per_split = tps;
        a.max_splits = max_splits;
        a.status = device_status_ptr();
        e = path == kPathMmaSplit ? launch_decode_split_mma(a, dtype, st)
                                  : launch_decode_split_fma(a, dtype, group, st);
        if (e == cudaSuccess && max_splits > 1) e = launch_decode_combine(a, dtype, st);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

int pa_decode_ex(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                 const int32_t* context_lens, float scale, int num_kv_heads, int num_seqs, int num_q_heads,
                 int head_dim, int block_size, int num_blocks, int max_blocks_per_seq, int dtype, void* workspace,
                 size_t workspace_bytes, void* stream, const pa_decode_options* opts) {
    return decode_impl(out, q, nullptr, nullptr, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                       num_seqs, num_q_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, dtype, workspace,
                       workspace_bytes, stream, opts);
}

int pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                     const int32_t* block_tables, const int32_t* context_lens, float scale, int num_kv_heads,
                     int num_seqs, int num_q_heads, int head_dim, int block_size, int num_blocks,
                     int max_blocks_per_seq, int dtype, void* workspace, size_t workspace_bytes, void* stream,
                     const pa_decode_options* opts) {
    if (!k_new || !v_new) return PA_ERR_INVALID_ARG;
    return decode_impl(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                       num_seqs, num_q_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, dtype, workspace,
                       workspace_bytes, stream, opts);
}

int pa_multi_query(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                   const int32_t* context_lens, const int32_t* query_start, float scale, int num_kv_heads,
                   int num_seqs, int num_q_tokens, int max_q_per_seq, int num_q_heads, int head_dim, int block_size,
                   int num_blocks, int max_blocks_per_seq, int dtype, void* workspace, size_t workspace_bytes,
                   void* stream, const pa_decode_options* opts) {
    if (num_q_tokens < 0 || !query_start) return PA_ERR_INVALID_ARG;
    if (num_q_tokens == 0) return num_seqs >= 0 ? PA_OK : PA_ERR_INVALID_ARG;
    return decode_impl(out, q, nullptr, nullptr, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                       num_seqs, num_q_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, dtype, workspace,
                       workspace_bytes, stream, opts, query_start, max_q_per_seq, num_q_tokens);
}

int pa_multi_query_append(void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
                          void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                          const int32_t* query_start, float scale, int num_kv_heads, int num_seqs, int num_q_tokens,
                          int max_q_per_seq, int num_q_heads, int head_dim, int block_size, int num_blocks,
                          int max_blocks_per_seq, int dtype, void* workspace, size_t workspace_bytes, void* stream,
                          const pa_decode_options* opts) {
    if (num_q_tokens < 0 || !query_start || !k_new || !v_new) return PA_ERR_INVALID_ARG;
    if (num_q_tokens == 0) return num_seqs >= 0 ? PA_OK : PA_ERR_INVALID_ARG;
    return decode_impl(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                       num_seqs, num_q_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, dtype, workspace,
                       workspace_bytes, stream, opts, query_start, max_q_per_seq, num_q_tokens);
}

static bool plan_adaptive(const pa_decode_options* opts) { return opts && (opts->flags & PA_PLAN_ADAPTIVE); }
static bool plan_runs(const pa_decode_options* opts) { return opts && (opts->flags & PA_PLAN_RUNS); }

static int planned_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int max_blocks_per_seq) {
    int rc = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq);
    if (rc != PA_OK) return rc;
    if (num_q_heads / num_kv_heads > 8 || num_seqs > kPlanMaxSeqs || num_kv_heads > 32767) return PA_ERR_UNSUPPORTED;
    // chunk indices and counts per segment are 16-bit in the plan
    if ((long long)max_blocks_per_seq * block_size > 32767LL * kStageTokens) return PA_ERR_UNSUPPORTED;
    if ((long long)num_seqs * num_kv_heads * (((long long)max_blocks_per_seq * block_size + kStageTokens - 1) /
                                              kStageTokens) > 0x7fffffffLL)
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

size_t pa_decode_plan_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int max_blocks_per_seq, const pa_decode_options* opts) {
    if (planned_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq) != PA_OK)
        return 0;
    if (opts && opts->num_ctas < 0) return 0;
    if (plan_runs(opts)) {
        if (plan_adaptive(opts) ||
            runs_planned_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq) != PA_OK)
            return 0;
        return planned_runs_plan_bytes(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, planned_ctas(opts));
    }
    return planned_plan_bytes(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, planned_ctas(opts),
                              plan_adaptive(opts));
}

int pa_decode_plan_sections(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, const pa_decode_options* opts, int* num_ctas,
                            size_t* bounds_offset, size_t* rates_offset) {
    int rc = planned_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq);
    if (rc != PA_OK) return rc;
    if ((opts && opts->num_ctas < 0) || !num_ctas || !bounds_offset || !rates_offset) return PA_ERR_INVALID_ARG;
    *num_ctas = planned_ctas(opts);
    planned_plan_offsets(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, *num_ctas, plan_adaptive(opts),
                         bounds_offset, rates_offset);
    return PA_OK;
}

size_t pa_decode_planned_workspace_size(const pa_decode_options* opts) {
    if (opts && opts->num_ctas < 0) return 0;
    return planned_workspace_bytes(planned_ctas(opts));
}

int pa_decode_planned_workspace_init(void* workspace, size_t bytes, void* stream) {
    if (bytes == 0) return PA_OK;
    if (!workspace) return PA_ERR_INVALID_ARG;
    if (cudaMemsetAsync(workspace, 0xFF, bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

int pa_decode_plan(void* plan, size_t plan_bytes, const int32_t* block_tables, const int32_t* context_lens,
                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   int max_blocks_per_seq, void* stream, const pa_decode_options* opts) {
    int rc = planned_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq);
    if (rc != PA_OK) return rc;
    if ((opts && opts->num_ctas < 0) || plan_runs(opts)) return PA_ERR_INVALID_ARG;
    if (num_blocks <= 0 || !plan || !aligned16(plan)) return PA_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!block_tables || !context_lens || !aligned4(block_tables) || !aligned4(context_lens)))
        return PA_ERR_INVALID_ARG;
    const int ctas = planned_ctas(opts);
    if (plan_bytes <
        planned_plan_bytes(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas, plan_adaptive(opts)))
        return PA_ERR_WORKSPACE;
    cudaError_t e = launch_decode_plan(plan, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                                       block_size, num_blocks, max_blocks_per_seq, ctas,
                                       plan_adaptive(opts), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

int pa_decode_plan_runs(void* plan, size_t plan_bytes, const int32_t* runs, const int32_t* seq_runs, int num_seqs,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                        int max_context, void* stream, const pa_decode_options* opts) {
    if (max_context <= 0 || num_seqs <= 0) return PA_ERR_INVALID_ARG;
    const int maxb = (max_context + block_size - 1) / block_size;
    int rc = runs_planned_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, maxb);
    if (rc != PA_OK) return rc;
    if ((opts && opts->num_ctas < 0) || plan_adaptive(opts)) return PA_ERR_INVALID_ARG;
    if (num_blocks <= 0 || !plan || !aligned16(plan) || !runs || !seq_runs || !aligned4(runs) || !aligned4(seq_runs))
        return PA_ERR_INVALID_ARG;
    if ((long long)num_blocks * num_kv_heads * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    const int ctas = planned_ctas(opts);
    if (plan_bytes < planned_runs_plan_bytes(num_seqs, num_kv_heads, block_size, maxb, ctas)) return PA_ERR_WORKSPACE;
    cudaError_t e = launch_decode_plan_runs(plan, runs, seq_runs, num_seqs, num_q_heads, num_kv_heads, block_size,
                                            num_blocks, maxb, max_context, ctas, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

int pa_decode_planned(void* out, const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      void* plan, size_t plan_bytes, float scale, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, int max_blocks_per_seq, int dtype, void* workspace,
                      size_t workspace_bytes, void* stream, const pa_decode_options* opts) {
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    int rc = planned_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq);
    if (rc != PA_OK) return rc;
    if (opts && opts->num_ctas < 0) return PA_ERR_INVALID_ARG;
    if (num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if ((long long)num_blocks * num_kv_heads * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !plan) return PA_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(plan) ||
        !aligned16(k_new) || !aligned16(v_new))
        return PA_ERR_INVALID_ARG;
    const int ctas = planned_ctas(opts);
    const bool runs = plan_runs(opts);
    if (runs && (k_new != nullptr || plan_adaptive(opts))) return PA_ERR_INVALID_ARG;
    if (runs) {
        rc = runs_planned_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq);
        if (rc != PA_OK) return rc;
    }
    const size_t plan_need =
        runs ? planned_runs_plan_bytes(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas)
             : planned_plan_bytes(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas, plan_adaptive(opts));
    if (plan_bytes < plan_need) return PA_ERR_WORKSPACE;
    const size_t need = planned_workspace_bytes(ctas);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_WORKSPACE;
    const bool early = opts && (opts->flags & PA_DECODE_EARLY_READS);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e =
        runs ? launch_decode_planned_runs(out, q, k_cache, v_cache, plan, workspace, scale, num_seqs, num_q_heads,
                                          num_kv_heads, block_size, num_blocks, max_blocks_per_seq, dtype, ctas, early,
                                          opts ? opts->timeline : nullptr, st)
             : launch_decode_planned(out, q, k_new, v_new, k_cache, v_cache, plan, workspace, scale, num_seqs,
                                     num_q_heads, num_kv_heads, block_size, num_blocks, max_blocks_per_seq, dtype,
                                     ctas, early, plan_adaptive(opts), opts ? opts->timeline : nullptr, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              const int32_t* context_lens, float scale, int num_kv_heads, int num_seqs, int num_q_heads,
              int head_dim, int block_size, int num_blocks, int max_blocks_per_seq, int dtype, void* workspace,
              size_t workspace_bytes, void* stream) {
    return pa_decode_ex(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads, num_seqs,
                        num_q_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, dtype, workspace,
                        workspace_bytes, stream, nullptr);
}

}  // extern "C"
