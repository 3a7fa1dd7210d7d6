// Several new query tokens per sequence on the fifth-generation tensor cores: tcgen05.mma with
// Q, K and V in shared memory, the softmax weights P and the accumulators in tensor memory,
// tiles of 128 query rows.
//
// What it computes (the same as the persistent kernel's several-token mode and the mma.sync
// tiles): sequence s owns query rows q_start[s] .. q_start[s+1]-1, its n newest tokens, the last
// n of its L cached ones; token i sits at position L - n + i and attends causally over positions
// 0 .. L - n + i ("显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结", §五.1: walk the
// logical blocks through block_tables, q.k, running-max softmax, weight V, normalise; the
// chunked prefill of its closing section).
//
// One CTA per (256 query rows, kv head, sequence), two tiles of 128 rows; rows r = i * G + g (new
// token i, group member g); a tile stops at the last stage its rows see.  The CTAs of one
// (sequence, kv head) are adjacent in the grid, so they stream its K/V close together in time and
// share it through L2 (launching the longest CTAs first instead measured 1.3 % slower).
//   warps 0-3, 4-7  softmax of tile 0, tile 1: thread t owns row t of its tile (tensor-memory lane t)
//   warp 8          producer: TMA copies of 64-token K and V stages into a 4-deep ring
//   warps 9, 10     MMA of tile 0, tile 1 (warp 9 allocates tensor memory); one thread each issues,
//                   per stage j,
//                     S_j  = Q K_j^T   (M 128, N 64, K 128: 8 MMAs, K-major operands in shared memory)
//                     O   += P_j V_j   (M 128, N 128, K 64: 4 MMAs, P K-major in tensor memory, V
//                                       N-major in shared memory)
//                   and the two tiles share every K and V stage.
// Tensor memory per tile: one 64-column S buffer, 64 columns of P, a 128-column O.  The softmax
// releases S_j as soon as its registers hold it (an mbarrier the issuer waits on), so S_{j+1} is
// computed under the softmax of S_j; P_j goes to its own columns (fp16: two 32-column buffers
// taken in turn; bf16: one buffer, the high part and the low part side by side), each reused only
// after the PV product that last read it has completed (its mbarrier): MMAs into different
// accumulators are not ordered by issue alone.
// The softmax keeps a lazy exponent base per row (moved to the running max only when a score
// exceeds it by more than 2^8, then O is rescaled in tensor memory), writes P = exp2(s - base)
// (bf16 as a high and a low part, two MMAs) and at the end normalises its O row.  Every wait is
// bounded; tensor memory is freed on every path.
#include "pa_internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <type_traits>

namespace pa {

namespace {

constexpr int kTRows = 128;                                  // query rows per tile: the MMA's M
constexpr int kTiles = 2;                                    // tiles per CTA, one softmax warpgroup each
constexpr int kCtaRows = kTiles * kTRows;
constexpr int kSoftWarps = 4 * kTiles;                       // one row per thread
constexpr int kProdWarp = kSoftWarps;
constexpr int kMmaWarp = kSoftWarps + 1;                     // + t: the MMA issuer of tile t
constexpr int kTThreads = (kSoftWarps + 1 + kTiles) * 32;
constexpr uint32_t kQHalf = kTRows * 128;                    // 16 KB: 128 rows x 64 dims
constexpr uint32_t kQTile = 2 * kQHalf;
constexpr uint32_t kKVHalf = kStageTokens * 128;             // 8 KB: 64 tokens x 64 dims
constexpr uint32_t kKBytes = 2 * kKVHalf;                    // 16 KB of K per stage (V the same)
constexpr uint32_t kStage = 2 * kKBytes;
constexpr uint32_t kOffQ = 0;                                // [tile][2 halves][128 rows][128 B]
constexpr uint32_t kOffRing = kTiles * kQTile;               // [stage][K, V][2 halves][64 tokens][128 B]
constexpr int kTStages = 4;                                  // Q 64 KB + 4 x 32 KB ring (5 measured 1 % slower)
constexpr int kNumBars = 2 * kTStages + 12 + kTiles + 1;
constexpr uint32_t kOffBar = kOffRing + kTStages * kStage;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;        // tensor-memory address, abort flag, issued count
constexpr size_t kSmemTc = 1024 /*alignment slack*/ + kOffMisc + 16;
static_assert(kSmemTc <= 227 * 1024, "one CTA's shared memory must fit in 227 KB");
constexpr uint32_t kTmemCols = 512;                          // per tile: S at +0, P at +64, O at +128
constexpr uint32_t kTileCols = 256;
constexpr uint32_t kColP = 64;    // fp16: P buffers at +64, +96; bf16: one buffer, high +64, low +96
constexpr uint32_t kColO = 128;
constexpr float kLazyLog2 = 8.f;                             // exponent-base slack (weights below 2^8)

struct TcMaps {
    CUtensorMap k;
    CUtensorMap v;
};

// Shared-memory matrix descriptor of a 128-byte-swizzled operand: start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, swizzle mode 2 (128 bytes).
// K-major tiles (rows of 64 16-bit elements): stride 1024 between groups of 8 rows, leading
// offset unused.  N-major tiles (V: rows of 64 dims per token): leading offset = the distance
// between the two 64-dim halves, stride 1024 between groups of 8 tokens.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both f16 or both bf16, A
// K-major, B K-major or N-major, M = 128, N = n.
template <typename T>
__host__ __device__ constexpr uint32_t idesc(int n, bool b_n_major) {
    return (1u << 4) | ((std::is_same<T, __nv_bfloat16>::value ? 1u : 0u) << 7) |
           ((std::is_same<T, __nv_bfloat16>::value ? 1u : 0u) << 10) | ((b_n_major ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTRows >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t id,
                                     uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(id), "r"(accumulate)
        : "memory");
}

// The same with A in tensor memory: row m of A in lane m, two 16-bit elements per 32-bit column
// (the lower k in the low half), K-major.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t id,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(id), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread has issued so far is complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's tensor-memory lane, one load.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,"
        "%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

// 2^x on the special-function unit (approximate, subnormal results flushed to zero): the
// softmax weights it produces lie in (0, 2^8], and weights below 2^-126 do not matter.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 lanes per instruction (the packed forms of the Blackwell FP32 pipe; each lane rounds
// as the scalar instruction does) and a three-input maximum.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("{\n.reg .b64 ra, rb, rc;\nmov.b64 ra, {%1, %2};\nmov.b64 rb, {%3, %4};\nmov.b64 rc, {%5, %6};\n"
        "fma.rn.f32x2 %0, ra, rb, rc;\n}"
        : "=l"(d)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
    return r;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    uint64_t d;
    asm("{\n.reg .b64 ra, rb;\nmov.b64 ra, {%1, %2};\nmov.b64 rb, {%3, %4};\nadd.rn.f32x2 %0, ra, rb;\n}"
        : "=l"(d)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
    return r;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Copies of one stage: the blocks holding tokens [base, min(base + 64, tok_end)), K and V,
// each 64-dim half of a block to [half][token] of the stage (tokens contiguous per half).
__device__ __forceinline__ void issue_stage(const DecodeArgs& a, const TcMaps& maps, const int32_t* table_row,
                                            int hk, int base, int tok_end, uint32_t kdst, uint64_t* bar,
                                            int R_log2) {
    const int B = a.block_size;
    const int R = 1 << R_log2;
    const int first = base / B;
    const int last = (min(base + kStageTokens, tok_end) - 1) / B;
    const int within = (B > kStageTokens) ? (base % B) : 0;
    int phys[4];
    uint32_t bytes = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        phys[j] = -1;
        if (first + j <= last) {
            const int p = table_row[first + j];
            if (p >= 0 && p < a.num_blocks) {
                phys[j] = p;
                bytes += 4u * (uint32_t)R * 128u;   // K and V, two 64-dim halves
            } else {
                flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
            }
        }
    }
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (phys[j] >= 0) {
            const int row = (phys[j] * a.num_kv_heads + hk) * B + within;
            const uint32_t off = (uint32_t)(j * R) * 128u;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tma_load_2d(kdst + h * kKVHalf + off, &maps.k, 64 * h, row, bar);
                tma_load_2d(kdst + kKBytes + h * kKVHalf + off, &maps.v, 64 * h, row, bar);
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kTThreads, 1)
    prefill_tc_kernel(const DecodeArgs a, const __grid_constant__ TcMaps maps, const int R_log2) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // 1024-aligned for the swizzle
    unsigned char* bp = smem_raw + (base - raw);
    constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
    uint64_t* bars = reinterpret_cast<uint64_t*>(bp + kOffBar);
    uint64_t* kv_full = bars;                    // [stage] a stage's K and V landed
    uint64_t* kv_empty = bars + kTStages;        // [stage] the MMAs reading a stage are done
    uint64_t* s_full = bars + 2 * kTStages;      // [tile] S_j of the tile is in tensor memory (phase j)
    uint64_t* s_free = s_full + 2;               // [tile] the softmax holds S_j in registers (4 warps)
    uint64_t* p_full = s_full + 4;               // [tile][2] P_j of the tile is in tensor memory (128 arrivals)
    uint64_t* pv_done = p_full + 4;              // [tile][2] O += P_j V_j of the tile is complete
    uint64_t* q_ready = pv_done + 4;             // [tile] the tile's Q rows are in shared memory (128 arrivals)
    uint64_t* drain = q_ready + kTiles;          // every MMA issued is complete
    volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(bp + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bp + kOffMisc + 4);
    volatile int* issued_count = abort_flag + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta_tile = blockIdx.x, hk = blockIdx.y, s = blockIdx.z;
    const int G = a.num_q_heads / a.num_kv_heads;
    const int cap = a.max_blocks_per_seq * a.block_size;

    grid_dependency_wait();
    int L = a.context_lens[s];
    if (L < 0 || L > cap) {
        if (tid == 0 && cta_tile == 0 && hk == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
        L = L < 0 ? 0 : cap;
    }
    if (tid == 0 && cta_tile == 0 && hk == 0) {
        const int n_raw = a.q_start[s + 1] - a.q_start[s];
        const int r0_raw = a.q_start[s];
        if (n_raw < 0 || n_raw > L || n_raw > a.max_q || r0_raw < 0 || r0_raw + n_raw > a.q_rows)
            flag_status(a.status, PA_DEV_BAD_CONTEXT);
    }
    const QSpan qs = q_span(a, s, L);
    const int rows = qs.n * G;
    const int r0 = cta_tile * kCtaRows;
    if (r0 >= rows) return;   // uniform for the CTA, before any tensor memory is held
    const int ntiles = min(kTiles, (rows - r0 + kTRows - 1) / kTRows);   // tiles with rows (1 or 2)
    const int r_last = min(r0 + kCtaRows, rows) - 1;
    const int t_end = L - qs.n + r_last / G + 1;   // tokens the CTA needs: up to its last row's position
    const int nst = (t_end + kStageTokens - 1) / kStageTokens;
    // stages tile t needs (up to its own last row's position; the last tile needs all nst), so a
    // tile skips the stages its causal limits mask whole
    auto tile_stages = [&](int t) {
        const int te = L - qs.n + (min(r0 + (t + 1) * kTRows, rows) - 1) / G + 1;
        return (te + kStageTokens - 1) / kStageTokens;
    };

    if (tid == 0) {
        prefetch_map(&maps.k);
        prefetch_map(&maps.v);
        for (int i = 0; i < kTStages; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], ntiles);   // one commit per tile's issuer
        }
        for (int b = 0; b < 2 * kTiles; ++b) {
            if (b < kTiles) {
                mbar_init(&s_full[b], 1);
                mbar_init(&s_free[b], 4);
            }
            mbar_init(&p_full[b], 128);
            mbar_init(&pv_done[b], 1);
        }
        for (int t = 0; t < kTiles; ++t) mbar_init(&q_ready[t], 128);
        mbar_init(drain, ntiles);
        *abort_flag = 0;
        *issued_count = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(
                         const_cast<uint32_t*>(tslot))),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    grid_launch_dependents();

    auto give_up = [&]() {
        flag_status(a.status, PA_DEV_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == kProdWarp) {
        // ---------------- producer: one lane keeps the ring full ----------------
        if (lane == 0) {
            const int32_t* table_row = a.block_tables + (size_t)s * a.max_blocks_per_seq;
            int i = 0;
            for (; i < nst; ++i) {
                const int st = i % kTStages;
                if (i >= kTStages && !mbar_wait_bounded(&kv_empty[st], (uint32_t)((i / kTStages) - 1) & 1u)) {
                    give_up();
                    break;
                }
                if (*abort_flag) break;
                issue_stage(a, maps, table_row, hk, i * kStageTokens, t_end, base + kOffRing + (uint32_t)st * kStage,
                            &kv_full[st], R_log2);
            }
            *issued_count = i;
        }
    } else if (warp >= kMmaWarp && warp < kMmaWarp + kTiles) {
        // ---------------- MMA issue: one thread per tile, in warps on different schedulers ----------------
        const int mt = warp - kMmaWarp;   // this issuer's tile
        if (lane == 0 && mt < ntiles) {
            constexpr uint32_t kIdS = idesc<T>(kStageTokens, false);
            constexpr uint32_t kIdPV = idesc<T>(kHeadDim, true);
            // descriptors of each operand region's first 16-byte unit; an MMA's operand is that plus
            // its byte offset / 16 (every address stays below 256 KB, inside the 14-bit field)
            const uint64_t dq0 = sdesc(base + kOffQ, 16, 1024);
            const uint64_t dk0 = sdesc(base + kOffRing, 16, 1024);
            const uint64_t dv0 = sdesc(base + kOffRing + kKBytes, kKVHalf, 1024);
            const int my_nst = tile_stages(mt);
            bool ok = mbar_wait_bounded(&q_ready[mt], 0u);
            tc_fence_after();
            // S_j = Q K_j^T of the tile into its S buffer: two 64-dim halves x four 16-dim steps
            auto issue_s = [&](int j) -> bool {
                const int st = j % kTStages;
                if (!mbar_wait_bounded(&kv_full[st], (uint32_t)(j / kTStages) & 1u)) return false;
                // S_j overwrites S_{j-1}: only once the softmax holds that in registers
                if (j >= 1 && !mbar_wait_bounded(&s_free[mt], (uint32_t)(j - 1) & 1u)) return false;
                tc_fence_after();
                const uint64_t dk = dk0 + (uint64_t)(((uint32_t)st * kStage) >> 4);
                {
                    const int t = mt;
                    const uint32_t d = tmem + (uint32_t)t * kTileCols;
                    const uint64_t dq = dq0 + (uint64_t)(((uint32_t)t * kQTile) >> 4);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma(d, dq + (uint64_t)((h * kQHalf + kk * 32) >> 4), dk + (uint64_t)((h * kKVHalf + kk * 32) >> 4),
                                 kIdS, (h | kk) != 0 ? 1u : 0u);
                    umma_commit(&s_full[t]);
                }
                return true;
            };
            if (!ok) give_up();
            if (ok && !*abort_flag) ok = issue_s(0);
            for (int j = 0; j < my_nst && ok; ++j) {
                if (*abort_flag) break;
                if (j + 1 < my_nst && !issue_s(j + 1)) {
                    ok = false;
                    break;
                }
                // O += P_j V_j of the tile: four 16-token steps (and the low part of P for bf16)
                const uint64_t dv = dv0 + (uint64_t)(((uint32_t)(j % kTStages) * kStage) >> 4);
                {
                    const int t = mt;
                    if (!mbar_wait_bounded(&p_full[t * 2 + (j & 1)], (uint32_t)(j >> 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    // the last stage's V rows past the context are zeroed by the last tile's softmax
                    // before its P arrives
                    if (t != ntiles - 1 && j == nst - 1 &&
                        !mbar_wait_bounded(&p_full[(ntiles - 1) * 2 + (j & 1)], (uint32_t)(j >> 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // P_j in its own columns: 8 columns per 16 tokens (bf16: the low part 32 columns on)
                    const uint32_t pt = tmem + (uint32_t)t * kTileCols + kColP + (kSplitP ? 0u : (uint32_t)(j & 1) * 32u);
                    const uint32_t o = tmem + (uint32_t)t * kTileCols + kColO;
#pragma unroll
                    for (int kt = 0; kt < 4; ++kt) {
                        const uint64_t vd = dv + (uint64_t)((kt * 2048) >> 4);
                        umma_ts(o, pt + (uint32_t)(kt * 8), vd, kIdPV, (j > 0 || kt > 0) ? 1u : 0u);
                        if (kSplitP) umma_ts(o, pt + 32u + (uint32_t)(kt * 8), vd, kIdPV, 1u);
                    }
                    umma_commit(&pv_done[t * 2 + (j & 1)]);
                }
                if (ok) umma_commit(&kv_empty[j % kTStages]);
            }
            // the stages past this tile's last row: nothing to read, the stage's release is a plain
            // arrival (once the stage holds them, i.e. its previous use is released)
            for (int j = my_nst; j < nst && ok; ++j) {
                if (*abort_flag) break;
                if (!mbar_wait_bounded(&kv_full[j % kTStages], (uint32_t)(j / kTStages) & 1u)) {
                    ok = false;
                    break;
                }
                mbar_arrive(&kv_empty[j % kTStages]);
            }
            if (!ok) give_up();
            // nothing of this CTA's may still run on the tensor cores when it frees its memory
            umma_commit(drain);
            (void)mbar_wait_bounded(drain, 0u);
        }
    } else if (warp / 4 < ntiles) {
        // ------- softmax: warpgroup t owns tile t; thread wt owns its row wt (tensor-memory lane wt) -------
        const int t = warp / 4, wt = tid - t * 128;
        const int r = r0 + t * kTRows + wt;
        const bool row_ok = r < rows;
        const int lim = row_ok ? L - qs.n + r / G : -1;   // newest position the row attends to
        const uint32_t lane_addr = tmem + (uint32_t)t * kTileCols + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t sw = (uint32_t)(wt & 7);           // 128-byte swizzle phase of this row
        uint64_t* t_s_full = s_full + t;
        uint64_t* t_p_full = p_full + 2 * t;
        uint64_t* t_pv_done = pv_done + 2 * t;
        // Q row into the K-major operand tile (two 64-dim halves); rows past the segment are zero
        {
            const uint4* src = row_ok ? reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) +
                                                                      q_offset(a, qs, hk, G, r))
                                      : nullptr;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(base + kOffQ + t * kQTile + h * kQHalf + wt * 128 + ((c ^ sw) << 4),
                                 row_ok ? src[h * 8 + c] : make_uint4(0, 0, 0, 0));
        }
        fence_proxy_async_smem();
        mbar_arrive(&q_ready[t]);

        // waits and give-ups are decided per warp: the tensor-memory accesses are warp-wide
        auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
        };
        const float sl = a.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool dead = false;
        const int my_nst = tile_stages(t);
        for (int j = 0; j < my_nst && !dead; ++j) {
            if (__any_sync(0xffffffffu, *abort_flag != 0) || !warp_wait(t_s_full, (uint32_t)j & 1u)) {
                dead = true;
                break;
            }
            tc_fence_after();
            float x[64];
            tmem_ld64(lane_addr, x);
            // S_j is in registers: the buffer may take S_{j+1}
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[t]);
            const int t0 = j * kStageTokens;
            // raw scores; the scale (log2 units) enters the exponent's FMA.  Stages every row of the
            // warp sees whole skip the causal mask.
            if (!__all_sync(0xffffffffu, t0 + kStageTokens - 1 <= lim)) {
#pragma unroll
                for (int c = 0; c < 64; ++c) x[c] = (t0 + c <= lim) ? x[c] : -INFINITY;
            }
            // maximum as a tree (eight independent chains of three-input steps), not one 64-long
            // dependency chain
            float m8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float m = fmax3(x[e], x[e + 8], x[e + 16]);
                m = fmax3(m, x[e + 24], x[e + 32]);
                m = fmax3(m, x[e + 40], x[e + 48]);
                m8[e] = fmaxf(m, x[e + 56]);
            }
            float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
            if (sl > 0.f) {
                mx *= sl;   // the scaled maximum (-inf stays)
            } else {
                // a non-positive scale reverses the order: scale first, then take the maximum
                mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    x[c] = (x[c] == -INFINITY) ? -INFINITY : x[c] * sl;
                    mx = fmaxf(mx, x[c]);
                }
            }
            const float xs = (sl > 0.f) ? sl : 1.f;   // the factor still to apply to x
            if (j == nst - 1 && t == ntiles - 1) {
                // the last stage: V rows from t_end on are masked, but they can hold pool slots past
                // the context or stale data; zero them so that P = 0 never meets a non-finite V
                // (the last tile does it before its P arrives, which every issuer that reaches the
                // last stage waits for)
                const int nvalid = t_end - t0;
                const uint32_t vst = base + kOffRing + (uint32_t)(j % kTStages) * kStage + kKBytes;
                for (int idx = wt; idx < (kStageTokens - nvalid) * 16; idx += 128) {
                    const int t = nvalid + (idx >> 4);
                    st_shared_v4(vst + ((idx >> 3) & 1) * kKVHalf + t * 128 + (idx & 7) * 16, make_uint4(0, 0, 0, 0));
                }
            }
            // Exponent base: moved to the running max only when a score passes it by more than
            // kLazyLog2; O (which then holds stages 0 .. j-1) is rescaled in tensor memory.
            const bool move = mx > m_run + kLazyLog2;
            if (__any_sync(0xffffffffu, move && j > 0 && m_run != -INFINITY)) {
                // some row of the warp rescales O, which holds stages 0 .. j-1: wait (warp-wide) for
                // O += P_{j-1} V_{j-1}; tensor-memory accesses are warp-wide, so every lane scales
                // its O row (by 1 where the base stays)
                if (!warp_wait(&t_pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u)) {
                    dead = true;
                    break;
                }
                tc_fence_after();
                const float alpha = (move && j > 0 && m_run != -INFINITY) ? exp2f(m_run - mx) : 1.f;
#pragma unroll
                for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
                    float o[32];
                    tmem_ld32(lane_addr + kColO + c0, o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] *= alpha;
                    tmem_st32(lane_addr + kColO + c0, o);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                l_run *= alpha;
            }
            if (move) m_run = mx;
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
            // P_j into its tensor-memory P buffer (fp16: two, alternating; bf16: one, high and low)
            float2 rs2[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};   // eight partial row sums
            uint32_t hi[32];
            uint32_t lo[kSplitP ? 32 : 1];
            const float2 xs2 = make_float2(xs, xs), nm2 = make_float2(-m_use, -m_use);
#pragma unroll
            for (int c2 = 0; c2 < 32; ++c2) {
                const float2 e2 = ffma2(make_float2(x[2 * c2], x[2 * c2 + 1]), xs2, nm2);
                const float p0 = ex2(e2.x);
                const float p1 = ex2(e2.y);
                rs2[c2 & 3] = fadd2(rs2[c2 & 3], make_float2(p0, p1));
                hi[c2] = Elem<T>::pack2(p0, p1);
                if (kSplitP) {
                    const float2 h = Elem<T>::to_float2(hi[c2]);
                    lo[kSplitP ? c2 : 0] = Elem<T>::pack2(p0 - h.x, p1 - h.y);
                }
            }
            // the P buffer was last read by O += P_{j-k} V_{j-k}, k = the number of buffers
            {
                const int k = kSplitP ? 1 : 2;
                if (j >= k && !warp_wait(&t_pv_done[(j - k) & 1], (uint32_t)((j - k) >> 1) & 1u)) {
                    dead = true;
                    break;
                }
                tc_fence_after();
            }
            const uint32_t pcol = lane_addr + kColP + (kSplitP ? 0u : (uint32_t)(j & 1) * 32u);
            tmem_st32u(pcol, hi);
            if (kSplitP) tmem_st32u(pcol + 32u, reinterpret_cast<const uint32_t (&)[32]>(lo));
            l_run += ((rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y)) + ((rs2[2].x + rs2[2].y) + (rs2[3].x + rs2[3].y));
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            if (j == nst - 1) fence_proxy_async_smem();   // the zeroed V rows are read by the tensor cores
            tc_fence_before();
            mbar_arrive(&t_p_full[j & 1]);
        }
        // ---- normalise and write the row ----
        if (!dead && warp_wait(&t_pv_done[(my_nst - 1) & 1], (uint32_t)((my_nst - 1) >> 1) & 1u)) {
            tc_fence_after();
            const float inv = 1.f / l_run;
            uint4* dst = row_ok ? reinterpret_cast<uint4*>(static_cast<T*>(a.out) + q_offset(a, qs, hk, G, r))
                                : nullptr;
#pragma unroll
            for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
                float o[32];
                tmem_ld32(lane_addr + kColO + c0, o);
                if (row_ok) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 u;
                        u.x = Elem<T>::pack2(o[q4 * 8 + 0] * inv, o[q4 * 8 + 1] * inv);
                        u.y = Elem<T>::pack2(o[q4 * 8 + 2] * inv, o[q4 * 8 + 3] * inv);
                        u.z = Elem<T>::pack2(o[q4 * 8 + 4] * inv, o[q4 * 8 + 5] * inv);
                        u.w = Elem<T>::pack2(o[q4 * 8 + 6] * inv, o[q4 * 8 + 7] * inv);
                        dst[c0 / 8 + q4] = u;
                    }
                }
            }
        } else {
            give_up();
        }
    }

    // ---- teardown: nothing in flight on the tensor cores or the copy engine, then free ----
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && tid == 0) {
        // let every copy still in flight land before the CTA's shared memory is released
        const int n = *issued_count;
        for (int st = 0; st < kTStages; ++st) {
            int last = -1;
            for (int i = st; i < n; i += kTStages) last = i;
            if (last >= 0) (void)mbar_wait_bounded(&kv_full[st], (uint32_t)(last / kTStages) & 1u);
        }
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::atomic<int> state{0};
    if (state.load() == 0) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
        state.store(1);
    }
    return fn;
}

// A pool as [rows][128] 16-bit elements, boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool tc_encode_map(const void* base, unsigned long long rows, int box_rows, CUtensorMap* out) {
    auto fn = tc_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(out, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
cudaError_t launch_tc(const DecodeArgs& a, const TcMaps& maps, int R_log2, cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    auto kernel = prefill_tc_kernel<T>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTc);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    const int G = a.num_q_heads / a.num_kv_heads;
    const long long tiles = ((long long)a.max_q * G + kCtaRows - 1) / kCtaRows;
    if (tiles > 0x7fffffffLL || a.num_kv_heads > 65535 || a.num_seqs > 65535) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, a.num_kv_heads, a.num_seqs);
    cfg.blockDim = dim3(kTThreads);
    cfg.dynamicSmemBytes = kSmemTc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, a, maps, R_log2);
    if (e == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_prefill_tc(const DecodeArgs& a, int dtype, cudaStream_t stream) {
    const int R = a.block_size < kStageTokens ? a.block_size : kStageTokens;
    int R_log2 = 0;
    while ((1 << R_log2) < R) ++R_log2;
    const unsigned long long rows = (unsigned long long)a.num_blocks * a.num_kv_heads * a.block_size;
    if (rows == 0 || rows > 0x7fffffffull) return cudaErrorInvalidValue;
    TcMaps maps;
    if (!tc_encode_map(a.k_cache, rows, R, &maps.k) || !tc_encode_map(a.v_cache, rows, R, &maps.v))
        return cudaErrorInvalidValue;
    return dtype == PA_BF16 ? launch_tc<__nv_bfloat16>(a, maps, R_log2, stream)
                            : launch_tc<__half>(a, maps, R_log2, stream);
}

}  // namespace pa
