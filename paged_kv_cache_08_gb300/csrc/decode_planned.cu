// Paged decode attention with a per-step plan: one planning launch per decode step, then one
// decode launch per layer that reads the plan instead of the block tables.
//
// What it computes is pa_decode's (and, with the new K/V rows, pa_decode_append's):
// "显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结", §五.1 -- for every sequence and query
// head, walk the sequence's logical blocks through its block-table row, q.k for every cached
// token, softmax with a running maximum, weight V, normalise at the end; the address rule of
// "端侧 SLM 显存保活术：在 4GB 内存板卡上实现轻量 PagedAttention 与 KV 缓存分块", section
// "注意力寻址：非连续物理块的间接寻址内核".  Every layer of a decode step shares the block tables
// and the lengths, so everything derived from them alone is computed once per step:
//
// The plan (decode_plan_kernel).  A segment is one (sequence, kv head), cut into 64-token
// chunks; the chunks of all segments form one list (sequence-major, then kv head).  For every
// chunk the plan holds its sequence, kv head, position in the segment, valid tokens and the
// physical ids of the blocks it touches, read from the block table once.  The list is cut into
// 2C equal contiguous ranges, two per CTA (C CTAs, one per SM): group 0 of a CTA streams its
// range forwards, group 1 backwards.  So the range ends that border another CTA are streamed
// first by both CTAs, and a segment cut there leaves pieces that are done early; the cut between
// the two groups of one CTA is streamed last by both, and its two pieces meet in shared memory.
// For a segment cut between CTAs the plan names the CTA that combines the pieces (the merger):
// the first CTA whose piece finishes late (last in its group's order), else the first CTA.
//
// The decode launch (decode_planned_kernel), per CTA:
//   warps 0-3, 4-7  consumers of group 0, 1: each warp owns 16 tokens of a 64-token stage and
//                   runs S^T = K Q^T and O^T += V^T P^T on mma.sync m16n8k16 (the GQA group's
//                   query rows on the 8-column side), online softmax with a lazy exponent base;
//                   at a segment's end the four warps merge through the consumed stage and the
//                   result goes to the output, to the other group (shared memory), to the
//                   epilogue warp (shared memory) or, for another CTA's merger, to the workspace;
//   warps 8, 9      producers of group 0, 1: read the group's chunk descriptors from the plan
//                   (32 per load, one per lane) and issue the 2-D TMA copies (128-byte swizzle)
//                   of K and V, the query rows at a segment's first chunk and, when appending,
//                   the new token's K/V rows, into a 3-stage ring per group;
//   warp 10         epilogue: publishes this CTA's pieces of cut segments (a release store of a
//                   flag per piece after the consumers' partial stores) and, where this CTA is the
//                   merger, folds the other CTAs' pieces in as their flags appear, then its own,
//                   and writes the output.  The consumers never wait on another CTA.
// Every wait is bounded (about one second); a wait that gives up sets PA_DEV_TIMEOUT.
#include "decode_common.cuh"

#include <atomic>
#include <cstddef>
#include <cstring>
#include <climits>
#include <type_traits>

namespace pa {

namespace {

constexpr int kGroups = 2;
constexpr int kGroupWarps = 4;
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kConsWarps = kGroups * kGroupWarps;       // 8
constexpr int kProdWarp0 = kConsWarps;                  // producers: warps 8, 9
constexpr int kEpiWarp = kConsWarps + kGroups;          // 10
constexpr int kPThreads = (kEpiWarp + 1) * 32;          // 352
constexpr int kRows = 8;                                // query rows per segment (the GQA group, G <= 8)
constexpr int kRedStride = kHeadDim + 4;                // padded rows of the merge scratch
constexpr uint32_t kSlotB = kRows * kHeadDim * 4 + kRows * 8;   // partial (o rows, then (m, l) per row)
constexpr uint32_t kMiscB = 128;
// Runs stages: a chunk's 64 tokens as 8 octets of 8 consecutive tokens; octet k is 8 rows of 256
// bytes in a row at k * 2064 (16 bytes of pad per octet).  Staged row t (the consumers' index)
// holds token 8 (t mod 8) + t / 8, so the 8 rows one ldmatrix reads lie in 8 different octets,
// 16 bytes apart in the bank map (no conflict), and the rows of one octet, consecutive tokens, take
// one bulk copy wherever they are consecutive rows of the pool.
constexpr uint32_t kOctB = 8 * kHeadDim * 2 + 16;        // 2064

// Shared-memory layout of a decode CTA: per group 3 stages of 35 KB.  Block-table plans: K and V
// as TMA boxes with the 128-byte swizzle.  Runs plans (contexts given as slot runs): K and V as the
// quads above, filled by bulk copies; no new-token rows (runs plans do not append).
template <bool kRuns>
struct Lay {
    static constexpr int kPStages = 3;
    static constexpr uint32_t kKB = kRuns ? 8 * kOctB : kStageTokens * kHeadDim * 2;   // K per stage (V the same)
    static constexpr uint32_t kKVB = 2 * kKB;
    static constexpr uint32_t kQOff = kKVB;                          // q rows: 8 x 256 B
    static constexpr uint32_t kNewOff = kQOff + kRows * kHeadDim * 2;   // new K row, new V row: 2 x 256 B
    static constexpr uint32_t kMetaOff = kNewOff + (kRuns ? 0u : 2u * kHeadDim * 2);   // stage metadata (64 B)
    static constexpr uint32_t kStageB = 35 * 1024;                   // 1024-aligned stages
    static constexpr uint32_t kRingB = kGroups * kPStages * kStageB;
    static constexpr uint32_t kPairOff = kRingB;                     // the two groups' meeting slot
    static constexpr uint32_t kHandOff = kPairOff + kSlotB;          // [2 sides] this CTA's piece for the epilogue
    static constexpr uint32_t kBarOff = kHandOff + 2 * kSlotB;
    // barriers: full[2][stages], empty[2][stages], qbar[2], pair, ready[2]
    static constexpr int kNumBars = 2 * kGroups * kPStages + kGroups + 1 + 2;
    static constexpr uint32_t kMiscOff = (kBarOff + kNumBars * 8 + 15u) & ~15u;
    static constexpr uint32_t kHdrOff = kMiscOff + kMiscB;           // copy of this CTA's plan header (128 B)
    static constexpr size_t kSmem = 1024 + kHdrOff + 128;
    static_assert(kMetaOff + 64 <= kStageB, "stage layout");
    static_assert(kGroupWarps * 8 * kRedStride * 4 + kGroupWarps * 8 * 8 <= kKVB, "merge scratch fits a stage");
    static_assert(kHdrOff % 16 == 0 && kPairOff % 16 == 0 && kHandOff % 16 == 0, "16-byte aligned smem sections");
    static_assert(kSmem <= 227 * 1024, "one CTA's shared memory must fit in 227 KB");
};

// Byte address of 16-byte chunk c (0..15 over the 128 columns) of staged token t: swizzled
// boxes, or padded rows for runs.
template <bool kRuns>
__device__ __forceinline__ uint32_t kv_addr(uint32_t base, int t, int c, int R_log2) {
    if (kRuns) return base + (uint32_t)(t & 7) * kOctB + (uint32_t)(t >> 3) * (kHeadDim * 2) + ((uint32_t)c << 4);
    return chunk_addr(base, t, c, R_log2);
}
constexpr float kLazyLog2 = 8.f;
constexpr int kPlanMagic = 0x31504150;                  // "PAP1"
constexpr int kPlanMagicAdaptive = 0x41504150;          // "PAPA": an adaptive plan (another layout)
constexpr int kPlanMagicRuns = 0x52504150;              // "PAPR": a plan of runs (token table, no block ids)

// Stage flags.
enum : int { kBegin = 1, kEnd = 2, kNewRow = 4 };

struct PlanHeader {
    int magic;
    int num_seqs, num_q_heads, num_kv_heads, block_size, num_blocks, max_blocks_per_seq;
    int num_ctas;     // C: two groups each
    int num_chunks;   // N
    int max_chunks;
    int adaptive;     // 0: equal shares; kAdaptiveFirst / kAdaptiveFold: see PlanRates
    int cap;          // chunk slots per group (the layout: larger for adaptive plans)
    int pad[4];
};
static_assert(sizeof(PlanHeader) == 64, "plan header");

// Adaptive shares.  SMs stream the same bytes at different rates (on GB300 the per-SM finishing
// times of equal ranges of one layer differ by up to 14 %, and the same SMs stay slow from launch
// to launch), so a plan built with PA_PLAN_ADAPTIVE gives CTA c a share of the weight proportional
// to rate[c]: every decode launch on the plan measures each CTA's rate (the weight of its range
// per SM cycle of the CTA's life) and folds it into rate[c] (an exponential average); the next
// pa_decode_plan into the same buffer reads the rates.  The section outlives rebuilds; the first
// adaptive build into a buffer (or one for another grid) cuts equal shares.
struct PlanRates {
    int magic;
    int ctas;
    int pad[2];
    float rate[1];   // [ctas]; <= 0: no measurement
};
constexpr int kRatesMagic = 0x52415031;   // "RAP1"
constexpr int kAdaptiveFold = 1;          // PlanHeader::adaptive: the rates hold measurements
constexpr int kAdaptiveFirst = 2;         //   ... they hold none yet: launches write theirs
constexpr float kRateAlpha = 0.125f;      // weight of a new measurement in the average
constexpr float kRateMax = 1.0e4f;        // rates are row units per SM cycle (about 0.1): above is garbage

// One chunk of the list (32 bytes, two 16-byte loads).
struct __align__(16) PlanChunk {
    int ids[4];       // physical block of each block the chunk touches; -1: none or outside the pool
    short s, h;       // sequence, kv head
    short k, n;       // chunk of the segment, chunks of the segment
    short nvalid;     // cached tokens of the chunk (1..64)
    short gf, gl;     // first and last group holding the segment's chunks
    short merger;     // CTA combining the segment's pieces; -1: the segment stays inside one CTA
};
static_assert(sizeof(PlanChunk) == 32, "plan chunk");

// A cut segment seen from one CTA: the segment holding the CTA's first chunk (side 0) or, if
// another, its last chunk (side 1), when that segment also has chunks in other CTAs.
struct PlanEvent {
    int exists;
    int g0;             // the segment's first chunk in the list
    int s, h;
    int cf, cl;         // first and last CTA holding its chunks
    int merger;         // 1: this CTA combines the pieces
    int by_consumers;   // 1: this CTA's piece ends one of its groups' order, the consumers finish it
    int nrem;           // merger: the other CTAs' published pieces
    int rem[5];         // merger: their workspace slots (the first five; beyond, from the bounds)
};
static_assert(sizeof(PlanEvent) == 56, "plan event");

// Per CTA: its range and its cut segments, then each group's chunks in the order it streams them.
struct CtaHeader {
    int b0, b1, b2;     // group 0 streams [b0, b1) forwards, group 1 [b1, b2) backwards
    float weight;       // adaptive plans: the weight of [b0, b2), negative while the rates hold no
                        // measurement; 0: not adaptive
    PlanEvent ev[2];
};
static_assert(sizeof(CtaHeader) == 128, "CTA header");

// Byte offsets of the plan's sections: header, lengths [S], group bounds [2C + 1], then per CTA
// its header and two groups of `cap` chunk slots.
struct PlanLayout {
    size_t lens, bounds, cta, cta_bytes, rates, total;
    int cap;            // chunk slots per group
};

inline size_t al256(size_t n) { return (n + 255) & ~size_t(255); }

__host__ __device__ inline long long plan_max_chunks(int num_seqs, int num_kv_heads, int block_size,
                                                     int max_blocks_per_seq) {
    const long long cap = (long long)max_blocks_per_seq * block_size;
    return (long long)num_seqs * num_kv_heads * ((cap + kStageTokens - 1) / kStageTokens);
}

PlanLayout plan_layout(int num_seqs, int num_kv_heads, int block_size, int max_blocks_per_seq, int ctas, bool adaptive) {
    PlanLayout L;
    const long long maxc = plan_max_chunks(num_seqs, num_kv_heads, block_size, max_blocks_per_seq);
    // A group gets at most (its share of the weight + one chunk) / the lightest chunk's weight.
    // Chunks weigh 64 to 112 (at most 1.75x the lightest; with one row per kv head 336 to 500,
    // 1.5x): equal shares need fewer than two equal shares of chunks, adaptive ones (at most 1.5x
    // the equal share) fewer than three.
    const int eq = (int)((maxc + 2 * ctas - 1) / (2 * ctas));
    L.cap = adaptive ? 3 * eq + 6 : 2 * eq + 4;
    L.lens = 256;
    L.bounds = L.lens + al256((size_t)num_seqs * 4);
    L.cta = L.bounds + al256((size_t)(2 * ctas + 1) * 4);
    L.cta_bytes = sizeof(CtaHeader) + (size_t)2 * L.cap * sizeof(PlanChunk);
    L.rates = al256(L.cta + (size_t)ctas * L.cta_bytes);
    L.total = L.rates + al256(16 + (size_t)ctas * sizeof(float));
    return L;
}

// ---------------------------------------------------------------------------------------------
// The plan
// ---------------------------------------------------------------------------------------------

struct PlanArgs {
    unsigned char* plan;
    const int32_t* block_tables;
    const int32_t* context_lens;
    unsigned int* status;
    int num_seqs, num_q_heads, num_kv_heads, block_size, num_blocks, max_blocks_per_seq, ctas;
    size_t lens_off, bounds_off, cta_off, cta_bytes, rates_off;
    int cap;
    int adaptive;
    int tok_stride;   // runs plans: the token table's stride per sequence (0: block-table plan)
    long long max_chunks;
};

constexpr int kPlanThreads = 256;

// The cut of the chunk list into the 2C group ranges weighs each chunk by what it costs a group:
// the K/V rows its boxes fetch (a partly valid last block still costs its whole box), a fixed
// share for the consumers' per-chunk work and, at a segment's last chunk, the four warps' merge
// and output (row units).  Ranges of many short contexts then get fewer chunks than ranges of
// long ones.  With one query row per kv head the fixed shares are a fit of the groups' end times
// on 256 sequences x 32 kv heads of short contexts (about 2.6 ns per row fetched, 0.87 us per
// chunk, 0.43 us per segment end); with groups of 4-6 rows the smaller shares measured better
// (128 sequences of 6 rows per kv head, 16-token blocks: 2 % faster).
struct ChunkWeights {
    int chunk;   // fixed share per chunk (rows)
    int end;     // extra at a segment's last chunk (rows)
};
__host__ __device__ inline ChunkWeights chunk_weights(int group_rows) {
    return group_rows == 1 ? ChunkWeights{272, 164} : ChunkWeights{16, 32};
}

// Weight of one (sequence, kv head) segment of L tokens with boxes of R rows.
__device__ __forceinline__ long long segment_weight(int L, int R, ChunkWeights w) {
    if (L <= 0) return 0;
    const int n = (L + kStageTokens - 1) / kStageTokens;
    const int last = L - (n - 1) * kStageTokens;                  // valid rows of the last chunk
    const int last_rows = ((last + R - 1) / R) * R;
    return (long long)(n - 1) * (kStageTokens + w.chunk) + last_rows + w.chunk + w.end;
}

// The group holding chunk x: the largest g with bnd[g] <= x (bnd ascending, bnd[G2] = N).
__device__ __forceinline__ int group_of(const int32_t* bnd, int G2, long long x) {
    int lo = 0, hi = G2 - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (bnd[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Whether CTA c's piece of the segment [g0, g1) finishes late: a group streams its range from
// one end, so a piece that starts its group's order (group 0's first chunks, group 1's last)
// and is not the whole range is done early; any other piece is done at the group's end.
__device__ __forceinline__ bool piece_is_late(const int32_t* bnd, int c, long long g0, long long g1) {
    const long long b0 = bnd[2 * c], b1 = bnd[2 * c + 1], b2 = bnd[2 * c + 2];
    if (b0 < b1 && g0 < b1 && g1 > b0 && !(g0 <= b0 && g1 < b1)) return true;
    if (b1 < b2 && g0 < b2 && g1 > b1 && !(g1 >= b2 && g0 > b1)) return true;
    return false;
}

// Block-wide sums over kPlanThreads threads (every thread gets the result; `scratch` is reused
// only after a barrier).
__device__ __forceinline__ float2 block_sum2(float2 v, float2* scratch, int lane, int warp) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float2 t = make_float2(0.f, 0.f);
    for (int w = 0; w < kPlanThreads / 32; ++w) {
        t.x += scratch[w].x;
        t.y += scratch[w].y;
    }
    return t;
}

// Block-wide maximum (every thread gets it).
__device__ __forceinline__ float block_max(float v, float2* scratch, int lane, int warp) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) scratch[warp].x = v;
    __syncthreads();
    float t = scratch[0].x;
    for (int w = 1; w < kPlanThreads / 32; ++w) t = fmaxf(t, scratch[w].x);
    return t;
}

// Block-wide exclusive prefix sum of v in thread order, and the total.
__device__ __forceinline__ void block_scan(float v, float2* scratch, int lane, int warp, float& excl, float& total) {
    float incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    __syncthreads();
    if (lane == 31) scratch[warp].x = incl;
    __syncthreads();
    excl = incl - v;
    total = 0.f;
    for (int w = 0; w < kPlanThreads / 32; ++w) {
        if (w < warp) excl += scratch[w].x;
        total += scratch[w].x;
    }
}

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const PlanArgs a) {
    extern __shared__ long long plan_smem[];
    const int S = a.num_seqs, Hkv = a.num_kv_heads, B = a.block_size;
    const int G2 = 2 * a.ctas;
    const ChunkWeights cw = chunk_weights(a.num_q_heads / Hkv);
    long long* PW = plan_smem;                                     // [S + 1] exclusive prefix of weights
    int* nch = reinterpret_cast<int*>(PW + S + 1);                 // [S] chunks per kv head of each sequence
    int* P = nch + S;                                              // [S + 1] exclusive prefix of nch
    int* Ls = P + S + 1;                                           // [S] clamped lengths
    int32_t* bnd = Ls + S;                                         // [2C + 1] group bounds
    float* rc = reinterpret_cast<float*>(bnd + G2 + 1);            // [C + 1] adaptive: share before CTA c
    __shared__ int warp_tot[kPlanThreads / 32];
    __shared__ long long warp_wt[kPlanThreads / 32];
    __shared__ float2 warp_f2[kPlanThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long cap = (long long)a.max_blocks_per_seq * B;
    // rows a chunk's last block costs: whole boxes of R rows, or (runs) exactly its rows
    const int R = a.tok_stride ? 1 : (B < kStageTokens ? B : kStageTokens);

    grid_dependency_wait();
    // lengths, chunk counts and weights; a thread owns a contiguous run of sequences
    const int per = (S + kPlanThreads - 1) / kPlanThreads;
    const int lo = min(S, tid * per), hi = min(S, lo + per);
    int local = 0;
    long long local_w = 0;
    for (int s = lo; s < hi; ++s) {
        int L = a.context_lens[s];
        if (L < 0 || L > cap) {
            if (blockIdx.x == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
            L = L < 0 ? 0 : (int)cap;
        }
        Ls[s] = L;
        nch[s] = (L + kStageTokens - 1) / kStageTokens;
        local += nch[s];
        local_w += (long long)Hkv * segment_weight(L, R, cw);
    }
    int incl = local;
    long long incl_w = local_w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        const long long vw = __shfl_up_sync(0xffffffffu, incl_w, o);
        if (lane >= o) {
            incl += v;
            incl_w += vw;
        }
    }
    if (lane == 31) {
        warp_tot[warp] = incl;
        warp_wt[warp] = incl_w;
    }
    __syncthreads();
    int run = incl - local, tot = 0;
    long long run_w = incl_w - local_w, tot_w = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) {
        if (w < warp) {
            run += warp_tot[w];
            run_w += warp_wt[w];
        }
        tot += warp_tot[w];
        tot_w += warp_wt[w];
    }
    for (int s = lo; s < hi; ++s) {
        P[s] = run;
        PW[s] = run_w;
        run += nch[s];
        run_w += (long long)Hkv * segment_weight(Ls[s], R, cw);
    }
    if (tid == 0) {
        P[S] = tot;
        PW[S] = tot_w;
    }
    __syncthreads();

    const long long N = (long long)Hkv * tot;
    // CTA shares: equal, or (adaptive, once rates were measured) proportional to the CTAs'
    // measured rates, each clamped to within a factor of two of their mean (a CTA without a
    // measurement counts as the mean); rc[c] = the share before CTA c, rc[C] = 1.  No block of
    // this kernel writes the rates, so all blocks take the same shares.
    const PlanRates* rates = reinterpret_cast<const PlanRates*>(a.plan + a.rates_off);
    const int C = a.ctas;
    const bool rates_ok = a.adaptive && rates->magic == kRatesMagic && rates->ctas == C;
    if (rates_ok) {   // (the same branch in every thread: nothing writes the rates during this kernel)
        const int per_c = (C + kPlanThreads - 1) / kPlanThreads;
        const int clo = min(C, tid * per_c), chi = min(C, clo + per_c);
        float mine[4];   // C <= 4 * kPlanThreads (checked by the host)
        float sum = 0.f, cnt = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float r = -1.f;
            if (clo + j < chi) {
                r = rates->rate[clo + j];
                if (!(r > 0.f && r < kRateMax)) r = -1.f;   // unmeasured (0, negative, NaN, garbage)
            }
            mine[j] = r;
            if (r > 0.f) {
                sum += r;
                cnt += 1.f;
            }
        }
        float2 tw = block_sum2(make_float2(sum, cnt), warp_f2, lane, warp);
        const float mean = tw.y > 0.f ? tw.x / tw.y : 1.f;
        float run_r = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float r = clo + j >= chi ? 0.f : mine[j] > 0.f ? fminf(fmaxf(mine[j], 0.5f * mean), 2.f * mean) : mean;
            mine[j] = r;
            run_r += r;
        }
        float excl = 0.f, total = 0.f;
        block_scan(run_r, warp_f2, lane, warp, excl, total);
        // no share above 1.5x the equal one (the plan's slots per group assume it): mix the rates'
        // shares with equal ones, beta = 0.5 / (largest ratio - 1) where that ratio exceeds 1.5
        float top = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (clo + j < chi) top = fmaxf(top, mine[j] * (float)C / total);
        top = block_max(top, warp_f2, lane, warp);
        const float beta = top > 1.5f ? 0.5f / (top - 1.f) : 1.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (clo + j < chi) rc[clo + j] = (1.f - beta) * (float)(clo + j) / (float)C + beta * excl / total;
            excl += mine[j];
        }
        if (tid == 0) rc[C] = 1.f;
        __syncthreads();
    }
    // group bounds: group g starts at the first chunk whose starting weight reaches its share of
    // the total, W g / G2 (adaptive: its CTA's share, split in half between the two groups)
    for (int g = tid; g <= G2; g += kPlanThreads) {
        long long T;
        if (rates_ok) {
            const int cg = g >> 1;
            double f = (g & 1) ? 0.5 * ((double)rc[cg] + (double)rc[cg + 1]) : (double)rc[min(cg, C)];
            f = f >= 0.0 ? (f <= 1.0 ? f : 1.0) : 0.0;   // (NaN -> 0: cannot arise from sanitised rates)
            T = (g == G2) ? tot_w : (long long)(f * (double)tot_w);
            if (T > tot_w) T = tot_w;
        } else {
            T = tot_w * g / G2;
        }
        long long b = N;
        if (T < tot_w) {
            int l2 = 0, h2 = S - 1;   // the sequence holding weight position T (empty ones skipped)
            while (l2 < h2) {
                const int mid = (l2 + h2 + 1) >> 1;
                if (PW[mid] <= T) l2 = mid;
                else h2 = mid - 1;
            }
            const int n = nch[l2];
            const long long ws = segment_weight(Ls[l2], R, cw);
            const long long o = T - PW[l2];
            const long long h = o / ws, rem = o - h * ws;
            const long long k = (rem + kStageTokens + cw.chunk - 1) / (kStageTokens + cw.chunk);   // ceil
            b = (long long)Hkv * P[l2] + h * n + (k < n ? k : n);
        }
        bnd[g] = (int32_t)b;
    }
    __syncthreads();

    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(a.plan);
    int32_t* lens = reinterpret_cast<int32_t*>(a.plan + a.lens_off);
    int32_t* bounds = reinterpret_cast<int32_t*>(a.plan + a.bounds_off);
    auto cta_header = [&](int c) { return reinterpret_cast<CtaHeader*>(a.plan + a.cta_off + (size_t)c * a.cta_bytes); };
    // starting weight of chunk x (x == N: the total): the sequence is the last whose first chunk is
    // at or before x (empty sequences share the next one's first chunk, so that one is found)
    auto chunk_start_weight = [&](long long x) -> long long {
        if (x >= N) return tot_w;
        int l2 = 0, h2 = S - 1;
        while (l2 < h2) {
            const int mid = (l2 + h2 + 1) >> 1;
            if ((long long)Hkv * P[mid] <= x) l2 = mid;
            else h2 = mid - 1;
        }
        const int n = nch[l2];
        const long long o = x - (long long)Hkv * P[l2];
        const long long h = o / n, k = o - h * n;
        return PW[l2] + h * segment_weight(Ls[l2], R, cw) + k * (kStageTokens + cw.chunk);
    };
    if (blockIdx.x == 0) {
        for (int s = tid; s < S; s += kPlanThreads) lens[s] = Ls[s];
        for (int g = tid; g <= G2; g += kPlanThreads) bounds[g] = bnd[g];
        for (int c = tid; c < a.ctas; c += kPlanThreads) {
            CtaHeader* ch = cta_header(c);
            ch->b0 = bnd[2 * c];
            ch->b1 = bnd[2 * c + 1];
            ch->b2 = bnd[2 * c + 2];
            if (a.adaptive) {
                const float w = fmaxf(1.f, (float)(chunk_start_weight(bnd[2 * c + 2]) - chunk_start_weight(bnd[2 * c])));
                ch->weight = rates_ok ? w : -w;
            } else {
                ch->weight = 0.f;
            }
            if (bnd[2 * c] == bnd[2 * c + 2]) {   // no chunks: no events (nothing else writes them)
                ch->ev[0].exists = 0;
                ch->ev[1].exists = 0;
            }
        }
        if (tid == 0) {
            PlanHeader h = {};
            h.magic = a.tok_stride ? kPlanMagicRuns : a.adaptive ? kPlanMagicAdaptive : kPlanMagic;   // (layouts differ)
            h.num_seqs = S;
            h.num_q_heads = a.num_q_heads;
            h.num_kv_heads = Hkv;
            h.block_size = B;
            h.num_blocks = a.num_blocks;
            h.max_blocks_per_seq = a.max_blocks_per_seq;
            h.num_ctas = a.ctas;
            h.num_chunks = (int)N;
            h.max_chunks = (int)a.max_chunks;
            h.adaptive = a.adaptive ? (rates_ok ? kAdaptiveFold : kAdaptiveFirst) : 0;
            h.cap = a.cap;
            *hdr = h;
        }
    }
    // one descriptor per chunk, grid-stride
    for (long long g = (long long)blockIdx.x * kPlanThreads + tid; g < N; g += (long long)gridDim.x * kPlanThreads) {
        // the sequence: largest s with Hkv * P[s] <= g
        int l2 = 0, h2 = S - 1;
        while (l2 < h2) {
            const int mid = (l2 + h2 + 1) >> 1;
            if ((long long)Hkv * P[mid] <= g) l2 = mid;
            else h2 = mid - 1;
        }
        const int s = l2;
        const int n = nch[s];
        const int r = (int)(g - (long long)Hkv * P[s]);
        const int h = r / n, k = r - h * n;
        const int L = Ls[s];
        const int t0 = k * kStageTokens, t1 = min(t0 + kStageTokens, L);
        const int first = t0 / B, nblk = (t1 - 1) / B - first + 1;
        PlanChunk d;
        if (a.tok_stride) {   // runs: where the chunk's tokens start in the token table
            d.ids[0] = (int)((long long)s * a.tok_stride + t0);
            d.ids[1] = d.ids[2] = d.ids[3] = -1;
        } else {
            const int32_t* row = a.block_tables + (size_t)s * a.max_blocks_per_seq + first;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                d.ids[e] = -1;
                if (e < nblk) {
                    const int id = row[e];
                    if (id >= 0 && id < a.num_blocks) d.ids[e] = id;
                    else flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
                }
            }
        }
        d.s = (short)s;
        d.h = (short)h;
        d.k = (short)k;
        d.n = (short)n;
        d.nvalid = (short)(t1 - t0);
        const long long g0 = g - k, g1 = g0 + n;
        const int gf = group_of(bnd, G2, g0), gl = group_of(bnd, G2, g1 - 1);
        d.gf = (short)gf;
        d.gl = (short)gl;
        int merger = -1;
        if (gf / 2 != gl / 2) {
            merger = gf / 2;
            for (int c = gf / 2; c <= gl / 2; ++c)
                if (piece_is_late(bnd, c, g0, g1)) {
                    merger = c;
                    break;
                }
        }
        d.merger = (short)merger;
        // stored where its group streams it: group 0 forwards from b0, group 1 backwards from b2 - 1
        const int grp = group_of(bnd, G2, g);
        const int c = grp / 2, side_g = grp & 1;
        const long long b0 = bnd[2 * c], b1 = bnd[2 * c + 1], b2 = bnd[2 * c + 2];
        const long long pos = side_g ? (b2 - 1 - g) : (g - b0);
        CtaHeader* ch = cta_header(c);
        PlanChunk* slots = reinterpret_cast<PlanChunk*>(reinterpret_cast<unsigned char*>(ch) + sizeof(CtaHeader));
        const uint4* src = reinterpret_cast<const uint4*>(&d);
        uint4* dst = reinterpret_cast<uint4*>(slots + (size_t)side_g * a.cap + pos);
        dst[0] = src[0];
        dst[1] = src[1];
        // the CTA's cut segments: written by the threads of its first and last chunks
        for (int side = 0; side < 2; ++side) {
            if (g != (side == 0 ? b0 : b2 - 1)) continue;
            PlanEvent ev = {};
            const bool cross = gf / 2 != gl / 2;
            ev.exists = cross && (side == 0 || g0 > b0) ? 1 : 0;   // side 1: another segment than side 0's
            ev.g0 = (int)g0;
            ev.s = s;
            ev.h = h;
            ev.cf = gf / 2;
            ev.cl = gl / 2;
            ev.merger = merger == c ? 1 : 0;
            // the piece ends a group's order: it reaches b1 (side 0) or starts by b1 (side 1), or
            // the other group is empty
            ev.by_consumers = side == 0 ? ((b0 < b1) ? (g1 >= b1) : 1) : ((b1 < b2) ? (g0 <= b1) : 1);
            int nrem = 0;
            if (ev.merger) {
                for (int cc = gf / 2; cc <= gl / 2; ++cc) {
                    const long long cb0 = bnd[2 * cc], cb2 = bnd[2 * cc + 2];
                    if (cc == c || cb0 == cb2) continue;
                    if (nrem < 5) ev.rem[nrem] = 2 * cc + (g0 <= cb0 ? 0 : 1);
                    ++nrem;
                }
            }
            ev.nrem = nrem;
            ch->ev[side] = ev;
        }
    }
    grid_launch_dependents();
}

// ---------------------------------------------------------------------------------------------
// The decode launch
// ---------------------------------------------------------------------------------------------

struct PlannedArgs {
    void* out;                  // [S][Hq][D]
    const void* q;              // [S][Hq][D]
    const void* k_new;          // append: [S][Hkv][D] rows written at position L - 1; null = off
    const void* v_new;
    const void* k_cache;        // [NB][Hkv][B][D]
    const void* v_cache;
    const unsigned char* plan;
    float* part_o;              // [2C][8][D] unnormalised partial outputs of cut segments
    float2* part_ml;            // [2C][8] (running max in log2 units, sum); every word holds kEmptyWord
                                // between launches, so that a word another CTA reads is either empty
                                // or the published value (32-bit words are read and written whole)
    unsigned int* status;
    unsigned long long* timeline;
    PlanRates* rates;           // the plan's rates section (adaptive plans: updated at the end)
    const int32_t* tok;         // runs plans: per token of a sequence, (block * Hkv) * B + slot; a chunk
                                // descriptor's ids[0] indexes its first token
    float scale_log2;
    int num_seqs, num_q_heads, num_kv_heads, block_size, num_blocks, max_blocks_per_seq;
    int early;
    int cap;                    // chunk slots per group in the plan
    size_t lens_off, bounds_off, cta_off, cta_bytes;
};

// Tensor maps of the two pools: boxes of R = min(block_size, 64) rows.
struct MmaMapsP {
    CUtensorMap k, v;
};

// Flush modes of a segment's last chunk in a group's order.
//   kOut          the segment lies in this group: write the output
//   kPair         it spans both groups of this CTA: meet the other group in shared memory
//   kPublish      another CTA merges: store the partial into this CTA's workspace slot (the
//                 stored words are the publication: the merger waits for them to stop being empty)
//   kMerge        this CTA merges, its piece ends early: hand it to the epilogue warp
//   kMergeHere    this CTA merges at the end of this group's order: fold the others' pieces here
enum : int { kOutM = 0, kPairM = 1, kPublishM = 2, kMergeM = 3, kMergeHereM = 5 };

// The value of every workspace word between launches: a NaN bit pattern no arithmetic here
// produces (fp32 operations return the canonical 0x7fffffff, and NaN inputs keep part of their
// fp16/bf16 payload), so a word that differs from it holds a published value.
constexpr uint32_t kEmptyWord = 0xffffffffu;

struct StageMeta {
    int s, h, k, n;
    int nvalid;
    int flags;        // kBegin / kEnd / kNewRow
    int mode;         // flush mode at kEnd
    int post;         // after the two groups have met (kPairM): kOutM, kPublishM or kMergeHereM
    int side;         // which of the CTA's two cut segments (0: the one holding its first chunk)
    int new_phys;     // block of the new token (-1: none, -2: outside the pool)
    int new_off;      // its row within the block
    int pad[5];
};
static_assert(sizeof(StageMeta) == 64, "stage metadata");

__device__ __forceinline__ void group_sync(int grp) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kGroupThreads) : "memory");
}

// A barrier of the group's 128 consumer threads that also returns whether `v` holds in all of
// them, so that the group takes one decision together.
__device__ __forceinline__ bool group_all(int grp, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(1 + grp), "n"(kGroupThreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// GPU-scope relaxed accesses of the workspace: each 32-bit element is read or written whole.
__device__ __forceinline__ uint4 ld_relaxed4(const void* p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint2 ld_relaxed2(const void* p) {
    uint2 v;
    asm volatile("ld.relaxed.gpu.global.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed4(void* p, uint4 v) {
    asm volatile("st.relaxed.gpu.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_relaxed2(void* p, uint2 v) {
    asm volatile("st.relaxed.gpu.global.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ bool full4(uint4 v) {
    return v.x != kEmptyWord && v.y != kEmptyWord && v.z != kEmptyWord && v.w != kEmptyWord;
}


__device__ __forceinline__ void load_chunk(const PlanChunk* src, PlanChunk& d) {
    const uint4* p = reinterpret_cast<const uint4*>(src);
    uint4* q = reinterpret_cast<uint4*>(&d);
    q[0] = __ldcg(p);
    q[1] = __ldcg(p + 1);
}

// A running combination of partial results (m, l, o) of one query row, 8 columns per thread.
struct Fold8 {
    float M, den, num[8];
    __device__ __forceinline__ void init() {
        M = -INFINITY;
        den = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) num[j] = 0.f;
    }
    __device__ __forceinline__ void add(float m, float l, const float (&o)[8]) {
        const float Mn = fmaxf(M, m);
        const float a = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
        const float b = exp2f(m - Mn);
        den = den * a + l * b;
#pragma unroll
        for (int j = 0; j < 8; ++j) num[j] = num[j] * a + o[j] * b;
        M = Mn;
    }
};

template <typename T>
__device__ __forceinline__ uint4 pack8(const float (&v)[8], float inv) {
    uint4 u;
    u.x = Elem<T>::pack2(v[0] * inv, v[1] * inv);
    u.y = Elem<T>::pack2(v[2] * inv, v[3] * inv);
    u.z = Elem<T>::pack2(v[4] * inv, v[5] * inv);
    u.w = Elem<T>::pack2(v[6] * inv, v[7] * inv);
    return u;
}

// Partial slot (global or shared): o [8][D] fp32, then (m, l) [8].
__device__ __forceinline__ void slot_store(float* o, float2* ml, int r, int d0, const Fold8& f, bool write_ml) {
    *reinterpret_cast<float4*>(o + r * kHeadDim + d0) = make_float4(f.num[0], f.num[1], f.num[2], f.num[3]);
    *reinterpret_cast<float4*>(o + r * kHeadDim + d0 + 4) = make_float4(f.num[4], f.num[5], f.num[6], f.num[7]);
    if (write_ml) ml[r] = make_float2(f.M, f.den);
}

__device__ __forceinline__ void slot_load(const float* o, const float2* ml, int r, int d0, float& m, float& l,
                                          float (&v)[8]) {
    const float2 x = ml[r];
    m = x.x;
    l = x.y;
    const float4 a0 = *reinterpret_cast<const float4*>(o + r * kHeadDim + d0);
    const float4 a1 = *reinterpret_cast<const float4*>(o + r * kHeadDim + d0 + 4);
    v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
    v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
}

// Publish this thread's share of a partial (row r, columns d0 .. d0 + 7; (m, l) by one thread of
// the row) into a workspace slot.
__device__ __forceinline__ void publish8(float* o, float2* ml, int r, int d0, const Fold8& f, bool write_ml) {
    float* dst = o + r * kHeadDim + d0;
    st_relaxed4(dst, make_uint4(__float_as_uint(f.num[0]), __float_as_uint(f.num[1]), __float_as_uint(f.num[2]),
                                __float_as_uint(f.num[3])));
    st_relaxed4(dst + 4, make_uint4(__float_as_uint(f.num[4]), __float_as_uint(f.num[5]), __float_as_uint(f.num[6]),
                                    __float_as_uint(f.num[7])));
    if (write_ml) st_relaxed2(ml + r, make_uint2(__float_as_uint(f.M), __float_as_uint(f.den)));
}

// Fetch this thread's share of a published partial into (m, l, v) once every word of it has been
// written; false if some word is still empty.
__device__ __forceinline__ bool fetch8(const float* o, const float2* ml, int r, int d0, float& m, float& l,
                                       float (&v)[8]) {
    const uint4 a0 = ld_relaxed4(o + r * kHeadDim + d0);
    const uint4 a1 = ld_relaxed4(o + r * kHeadDim + d0 + 4);
    const uint2 x = ld_relaxed2(ml + r);
    if (!full4(a0) || !full4(a1) || x.x == kEmptyWord || x.y == kEmptyWord) return false;
    m = __uint_as_float(x.x);
    l = __uint_as_float(x.y);
    v[0] = __uint_as_float(a0.x); v[1] = __uint_as_float(a0.y); v[2] = __uint_as_float(a0.z); v[3] = __uint_as_float(a0.w);
    v[4] = __uint_as_float(a1.x); v[5] = __uint_as_float(a1.y); v[6] = __uint_as_float(a1.z); v[7] = __uint_as_float(a1.w);
    return true;
}

// Return a consumed share to empty for the next launch.
__device__ __forceinline__ void clear8(float* o, float2* ml, int r, int d0, bool write_ml) {
    const uint4 e = make_uint4(kEmptyWord, kEmptyWord, kEmptyWord, kEmptyWord);
    st_relaxed4(o + r * kHeadDim + d0, e);
    st_relaxed4(o + r * kHeadDim + d0 + 4, e);
    if (write_ml) st_relaxed2(ml + r, make_uint2(kEmptyWord, kEmptyWord));
}

// The k-th other CTA's workspace slot for a merge event: from the plan's list for the first
// five, else counted out of the bounds (CTA order, skipping this CTA and CTAs without chunks).
__device__ __forceinline__ int remote_slot(const PlanEvent& ev, const int32_t* bounds, int c, int k) {
    if (k < 5) return ev.rem[k];
    int seen = 0;
    for (int cc = ev.cf; cc <= ev.cl; ++cc) {
        const int cb0 = __ldcg(bounds + 2 * cc);
        if (cc == c || cb0 == __ldcg(bounds + 2 * cc + 2)) continue;
        if (seen++ == k) return 2 * cc + (ev.g0 <= cb0 ? 0 : 1);
    }
    return 0;
}

template <typename T, bool kAdaptive, bool kRuns>
__global__ void __launch_bounds__(kPThreads, 1)
    decode_planned_kernel(const PlannedArgs a, const __grid_constant__ MmaMapsP maps, const int R_log2) {
    using Y = Lay<kRuns>;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* bp = smem_raw + (base - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(bp + Y::kBarOff);
    uint64_t* full = bars;                                  // [2][3]
    uint64_t* empty = bars + kGroups * Y::kPStages;            // [2][3]
    uint64_t* qbar = bars + 2 * kGroups * Y::kPStages;         // [2] deferred q / new rows of the first stages
    uint64_t* pair_bar = qbar + kGroups;                    // the first group's piece is in the pair slot
    uint64_t* ready = pair_bar + 1;                         // [2] this CTA's piece of cut segment `side`
    volatile int* misc = reinterpret_cast<volatile int*>(bp + Y::kMiscOff);
    volatile int* abort_flag = misc;
    volatile int* pair_count = misc + 1;
    volatile int* pair_role = misc + 2;                     // [2]
    volatile int* issued = misc + 4;                        // [2]
    volatile int* qdef = misc + 8;                          // [2][3]: deferred q row (s * Hkv + h) or -1
    volatile int* ndef = misc + 16;                         // [2][3]: deferred new rows (s * Hkv + h) or -1
    // misc + 29: this CTA's rate before the launch (bits, copied by thread 0), + 30: the SM clock
    // when the CTA started (adaptive plans)
    // this CTA's header, copied by each producer before its first stage is released
    CtaHeader* sh_hdr = reinterpret_cast<CtaHeader*>(bp + Y::kHdrOff);
    float* pair_o = reinterpret_cast<float*>(bp + Y::kPairOff);
    float2* pair_ml = reinterpret_cast<float2*>(bp + Y::kPairOff + kRows * kHeadDim * 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads, G = Hq / Hkv, B = a.block_size;
    const int32_t* bounds = reinterpret_cast<const int32_t*>(a.plan + a.bounds_off);
    const unsigned char* cta_area = a.plan + a.cta_off + (size_t)c * a.cta_bytes;
    const CtaHeader* g_hdr = reinterpret_cast<const CtaHeader*>(cta_area);
    const PlanChunk* slots = reinterpret_cast<const PlanChunk*>(cta_area + sizeof(CtaHeader));
    const bool append = a.k_new != nullptr;

    if (tid == 0) {
        trace(a.timeline, c, 0);
        if (!kRuns) {
            prefetch_map(&maps.k);
            prefetch_map(&maps.v);
        }
        for (int i = 0; i < kGroups * Y::kPStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kGroupThreads);
        }
        for (int i = 0; i < kGroups; ++i) mbar_init(&qbar[i], 1);
        mbar_init(pair_bar, kGroupThreads);
        mbar_init(&ready[0], kGroupThreads);
        mbar_init(&ready[1], kGroupThreads);
        *abort_flag = 0;
        *pair_count = 0;
        if (kAdaptive) {
            misc[30] = (int)clock();
            // this CTA's rate so far (folded at the end), copied without a register; this thread
            // waits for the copy at the end of its consumer loop
            cp_async4(smem_u32(const_cast<int*>(misc + 29)), &a.rates->rate[c]);
        }   // adaptive plans time the CTA's life from here
        for (int i = 0; i < kGroups * Y::kPStages; ++i) {
            qdef[i] = -1;
            ndef[i] = -1;
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (!a.early) grid_dependency_wait();
    // Every warp reads the plan's header (is it this launch's?) and this CTA's range together in
    // one round trip; the producers also read their first descriptors in it.
    const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(a.plan);
    const int h_magic = __ldcg(&hdr->magic), h_seqs = __ldcg(&hdr->num_seqs), h_qh = __ldcg(&hdr->num_q_heads),
              h_kvh = __ldcg(&hdr->num_kv_heads), h_bs = __ldcg(&hdr->block_size), h_nb = __ldcg(&hdr->num_blocks),
              h_mb = __ldcg(&hdr->max_blocks_per_seq), h_c = __ldcg(&hdr->num_ctas);
    const int b0 = __ldcg(&g_hdr->b0), b1 = __ldcg(&g_hdr->b1), b2 = __ldcg(&g_hdr->b2);
    const bool is_prod = warp >= kProdWarp0 && warp < kEpiWarp;
    const int pgrp = warp - kProdWarp0;
    const int plo = pgrp ? b1 : b0, phi = pgrp ? b2 : b1;   // producer's group range (valid for producers)
    PlanChunk cur;
    if (is_prod && lane < min(32, a.cap)) load_chunk(slots + (size_t)pgrp * a.cap + lane, cur);
    uint4 hdr_part = make_uint4(0, 0, 0, 0);   // producers: lane j < 8 holds bytes 16 j .. of the CTA header
    if (is_prod && lane < 8) hdr_part = __ldcg(reinterpret_cast<const uint4*>(g_hdr) + lane);
    const bool plan_ok = h_magic == (kRuns ? kPlanMagicRuns : kAdaptive ? kPlanMagicAdaptive : kPlanMagic) &&
                         h_seqs == a.num_seqs &&
                         h_qh == Hq && h_kvh == Hkv && h_bs == B && h_nb == a.num_blocks && h_mb == a.max_blocks_per_seq && h_c == (int)gridDim.x &&
                         b0 <= b1 && b1 <= b2 && b1 - b0 <= a.cap && b2 - b1 <= a.cap;
    if (!plan_ok) {
        // the same decision in every thread (same bytes read); nothing was started
        if (a.early) grid_dependency_wait();
        grid_launch_dependents();
        if (tid == 0 && c == 0) flag_status(a.status, PA_DEV_BAD_PLAN);
        if (kAdaptive && tid == 0) cp_async_wait_all();
        return;
    }
    if (!a.early) grid_launch_dependents();

    if (is_prod) {
        // ============================ producer of one group ============================
        const int grp = pgrp, lo = plo, hi = phi;
        const int cnt = hi - lo;
        auto chunk_at = [&](int p) { return grp ? hi - 1 - p : lo + p; };
        uint64_t* gfull = full + grp * Y::kPStages;
        uint64_t* gempty = empty + grp * Y::kPStages;
        const uint32_t ring = base + (uint32_t)grp * Y::kPStages * Y::kStageB;
        const uint32_t group_bytes = (uint32_t)G * kHeadDim * 2u;
        const int R = 1 << R_log2;
        // the CTA header into shared memory (both producers write the same bytes): consumers read it
        // after a stage of this producer has landed
        if (lane < 8) reinterpret_cast<uint4*>(sh_hdr)[lane] = hdr_part;
        __syncwarp();
        bool deps_done = !a.early;
        auto dependency_point = [&](int n_issued) {
            grid_dependency_wait();
            grid_launch_dependents();
            if (lane == 0) {
                const int n = min(n_issued, Y::kPStages);
                uint32_t bytes = 0;
                for (int e = 0; e < n; ++e) {
                    if (qdef[grp * Y::kPStages + e] >= 0) bytes += group_bytes;
                    if (ndef[grp * Y::kPStages + e] >= 0) bytes += 4u * kHeadDim;
                }
                mbar_arrive_expect_tx(&qbar[grp], bytes);
                for (int e = 0; e < n; ++e) {
                    const uint32_t dst = ring + (uint32_t)e * Y::kStageB;
                    const int sh = qdef[grp * Y::kPStages + e];
                    if (sh >= 0)
                        bulk_g2s(dst + Y::kQOff,
                                 static_cast<const T*>(a.q) + ((size_t)(sh / Hkv) * Hq + (sh % Hkv) * G) * kHeadDim,
                                 group_bytes, &qbar[grp]);
                    const int nh = ndef[grp * Y::kPStages + e];
                    if (nh >= 0) {
                        bulk_g2s(dst + Y::kNewOff, static_cast<const T*>(a.k_new) + (size_t)nh * kHeadDim, 2u * kHeadDim,
                                 &qbar[grp]);
                        bulk_g2s(dst + Y::kNewOff + 2u * kHeadDim, static_cast<const T*>(a.v_new) + (size_t)nh * kHeadDim,
                                 2u * kHeadDim, &qbar[grp]);
                    }
                }
            }
            __syncwarp();
        };
        if (grp == 0 && lane == 0) trace(a.timeline, c, 3);
        // runs: the token entries of this lane's octet (tokens 8 (lane mod 8) .. + 7; lanes 0-15) of
        // the chunk about to be issued
        int tokq[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (kRuns && cnt > 0) {
            const uint4 c0 = reinterpret_cast<const uint4*>(&cur)[0];
            const uint4 c1 = reinterpret_cast<const uint4*>(&cur)[1];
            const int idx = (int)__shfl_sync(0xffffffffu, c0.x, 0);
            const int nv0 = (int)(short)(__shfl_sync(0xffffffffu, c1.z, 0) & 0xffffu);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                tokq[e] = lane < 16 && 8 * (lane & 7) + e < nv0 ? __ldg(a.tok + idx + 8 * (lane & 7) + e) : 0;
        }
        bool ok = true;
        int i = 0;
        for (int pb = 0; pb < cnt && ok; pb += 32) {
            PlanChunk nxt;
            if (pb + 32 + lane < cnt) load_chunk(slots + (size_t)grp * a.cap + pb + 32 + lane, nxt);
            const int m = min(32, cnt - pb);
            for (int j = 0; j < m; ++j, ++i) {
                const int st = i % Y::kPStages;
                if (i == Y::kPStages && !deps_done) {
                    dependency_point(i);
                    deps_done = true;
                }
                if (i >= Y::kPStages) {
                    bool w = true;
                    if (lane == 0) w = mbar_wait_bounded(&gempty[st], (uint32_t)((i / Y::kPStages) - 1) & 1u);
                    w = __shfl_sync(0xffffffffu, w, 0);
                    if (!w) {
                        if (lane == 0) {
                            flag_status(a.status, PA_DEV_TIMEOUT);
                            *abort_flag = 1;
                        }
                        ok = false;
                        break;
                    }
                }
                // chunk j of this batch, from lane j
                const uint4 w0 = reinterpret_cast<const uint4*>(&cur)[0];
                const uint4 w1 = reinterpret_cast<const uint4*>(&cur)[1];
                PlanChunk d;
                uint4* dw = reinterpret_cast<uint4*>(&d);
                dw[0] = make_uint4(__shfl_sync(0xffffffffu, w0.x, j), __shfl_sync(0xffffffffu, w0.y, j),
                                   __shfl_sync(0xffffffffu, w0.z, j), __shfl_sync(0xffffffffu, w0.w, j));
                dw[1] = make_uint4(__shfl_sync(0xffffffffu, w1.x, j), __shfl_sync(0xffffffffu, w1.y, j),
                                   __shfl_sync(0xffffffffu, w1.z, j), __shfl_sync(0xffffffffu, w1.w, j));
                if (lane == 0) {
                    if (*abort_flag) {
                        ok = false;
                    } else {
                        const int p = pb + j;
                        const int g = chunk_at(p);
                        const int s = d.s, h = d.h, k = d.k, n = d.n, nvalid = d.nvalid;
                        const int g0 = g - k, g1 = g0 + n;
                        int flags = 0;
                        if (grp == 0) {
                            if (k == 0 || g == lo) flags |= kBegin;
                            if (k == n - 1 || g == hi - 1) flags |= kEnd;
                        } else {
                            if (k == n - 1 || g == hi - 1) flags |= kBegin;
                            if (k == 0 || g == lo) flags |= kEnd;
                        }
                        int mode = kOutM, post = kOutM, side = 0;
                        if (flags & kEnd) {
                            const bool in_group = g0 >= lo && g1 <= hi;
                            const bool cross_cta = d.gf / 2 != d.gl / 2;
                            const bool spans_pair = g0 < b1 && g1 > b1 && b0 < b1 && b1 < b2;
                            const bool here = p == cnt - 1;   // the group's last chunk: nothing after it to stream
                            side = (g0 <= b0) ? 0 : 1;
                            const int role =
                                cross_cta ? (d.merger == c ? (here ? kMergeHereM : kMergeM) : kPublishM) : kOutM;
                            if (in_group) {
                                mode = kOutM;
                            } else if (spans_pair) {
                                mode = kPairM;   // pair pieces end both groups' orders
                                post = cross_cta ? (d.merger == c ? kMergeHereM : kPublishM) : kOutM;
                            } else {
                                mode = role;
                            }
                        }
                        const bool newrow = append && (k == n - 1);
                        int new_phys = -1, new_off = 0;
                        if (newrow) {
                            const int t0 = k * kStageTokens, tl = t0 + nvalid - 1;
                            const int e = tl / B - t0 / B;
                            int id = -2;
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4)
                                if (q4 == e) id = d.ids[q4] >= 0 ? d.ids[q4] : -2;
                            new_phys = id;
                            new_off = tl % B;
                            flags |= kNewRow;
                        }
                        const uint32_t dst = ring + (uint32_t)st * Y::kStageB;
                        StageMeta* meta = reinterpret_cast<StageMeta*>(bp + (dst - base) + Y::kMetaOff);
                        meta->s = s;
                        meta->h = h;
                        meta->k = k;
                        meta->n = n;
                        meta->nvalid = nvalid;
                        meta->flags = flags;
                        meta->mode = mode;
                        meta->post = post;
                        meta->side = side;
                        meta->new_phys = new_phys;
                        meta->new_off = new_off;
                        const bool defer = !deps_done;   // q and the new rows come after the dependency wait
                        const int sh = s * Hkv + h;
                        if (defer) {
                            qdef[grp * Y::kPStages + i] = (flags & kBegin) ? sh : -1;
                            ndef[grp * Y::kPStages + i] = newrow ? sh : -1;
                        }
                        const int t0 = k * kStageTokens;
                        const int within = (B > kStageTokens) ? (t0 % B) : 0;
                        const int nblk = (t0 + nvalid - 1) / B - t0 / B + 1;
                        uint32_t bytes = 0;
                        if ((flags & kBegin) && !defer) bytes += group_bytes;
                        if (newrow && !defer) bytes += 4u * kHeadDim;
                        if (kRuns) {
                            bytes += 4u * kHeadDim * (uint32_t)nvalid;   // a K and a V row per token
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (e < nblk && d.ids[e] >= 0) bytes += 4u * (uint32_t)R * 128u;
                        }
                        if (i >= Y::kPStages) fence_proxy_async_smem();
                        mbar_arrive_expect_tx(&gfull[st], bytes);   // release: the metadata and header above
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (!kRuns && e < nblk && d.ids[e] >= 0) {
                                const int row = (d.ids[e] * Hkv + h) * B + within;
                                const uint32_t box = dst + (uint32_t)(e * 2 * R) * 128u;
                                tma_load_2d(box, &maps.k, 0, row, &gfull[st]);
                                tma_load_2d(box + (uint32_t)R * 128u, &maps.k, 64, row, &gfull[st]);
                                tma_load_2d(box + Y::kKB, &maps.v, 0, row, &gfull[st]);
                                tma_load_2d(box + Y::kKB + (uint32_t)R * 128u, &maps.v, 64, row, &gfull[st]);
                            }
                        }
                        if (grp == 0 && i == 0) trace(a.timeline, c, 4);
                        if ((flags & kBegin) && !defer)
                            bulk_g2s(dst + Y::kQOff, static_cast<const T*>(a.q) + ((size_t)s * Hq + h * G) * kHeadDim,
                                     group_bytes, &gfull[st]);
                        if (newrow && !defer) {
                            bulk_g2s(dst + Y::kNewOff, static_cast<const T*>(a.k_new) + (size_t)sh * kHeadDim,
                                     2u * kHeadDim, &gfull[st]);
                            bulk_g2s(dst + Y::kNewOff + 2u * kHeadDim,
                                     static_cast<const T*>(a.v_new) + (size_t)sh * kHeadDim, 2u * kHeadDim,
                                     &gfull[st]);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (kRuns && lane < 16) {
                    // lane l copies octet l mod 8 of the chunk (its K rows; lanes 8-15 its V rows):
                    // one bulk copy per stretch of tokens that are consecutive pool rows
                    const int nv = (int)(short)(d.nvalid), hh = d.h, oc = lane & 7;
                    const uint32_t dst = ring + (uint32_t)st * Y::kStageB + (lane >= 8 ? Y::kKB : 0u) +
                                         (uint32_t)oc * kOctB;
                    const T* pool = static_cast<const T*>(lane >= 8 ? a.v_cache : a.k_cache);
                    if (i >= Y::kPStages) fence_proxy_async_smem();
                    bool valid[8], start[8];
                    int len[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        valid[e] = 8 * oc + e < nv;
                        start[e] = valid[e] && (e == 0 || tokq[e] != tokq[e - 1] + 1);
                    }
#pragma unroll
                    for (int e = 7; e >= 0; --e)
                        len[e] = !valid[e] ? 0 : (e < 7 && valid[e + 1] && !start[e + 1]) ? len[e + 1] + 1 : 1;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (start[e])
                            bulk_g2s(dst + (uint32_t)e * (kHeadDim * 2),
                                     pool + ((size_t)tokq[e] + (size_t)hh * B) * kHeadDim,
                                     (uint32_t)len[e] * (kHeadDim * 2), &gfull[st]);
                }
                if (kRuns) {
                    // the next chunk's token entries, in flight while this one lands
                    if (pb + j + 1 < cnt) {
                        const uint4 n0 = reinterpret_cast<const uint4*>(j + 1 < m ? &cur : &nxt)[0];
                        const uint4 n1 = reinterpret_cast<const uint4*>(j + 1 < m ? &cur : &nxt)[1];
                        const int src_lane = j + 1 < m ? j + 1 : 0;
                        const int idx = (int)__shfl_sync(0xffffffffu, n0.x, src_lane);
                        const int nvn = (int)(short)(__shfl_sync(0xffffffffu, n1.z, src_lane) & 0xffffu);
                        const int oc = lane & 7;
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            tokq[e] = lane < 16 && 8 * oc + e < nvn ? __ldg(a.tok + idx + 8 * oc + e) : 0;
                    }
                }
            }
            cur = nxt;
        }
        if (!deps_done) dependency_point(i);
        if (lane == 0) issued[grp] = i;
    } else if (warp == kEpiWarp) {
        // ============================ epilogue ============================
        if (a.early) {
            grid_dependency_wait();   // outputs, partials and flags belong after this point
            grid_launch_dependents();
        }
        // zero the output rows of empty sequences (sequence s handled by CTA s mod C)
        {
            const int32_t* lens = reinterpret_cast<const int32_t*>(a.plan + a.lens_off);
            for (int s = c; s < a.num_seqs; s += (int)gridDim.x)
                if (__ldcg(lens + s) == 0) {
                    uint4* o = reinterpret_cast<uint4*>(static_cast<T*>(a.out) + (size_t)s * Hq * kHeadDim);
                    for (int e = lane; e < Hq * kHeadDim / 8; e += 32) o[e] = make_uint4(0, 0, 0, 0);
                }
        }
        // the cut segments this CTA merges whose pieces all end early (no CTA holds a late piece
        // of them): fold the other CTAs' pieces as their words appear, and this CTA's own
        PlanEvent ev[2];
        bool todo[2];
        for (int side = 0; side < 2; ++side) {
            // 8-byte loads: the second event sits at a multiple of 8 bytes only
            const int2* src = reinterpret_cast<const int2*>(&g_hdr->ev[side]);
            int2* dstv = reinterpret_cast<int2*>(&ev[side]);
#pragma unroll
            for (int j = 0; j < 7; ++j) dstv[j] = __ldcg(src + j);
            todo[side] = b0 < b2 && ev[side].exists && ev[side].merger && !ev[side].by_consumers;
        }
        // four fold lanes per row: lane = 4 r + q owns row r, columns 32 q .. 32 q + 31, as four
        // 8-column shares
        const int r = lane >> 2, cq = (lane & 3) * 32;
        Fold8 acc[2][4];
        int cursor[2];
        bool local_done[2];
        for (int e = 0; e < 2; ++e) {
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[e][j].init();
            cursor[e] = 0;
            local_done[e] = false;
        }
        const unsigned long long t_start = global_timer_ns();
        bool gave_up = false;
        while (todo[0] || todo[1]) {
            if (*abort_flag) break;
            bool progress = false;
            for (int side = 0; side < 2; ++side) {
                if (!todo[side]) continue;
                const PlanEvent& E = ev[side];
                // the other CTAs' pieces in order, each once all of its words are there
                while (cursor[side] < E.nrem) {
                    const int slot = remote_slot(E, bounds, c, cursor[side]);
                    float* po = a.part_o + (size_t)slot * kRows * kHeadDim;
                    float2* pml = a.part_ml + (size_t)slot * kRows;
                    float m[4], l[4], v[4][8];
                    bool got = true;
#pragma unroll
                    for (int j = 0; j < 4; ++j) got = fetch8(po, pml, r, cq + 8 * j, m[j], l[j], v[j]) && got;
                    if (!__all_sync(0xffffffffu, got)) break;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[side][j].add(m[j], l[j], v[j]);
                        clear8(po, pml, r, cq + 8 * j, j == 0 && (lane & 3) == 0);
                    }
                    ++cursor[side];
                    progress = true;
                }
                if (!local_done[side] && mbar_test(&ready[side], 0u)) {
                    const float* so = reinterpret_cast<const float*>(bp + Y::kHandOff + side * kSlotB);
                    const float2* sml =
                        reinterpret_cast<const float2*>(bp + Y::kHandOff + side * kSlotB + kRows * kHeadDim * 4);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float m2, l2, v2[8];
                        slot_load(so, sml, r, cq + 8 * j, m2, l2, v2);
                        acc[side][j].add(m2, l2, v2);
                    }
                    local_done[side] = true;
                    progress = true;
                    if (lane == 0) trace(a.timeline, c, 11);
                }
                if (local_done[side] && cursor[side] >= E.nrem) {
                    if (r < G) {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(a.out) +
                                                              ((size_t)E.s * Hq + (size_t)E.h * G + r) * kHeadDim + cq);
#pragma unroll
                        for (int j = 0; j < 4; ++j) dst[j] = pack8<T>(acc[side][j].num, 1.f / acc[side][j].den);
                    }
                    if (lane == 0 && a.timeline) {
                        a.timeline[(size_t)c * kTimelineSlots + 12] += 1;
                        trace(a.timeline, c, 13);
                    }
                    todo[side] = false;
                    progress = true;
                }
            }
            if (!progress) {
                if (global_timer_ns() - t_start > kWaitLimitNs) {
                    gave_up = true;
                    break;
                }
                __nanosleep(128);   // leave the issue slots to the consumers sharing this scheduler
            }
        }
        if (gave_up && lane == 0) {
            flag_status(a.status, PA_DEV_TIMEOUT);
            *abort_flag = 1;
        }
        if (lane == 0) trace(a.timeline, c, 10);
    } else {
        // ============================ consumers of one group ============================
        const int grp = warp / kGroupWarps, wq = warp % kGroupWarps, tg = tid - grp * kGroupThreads;
        const int gid = lane >> 2, tig = lane & 3;
        const int t_warp = wq * 16;
        const int lo = grp ? b1 : b0, hi = grp ? b2 : b1;
        const int cnt = hi - lo;
        uint64_t* gfull = full + grp * Y::kPStages;
        uint64_t* gempty = empty + grp * Y::kPStages;
        const uint32_t ring = base + (uint32_t)grp * Y::kPStages * Y::kStageB;
        unsigned char* ring_p = bp + (size_t)grp * Y::kPStages * Y::kStageB;
        const int tokA = t_warp + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int chA = lane >> 4;
        const int tokV = t_warp + (lane & 7) + ((lane >> 4) << 3);
        const int chV = (lane >> 3) & 1;
        float m_run[2], l_run[2], o[8][4];
        uint32_t qb[8][2];
        if (a.early) {
            grid_dependency_wait();   // q, the new rows and every output belong after this point
            grid_launch_dependents();
            if (tid == 0) trace(a.timeline, c, 1);
        }
        // A warp that gave up on a wait is "dead": it keeps walking the group's chunks without
        // waiting or writing.  Warps die only on the group's shared barriers (a stage that never
        // lands times every warp of the group out at the same chunk), so all four keep taking
        // the same named-barrier path through the segment ends.
        bool dead = false;
        for (int i = 0; i < cnt; ++i) {
            const int st = i % Y::kPStages;
            if (!dead && !__all_sync(0xffffffffu, mbar_wait_bounded(&gfull[st], (uint32_t)(i / Y::kPStages) & 1u))) {
                if (lane == 0) {
                    flag_status(a.status, PA_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
                dead = true;
            }
            if (grp == 0 && tid == 0 && a.timeline) {
                if (i == 0) trace(a.timeline, c, 5);
                if (i == cnt - 1) trace(a.timeline, c, 6);
            }
            const uint32_t kbase = ring + (uint32_t)st * Y::kStageB;
            const uint32_t vbase = kbase + Y::kKB;
            unsigned char* stage_p = ring_p + (size_t)st * Y::kStageB;
            const StageMeta* meta = reinterpret_cast<const StageMeta*>(stage_p + Y::kMetaOff);
            const int flags = dead ? 0 : meta->flags;
            const int nvalid = dead ? 0 : meta->nvalid;
            if ((flags & (kBegin | kNewRow)) && a.early && i < Y::kPStages) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&qbar[grp], 0u))) {
                    if (lane == 0) {
                        flag_status(a.status, PA_DEV_TIMEOUT);
                        *abort_flag = 1;
                    }
                    dead = true;
                }
            }
            if ((flags & kBegin) && !dead) {
                const uint32_t* qs = reinterpret_cast<const uint32_t*>(stage_p + Y::kQOff);
                const int row = gid;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int wcol = (ks * 16 + tig * 2) >> 1;
                    qb[ks][0] = (row < G) ? qs[row * 64 + wcol] : 0u;
                    qb[ks][1] = (row < G) ? qs[row * 64 + wcol + 4] : 0u;
                }
                m_run[0] = m_run[1] = -INFINITY;
                l_run[0] = l_run[1] = 0.f;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
            }
            // runs stages: this warp's row x (0..15) holds token 8 (x mod 8) + 2 wq + x / 8
            if ((kRuns ? 2 * wq < nvalid : t_warp < nvalid) && !dead) {
                if (kRuns) {
                    if (nvalid < 64) {
                        // V rows past the context: stale rows must not meet P = 0 as non-finite values
                        uint4* vz = reinterpret_cast<uint4*>(stage_p + Y::kKB);
                        for (int idx = lane; idx < 16 * 16; idx += 32) {
                            const int x = idx >> 4;
                            if (8 * (x & 7) + 2 * wq + (x >> 3) >= nvalid)
                                vz[((uint32_t)(x & 7) * kOctB + (uint32_t)(2 * wq + (x >> 3)) * (kHeadDim * 2)) / 16 +
                                   (idx & 15)] = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                } else if (nvalid < t_warp + 16) {
                    // V rows past the context: stale pool rows must not meet P = 0 as non-finite values
                    uint4* vz = reinterpret_cast<uint4*>(stage_p + Y::kKB);
                    for (int idx = lane; idx < (t_warp + 16 - nvalid) * 16; idx += 32) {
                        const int t = nvalid + (idx >> 4);
                        const int cc = idx & 15;
                        vz[line_of(t, cc >> 3, R_log2) * 8 + (cc & 7)] = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                const int tn = nvalid - 1;
                if ((flags & kNewRow) && (tn >> 4) == wq) {
                    // the new K/V row: into the staged tile and into its cache slot
                    const int cc = lane & 15;
                    const bool isv = lane >= 16;
                    const uint4 val = *reinterpret_cast<const uint4*>(stage_p + Y::kNewOff + (isv ? 2u * kHeadDim : 0u) +
                                                                      cc * 16);
                    st_shared_v4(kv_addr<kRuns>(isv ? vbase : kbase, tn, cc, R_log2), val);
                    const int phys = meta->new_phys;
                    if (phys >= 0) {
                        const size_t row = ((size_t)phys * Hkv + meta->h) * B + (size_t)meta->new_off;
                        T* cache = const_cast<T*>(static_cast<const T*>(isv ? a.v_cache : a.k_cache));
                        *reinterpret_cast<uint4*>(cache + row * kHeadDim + cc * 8) = val;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                // S^T = K Q^T over the warp's 16 tokens, two accumulator chains
                float sc[4] = {0.f, 0.f, 0.f, 0.f}, sc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(kv_addr<kRuns>(kbase, tokA, 2 * ks + chA, R_log2), a0, a1, a2, a3);
                    if (ks & 1) mma16816<T>(sc2, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                    else mma16816<T>(sc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                }
                const bool in0 = kRuns ? 8 * gid + 2 * wq < nvalid : t_warp + gid < nvalid;
                const bool in1 = kRuns ? 8 * gid + 2 * wq + 1 < nvalid : t_warp + gid + 8 < nvalid;
                constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
                float xs[4];
                bool move = false;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    xs[j] = in0 ? (sc[j] + sc2[j]) * a.scale_log2 : -INFINITY;
                    xs[2 + j] = in1 ? (sc[2 + j] + sc2[2 + j]) * a.scale_log2 : -INFINITY;
                    move = move || xs[j] > m_run[j] + kLazyLog2 || xs[2 + j] > m_run[j] + kLazyLog2;
                }
                if (__any_sync(0xffffffffu, move)) {
                    float alpha[2];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float mx = fmaxf(xs[j], xs[2 + j]);
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        const float m_new = fmaxf(m_run[j], mx);
                        alpha[j] = (m_new == -INFINITY) ? 1.f : exp2f(m_run[j] - m_new);
                        m_run[j] = m_new;
                        l_run[j] *= alpha[j];
                    }
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        o[mt][0] *= alpha[0];
                        o[mt][1] *= alpha[1];
                        o[mt][2] *= alpha[0];
                        o[mt][3] *= alpha[1];
                    }
                }
                float pv[4];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float m_use = (m_run[j] == -INFINITY) ? 0.f : m_run[j];
                    pv[j] = exp2f(xs[j] - m_use);
                    pv[2 + j] = exp2f(xs[2 + j] - m_use);
                    l_run[j] += pv[j] + pv[2 + j];
                }
                const uint32_t h0 = Elem<T>::pack2(pv[0], pv[1]), h1 = Elem<T>::pack2(pv[2], pv[3]);
                const uint32_t pb0 = movmatrix_trans(h0), pb1 = movmatrix_trans(h1);
                uint32_t pl0 = 0, pl1 = 0;
                if (kSplitP) {
                    const float2 r0 = Elem<T>::to_float2(h0), r1 = Elem<T>::to_float2(h1);
                    pl0 = movmatrix_trans(Elem<T>::pack2(pv[0] - r0.x, pv[1] - r0.y));
                    pl1 = movmatrix_trans(Elem<T>::pack2(pv[2] - r1.x, pv[3] - r1.y));
                }
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(kv_addr<kRuns>(vbase, tokV, 2 * mt + chV, R_log2), a0, a1, a2, a3);
                    mma16816<T>(o[mt], a0, a1, a2, a3, pb0, pb1);
                    if (kSplitP) mma16816<T>(o[mt], a0, a1, a2, a3, pl0, pl1);
                }
            }

            if (flags & kEnd) {
                // ---- the segment's last chunk in this group's order: merge the four warps ----
                float lr[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float v = l_run[j];
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    lr[j] = v;
                }
                float* red_o = reinterpret_cast<float*>(stage_p);                                  // [4][8][kRedStride]
                float2* red_ml = reinterpret_cast<float2*>(red_o + kGroupWarps * 8 * kRedStride);  // [4][8]
                group_sync(grp);   // every warp is past its reads of the stage
                // rows past the GQA group carry nothing: only the group's rows go through shared
                // memory, the others fold to a neutral (m 0, l 1, o 0) partial
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int row = tig * 2 + j;
                    if (row < G) {
                        float* dst = &red_o[(wq * 8 + row) * kRedStride + gid];
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            dst[mt * 16] = o[mt][j];
                            dst[mt * 16 + 8] = o[mt][2 + j];
                        }
                        if (gid == 0) red_ml[wq * 8 + row] = make_float2(m_run[j], lr[j]);
                    }
                }
                group_sync(grp);
                const int r = tg >> 4, d0 = (tg & 15) * 8;
                Fold8 f;
                f.init();
                if (r >= G) {
                    f.M = 0.f;
                    f.den = 1.f;
                } else {
                    float M = -INFINITY;
#pragma unroll
                    for (int w2 = 0; w2 < kGroupWarps; ++w2) M = fmaxf(M, red_ml[w2 * 8 + r].x);
                    f.M = M;
#pragma unroll
                    for (int w2 = 0; w2 < kGroupWarps; ++w2) {
                        const float2 ml = red_ml[w2 * 8 + r];
                        // a warp without a valid token (m = -inf) weighs 0
                        const float wgt = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
                        f.den = fmaf(wgt, ml.y, f.den);
                        const float4 x0 = *reinterpret_cast<const float4*>(&red_o[(w2 * 8 + r) * kRedStride + d0]);
                        const float4 x1 = *reinterpret_cast<const float4*>(&red_o[(w2 * 8 + r) * kRedStride + d0 + 4]);
                        f.num[0] = fmaf(wgt, x0.x, f.num[0]);
                        f.num[1] = fmaf(wgt, x0.y, f.num[1]);
                        f.num[2] = fmaf(wgt, x0.z, f.num[2]);
                        f.num[3] = fmaf(wgt, x0.w, f.num[3]);
                        f.num[4] = fmaf(wgt, x1.x, f.num[4]);
                        f.num[5] = fmaf(wgt, x1.y, f.num[5]);
                        f.num[6] = fmaf(wgt, x1.z, f.num[6]);
                        f.num[7] = fmaf(wgt, x1.w, f.num[7]);
                    }
                }
                const int s = meta->s, h = meta->h, side = meta->side;
                int mode = dead ? -1 : meta->mode;
                if (mode == kPairM) {
                    // the two groups of this CTA meet: the first to arrive leaves its piece in the
                    // pair slot, the second folds it in and carries on with the segment
                    if (tg == 0) pair_role[grp] = atomicAdd(const_cast<int*>(pair_count), 1);
                    group_sync(grp);
                    if (pair_role[grp] == 0) {
                        slot_store(pair_o, pair_ml, r, d0, f, (tg & 15) == 0);
                        mbar_arrive(pair_bar);
                        mode = -1;
                    } else if (!group_all(grp, mbar_wait_bounded(pair_bar, 0u))) {
                        if (tg == 0) {
                            flag_status(a.status, PA_DEV_TIMEOUT);
                            *abort_flag = 1;
                        }
                        mode = -1;
                    } else {
                        float m2, l2, v2[8];
                        slot_load(pair_o, pair_ml, r, d0, m2, l2, v2);
                        f.add(m2, l2, v2);
                        mode = meta->post;
                    }
                }
                if (mode == kMergeHereM) {
                    // the last piece of a segment this CTA merges: fold the other CTAs' pieces here,
                    // up to four at a time with all their loads in flight, each once every word of it
                    // has been published
                    const PlanEvent& E = sh_hdr->ev[side];
                    const int nrem = E.nrem;
                    const unsigned long long t0 = global_timer_ns();
                    bool ok = true;   // the same in every thread of the group
                    for (int k0 = 0; k0 < nrem && ok; k0 += 4) {
                        const int kn = min(4, nrem - k0);
                        int slot[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) slot[j] = j < kn ? remote_slot(E, bounds, c, k0 + j) : 0;
                        unsigned done_mask = 0, want = (1u << kn) - 1u;
                        while (done_mask != want) {
                            float m2[4], l2[4], v2[4][8];
                            bool got[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                got[j] = false;
                                if (j < kn && !(done_mask & (1u << j)))
                                    got[j] = fetch8(a.part_o + (size_t)slot[j] * kRows * kHeadDim,
                                                    a.part_ml + (size_t)slot[j] * kRows, r, d0, m2[j], l2[j], v2[j]);
                            }
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                if (got[j]) {
                                    f.add(m2[j], l2[j], v2[j]);
                                    done_mask |= 1u << j;
                                }
                            if (done_mask != want && global_timer_ns() - t0 > kWaitLimitNs) break;
                        }
                        // A row's (m, l) words are read by its 16 threads and cleared by one of them:
                        // clear only once every thread of the group has stopped reading the batch.
                        ok = group_all(grp, done_mask == want);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (done_mask & (1u << j))
                                clear8(a.part_o + (size_t)slot[j] * kRows * kHeadDim, a.part_ml + (size_t)slot[j] * kRows,
                                       r, d0, (tg & 15) == 0);
                    }
                    if (!ok) {
                        if (tg == 0) {
                            flag_status(a.status, PA_DEV_TIMEOUT);
                            *abort_flag = 1;
                        }
                        mode = -1;
                    } else {
                        mode = kOutM;
                    }
                    if (tg == 0 && a.timeline) a.timeline[(size_t)c * kTimelineSlots + 12] += 1;
                }
                if (mode == kOutM) {
                    if (r < G) {
                        const float inv = 1.f / f.den;
                        *reinterpret_cast<uint4*>(static_cast<T*>(a.out) + ((size_t)s * Hq + (size_t)h * G + r) * kHeadDim +
                                                  d0) = pack8<T>(f.num, inv);
                    }
                } else if (mode == kPublishM) {
                    // the stored words are the publication (the merger waits until none is empty)
                    const size_t slot = (size_t)2 * c + side;
                    publish8(a.part_o + slot * kRows * kHeadDim, a.part_ml + slot * kRows, r, d0, f, (tg & 15) == 0);
                } else if (mode == kMergeM) {
                    float* so = reinterpret_cast<float*>(bp + Y::kHandOff + side * kSlotB);
                    float2* sml = reinterpret_cast<float2*>(bp + Y::kHandOff + side * kSlotB + kRows * kHeadDim * 4);
                    slot_store(so, sml, r, d0, f, (tg & 15) == 0);
                    mbar_arrive(&ready[side]);
                }
                group_sync(grp);   // the scratch (this stage) is free again
                fence_proxy_async_smem();
            }
            mbar_arrive(&gempty[st]);
        }
        if (kAdaptive && tid == 0) cp_async_wait_all();   // the rate copied at the start
        if (grp == 0 && tid == 0) trace(a.timeline, c, 7);
        if (grp == 1 && tg == 0) trace(a.timeline, c, 9);
    }

    __syncthreads();
    if (kAdaptive && tid == kEpiWarp * 32 && sh_hdr->weight != 0.f && !*abort_flag) {
        // adaptive plan: this CTA's rate, the weight of its range per SM cycle of its life
        const float w = fabsf(sh_hdr->weight);
        const unsigned span = (unsigned)clock() - (unsigned)misc[30];
        const float r = (sh_hdr->b2 > sh_hdr->b0 && span > 0u && span < 0x40000000u) ? w / (float)span : 0.f;
        const float old_rate = __int_as_float(misc[29]);
        if (sh_hdr->weight < 0.f) {   // the rates hold no measurement yet
            a.rates->rate[c] = r;   // 0: no measurement
            if (c == 0) {
                a.rates->magic = kRatesMagic;
                a.rates->ctas = (int)gridDim.x;
            }
        } else if (r > 0.f) {
            a.rates->rate[c] = old_rate > 0.f && old_rate < kRateMax ? old_rate + kRateAlpha * (r - old_rate) : r;
        }
    }
    if (tid == 0 && a.timeline) {
        trace(a.timeline, c, 8);
        unsigned int smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        trace_put(a.timeline, c, 14, (unsigned long long)(b2 - b0));
        trace_put(a.timeline, c, 15, smid);
    }
    if (*abort_flag && tid == 0) {
        // let every copy still in flight land before the CTA's shared memory is released
        for (int grp = 0; grp < kGroups; ++grp) {
            const int n = issued[grp];
            for (int st = 0; st < Y::kPStages; ++st) {
                int last = -1;
                for (int i = st; i < n; i += Y::kPStages) last = i;
                if (last >= 0) (void)mbar_wait_bounded(&full[grp * Y::kPStages + st], (uint32_t)(last / Y::kPStages) & 1u);
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Contexts given as runs (block, slot offset, length): one warp per sequence lays its tokens out in
// a token table, (block * Hkv) * B + slot per token, and sums its length; the plan kernel then
// cuts chunks as for a block table and the decode's producers copy each token's K and V row.
// ---------------------------------------------------------------------------------------------

__global__ void __launch_bounds__(256) runs_prep_kernel(const int32_t* runs, const int32_t* seq_runs, int num_seqs,
                                                         int num_kv_heads, int block_size, int num_blocks,
                                                         int max_context, int stride, int32_t* lens, int32_t* tok,
                                                         unsigned int* status) {
    const int s = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (s >= num_seqs) return;
    int r0 = seq_runs[s], r1 = seq_runs[s + 1];
    if (r0 < 0 || r1 < r0) {   // a malformed run range: an empty context
        if (lane == 0) flag_status(status, PA_DEV_BAD_BLOCK_ID);
        r0 = r1 = 0;
    }
    int pos = 0;
    for (int rb = r0; rb < r1; rb += 32) {
        const int r = rb + lane;
        int blk = 0, off = 0, len = 0;
        if (r < r1) {
            blk = runs[3 * r];
            off = runs[3 * r + 1];
            len = runs[3 * r + 2];
            if (blk < 0 || blk >= num_blocks || off < 0 || len < 0 || off + len > block_size) {
                flag_status(status, PA_DEV_BAD_BLOCK_ID);   // the run counts as empty
                len = 0;
            }
        }
        int incl = len;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const int start = pos + incl - len;
        const int base = (blk * num_kv_heads) * block_size + off;
        for (int t = 0; t < len && start + t < max_context; ++t) tok[(size_t)s * stride + start + t] = base + t;
        pos += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        if (pos > max_context) {
            flag_status(status, PA_DEV_BAD_CONTEXT);
            pos = max_context;
        }
        lens[s] = pos;
    }
}

template <typename T, bool kAdaptive, bool kRuns>
cudaError_t launch_planned_impl(const PlannedArgs& a, const MmaMapsP& maps, int R_log2, int ctas, cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    auto kernel = decode_planned_kernel<T, kAdaptive, kRuns>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lay<kRuns>::kSmem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = Lay<kRuns>::kSmem;
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

int planned_ctas(const pa_decode_options* opts) {
    const int sms = sm_count_current();
    if (opts && opts->num_ctas > 0) return opts->num_ctas < sms ? opts->num_ctas : sms;
    return sms;
}

size_t planned_plan_bytes(int num_seqs, int num_kv_heads, int block_size, int max_blocks_per_seq, int ctas,
                          bool adaptive) {
    return plan_layout(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas, adaptive).total;
}

void planned_plan_offsets(int num_seqs, int num_kv_heads, int block_size, int max_blocks_per_seq, int ctas,
                          bool adaptive, size_t* bounds_offset, size_t* rates_offset) {
    const PlanLayout L = plan_layout(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas, adaptive);
    *bounds_offset = L.bounds;
    *rates_offset = L.rates + offsetof(PlanRates, rate);
}

size_t planned_workspace_bytes(int ctas) {
    const size_t slots = (size_t)2 * ctas;
    return al256(slots * kRows * kHeadDim * sizeof(float)) + al256(slots * kRows * sizeof(float2));
}

static cudaError_t launch_plan_kernel(void* plan, const int32_t* block_tables, const int32_t* context_lens,
                                      int num_seqs, int num_q_heads, int num_kv_heads, int block_size,
                                      int num_blocks, int max_blocks_per_seq, int ctas, bool adaptive,
                                      int tok_stride, cudaStream_t stream);

cudaError_t launch_decode_plan(void* plan, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                               int num_q_heads, int num_kv_heads, int block_size, int num_blocks,
                               int max_blocks_per_seq, int ctas, bool adaptive, cudaStream_t stream) {
    return launch_plan_kernel(plan, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads, block_size,
                              num_blocks, max_blocks_per_seq, ctas, adaptive, 0, stream);
}

static cudaError_t launch_plan_kernel(void* plan, const int32_t* block_tables, const int32_t* context_lens,
                                      int num_seqs, int num_q_heads, int num_kv_heads, int block_size,
                                      int num_blocks, int max_blocks_per_seq, int ctas, bool adaptive,
                                      int tok_stride, cudaStream_t stream) {
    if (ctas < 1 || ctas > 4 * kPlanThreads) return cudaErrorInvalidValue;
    const PlanLayout L = plan_layout(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas, adaptive);
    PlanArgs a;
    a.plan = static_cast<unsigned char*>(plan);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.status = device_status_ptr();
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.ctas = ctas;
    a.lens_off = L.lens;
    a.bounds_off = L.bounds;
    a.cta_off = L.cta;
    a.cta_bytes = L.cta_bytes;
    a.rates_off = L.rates;
    a.cap = L.cap;
    a.adaptive = adaptive ? 1 : 0;
    a.tok_stride = tok_stride;
    a.max_chunks = plan_max_chunks(num_seqs, num_kv_heads, block_size, max_blocks_per_seq);
    long long blocks = (a.max_chunks + kPlanThreads - 1) / kPlanThreads;
    const long long cap = 4LL * sm_count_current();
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const size_t smem = (size_t)(num_seqs + 1) * sizeof(long long) + (size_t)(3 * num_seqs + 1) * sizeof(int) +
                        (size_t)(2 * ctas + 1) * sizeof(int32_t) + (size_t)(ctas + 1) * sizeof(float);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(decode_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_plan_kernel, a);
    if (e == cudaSuccess) note_launches(1);
    return e;
}

cudaError_t launch_decode_planned(void* out, const void* q, const void* k_new, const void* v_new, const void* k_cache,
                                  const void* v_cache, void* plan, void* workspace, float scale, int num_seqs,
                                  int num_q_heads, int num_kv_heads, int block_size, int num_blocks,
                                  int max_blocks_per_seq, int dtype, int ctas, bool early, bool adaptive,
                                  unsigned long long* timeline, cudaStream_t stream) {
    const int R = block_size < kStageTokens ? block_size : kStageTokens;
    int R_log2 = 0;
    while ((1 << R_log2) < R) ++R_log2;
    const unsigned long long rows = (unsigned long long)num_blocks * num_kv_heads * block_size;
    if (rows == 0 || rows > 0x7fffffffull) return cudaErrorInvalidValue;
    MmaMapsP maps;
    if (!encode_pool_map(k_cache, rows, R, &maps.k) || !encode_pool_map(v_cache, rows, R, &maps.v))
        return cudaErrorInvalidValue;
    const PlanLayout L = plan_layout(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas, adaptive);
    PlannedArgs a;
    a.out = out;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.plan = static_cast<const unsigned char*>(plan);
    a.rates = reinterpret_cast<PlanRates*>(static_cast<unsigned char*>(plan) + L.rates);
    a.tok = nullptr;
    const size_t slots = (size_t)2 * ctas;
    char* w = static_cast<char*>(workspace);
    a.part_o = reinterpret_cast<float*>(w);
    a.part_ml = reinterpret_cast<float2*>(w + al256(slots * kRows * kHeadDim * sizeof(float)));

    a.status = device_status_ptr();
    a.timeline = timeline;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.early = early ? 1 : 0;
    a.cap = L.cap;
    a.lens_off = L.lens;
    a.bounds_off = L.bounds;
    a.cta_off = L.cta;
    a.cta_bytes = L.cta_bytes;
    if (adaptive)
        return dtype == PA_BF16 ? launch_planned_impl<__nv_bfloat16, true, false>(a, maps, R_log2, ctas, stream)
                                : launch_planned_impl<__half, true, false>(a, maps, R_log2, ctas, stream);
    return dtype == PA_BF16 ? launch_planned_impl<__nv_bfloat16, false, false>(a, maps, R_log2, ctas, stream)
                            : launch_planned_impl<__half, false, false>(a, maps, R_log2, ctas, stream);
}

// Runs plans: the plan, then the prep kernel's lengths and token table.
struct RunsLayout {
    PlanLayout plan;
    size_t lens, tok, total;
    int stride;
};

static RunsLayout runs_layout(int num_seqs, int num_kv_heads, int block_size, int max_blocks_per_seq, int ctas) {
    RunsLayout R;
    const long long max_context = (long long)max_blocks_per_seq * block_size;
    R.stride = (int)((max_context + kStageTokens - 1) / kStageTokens * kStageTokens);
    R.plan = plan_layout(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas, false);
    R.lens = al256(R.plan.total);
    R.tok = R.lens + al256((size_t)num_seqs * 4);
    R.total = R.tok + al256((size_t)num_seqs * R.stride * 4);
    return R;
}

size_t planned_runs_plan_bytes(int num_seqs, int num_kv_heads, int block_size, int max_blocks_per_seq, int ctas) {
    return runs_layout(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas).total;
}

cudaError_t launch_decode_plan_runs(void* plan, const int32_t* runs, const int32_t* seq_runs, int num_seqs,
                                    int num_q_heads, int num_kv_heads, int block_size, int num_blocks,
                                    int max_blocks_per_seq, int max_context, int ctas, cudaStream_t stream) {
    const RunsLayout RL = runs_layout(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas);
    unsigned char* buf = static_cast<unsigned char*>(plan);
    int32_t* lens = reinterpret_cast<int32_t*>(buf + RL.lens);
    int32_t* tok = reinterpret_cast<int32_t*>(buf + RL.tok);
    const unsigned warps_per_block = 8;
    runs_prep_kernel<<<(unsigned)((num_seqs + warps_per_block - 1) / warps_per_block), 32 * warps_per_block, 0,
                       stream>>>(runs, seq_runs, num_seqs, num_kv_heads, block_size, num_blocks, max_context,
                                 RL.stride, lens, tok, device_status_ptr());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    note_launches(1);
    return launch_plan_kernel(buf, nullptr, lens, num_seqs, num_q_heads, num_kv_heads, block_size, num_blocks,
                              max_blocks_per_seq, ctas, false, RL.stride, stream);
}

cudaError_t launch_decode_planned_runs(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const void* plan, void* workspace, float scale, int num_seqs,
                                       int num_q_heads, int num_kv_heads, int block_size, int num_blocks,
                                       int max_blocks_per_seq, int dtype, int ctas, bool early,
                                       unsigned long long* timeline, cudaStream_t stream) {
    const RunsLayout RL = runs_layout(num_seqs, num_kv_heads, block_size, max_blocks_per_seq, ctas);
    const PlanLayout& L = RL.plan;
    const unsigned char* buf = static_cast<const unsigned char*>(plan);
    PlannedArgs a;
    a.out = out;
    a.q = q;
    a.k_new = nullptr;
    a.v_new = nullptr;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.plan = buf;
    a.rates = nullptr;
    a.tok = reinterpret_cast<const int32_t*>(buf + RL.tok);
    const size_t slots = (size_t)2 * ctas;
    char* w = static_cast<char*>(workspace);
    a.part_o = reinterpret_cast<float*>(w);
    a.part_ml = reinterpret_cast<float2*>(w + al256(slots * kRows * kHeadDim * sizeof(float)));
    a.status = device_status_ptr();
    a.timeline = timeline;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.early = early ? 1 : 0;
    a.cap = L.cap;
    a.lens_off = L.lens;
    a.bounds_off = L.bounds;
    a.cta_off = L.cta;
    a.cta_bytes = L.cta_bytes;
    MmaMapsP maps;
    std::memset(&maps, 0, sizeof(maps));   // (the runs form copies rows, no tensor maps)
    return dtype == PA_BF16 ? launch_planned_impl<__nv_bfloat16, false, true>(a, maps, 6, ctas, stream)
                            : launch_planned_impl<__half, false, true>(a, maps, 6, ctas, stream);
}

}  // namespace pa
