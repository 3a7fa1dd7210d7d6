// Paged decode attention: persistent, load-balanced, tensor-core kernel (one launch per call).
//
// What it computes ("显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结", §五.1): for every
// sequence and query head, walk the sequence's logical blocks through its block-table row,
// q.k for every cached token, softmax with a running maximum, weight V, normalise at the end.
// Address rule: "端侧 SLM 显存保活术：在 4GB 内存板卡上实现轻量 PagedAttention 与 KV 缓存分块",
// section "注意力寻址：非连续物理块的间接寻址内核".
//
// Work decomposition.  A segment is one (sequence, kv head); it is cut into 64-token chunks.
// All chunks of all segments form one list of N chunks (sequence-major); the grid holds as many
// CTAs as can be resident at once, and CTA c streams the contiguous chunk range
// [N c / C, N (c + 1) / C).  Every CTA therefore moves the same number of bytes, and its TMA
// ring stays full across segment boundaries.  A segment that lies inside one CTA's range is
// finished there; a segment cut by range boundaries leaves one partial (m, l, o) per CTA and
// the last CTA to finish its piece (a per-segment arrival counter) merges the pieces.
//
// Inside a CTA: one producer warp issues, per chunk, the 2-D TMA tensor loads of the K and V
// rows (128-byte swizzle) and, at the first chunk of a segment, a bulk copy of the segment's
// query rows; four consumer warps each own 16 of the chunk's 64 tokens and run the products
// transposed, tokens and head dimensions on the 16-row side of mma.sync m16n8k16 and the GQA
// group's query rows on its 8-column side:
//   S^T = K Q^T  and  O^T += V^T P^T   (fp32 accumulation),
// so that a group of up to 8 query rows fills every row of every product, keeping a running
// max / sum per query row.  At a segment's last chunk the four warps merge
// through the stage buffer they just consumed.  Full / empty mbarriers per stage connect the
// producer and the consumers; every wait is bounded.
//
// Several query tokens per sequence (q_start): a segment's query rows are its new tokens x the
// GQA group (at most 16), token i of n sitting at position L - n + i and attending causally up
// to it; the per-row position limits enter the mask, the rest is unchanged.
//
// Finishing a cut segment costs dependent round trips to L2 (publish the partial, count the
// arrival, read the other pieces), slow while the copies of every CTA queue in front of them.
// Only the first piece of a range can end before the range does; the consumers hand it to an
// epilogue warp (publish on a shared-memory barrier, move on) which does the arrival and, if
// last, the merge while the stream continues.  The range's final piece is finished by the
// consumers themselves, with all their threads, when nothing is left to stream.
#include "decode_common.cuh"

#include <atomic>
#include <climits>
#include <type_traits>

namespace pa {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kProducerWarp = kConsumerWarps;      // issues the copies
constexpr int kEpilogueWarp = kConsumerWarps + 1;  // finishes the range's first piece off the stream
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kKBytes = kStageTokens * kHeadDim * 2;   // 16 KB of K per stage (V the same)
constexpr int kKVBytes = 2 * kKBytes;
constexpr int kRedStride = kHeadDim + 4;                // padded rows of the merge scratch (bank spread)
constexpr int kMergeBatch = 4;                          // pieces whose loads are in flight together
constexpr float kLazyLog2 = 8.f;                        // exponent base lags the running max by < 2^8

// Trace slots of one CTA: event times (global ns), then accumulated times and counters.
enum : int {
    kTrEntry = 0,       // CTA starts
    kTrDeps = 1,        // the dependency wait on the preceding kernel has passed
    kTrScan = 2,        // prefix sums of the chunk counts are in shared memory
    kTrIds = 3,         // producer: block ids of the first chunk have been read
    kTrIssue = 4,       // producer: copies of the first chunk issued
    kTrFirst = 5,       // consumers: first chunk landed
    kTrLastLanded = 6,  // consumers: last chunk landed
    kTrLoopEnd = 7,     // consumers: last chunk consumed and flushed
    kTrExit = 8,        // CTA ends
    kTrWaitFull = 9,    // consumer warp 0: ns spent waiting for chunks to land
    kTrFlush = 10,      // consumer warp 0: ns spent finishing segments (merges included)
    kTrWaitEmpty = 11,  // producer: ns spent waiting for a free stage
    kTrMerges = 12,     // cut segments this CTA merged
    kTrFlushes = 13,    // segment pieces this CTA finished
    kTrChunks = 14,     // chunks streamed
    kTrSm = 15          // SM the CTA ran on
};

// Shared-memory layout for a ring of kStages 64-token stages: 3 stages let two CTAs share an
// SM, 6 stages give one CTA the whole SM.
template <bool kG16, int kStages>
struct PLayout {
    static constexpr int kQRows = kG16 ? 16 : 8;
    static constexpr int kStageBytes = kKVBytes + kQRows * kHeadDim * 2;  // multiple of 1024
    static constexpr size_t kRing = (size_t)kStages * kStageBytes;
    static constexpr size_t kBars = kRing;   // full[kStages], empty[kStages], q, piece, landed barriers, pad
    static constexpr size_t kFlags = kBars + (2 * kStages + 4) * sizeof(uint64_t);
    static constexpr size_t kNewPhys = kFlags + 16;   // int [kStages] block of the new token, then
                                                       // int [kStages] deferred q rows (s * Hkv + h), then
                                                       // int [kStages] x 2 first q row / query tokens of
                                                       // the segment a stage starts
    static constexpr size_t kPrefix = kNewPhys + ((4 * kStages * sizeof(int32_t) + 15) & ~size_t(15));
    // then int P[S + 1], int L[S] and, for the weighted cut, int E[S + 1]
    static constexpr size_t total(int num_seqs, bool weighted = false) {
        return 1024 /*alignment slack*/ + kPrefix +
               (size_t)(2 * num_seqs + 1 + (weighted ? num_seqs + 1 : 0)) * sizeof(int32_t);
    }
    static_assert(1024 + kPrefix + (2 * kPersistMaxSeqs + 1) * sizeof(int32_t) <= 227 * 1024,
                  "one CTA's shared memory must fit in 227 KB");
    static_assert(kStageBytes % 1024 == 0, "stage buffers must stay 1024-aligned");
};
static_assert(kConsumerWarps * 8 * kRedStride * 4 + kConsumerWarps * 8 * 8 <= kKVBytes, "merge scratch");

// Tensor maps of the two pools, boxes of R = min(block_size, 64) rows.
struct MmaMaps {
    CUtensorMap k;
    CUtensorMap v;
};

// The kernel for many segment ends per CTA also has boxes of R / 2 and R / 4 rows: a chunk's last
// block is fetched with the lowest box that covers its valid rows.  (Other kernels keep the two
// maps: a rarely used descriptor is a cold fetch on a CTA's critical path.)
struct MmaMapsTails {
    CUtensorMap k;
    CUtensorMap v;
    CUtensorMap k2, v2;
    CUtensorMap k4, v4;
};

template <bool kManyEnds>
using MapsOf = typename std::conditional<kManyEnds, MmaMapsTails, MmaMaps>::type;

constexpr int kConsumerThreads = kConsumerWarps * 32;

// Barrier of the 128 consumer threads (hardware named barrier 1).  Every consumer warp walks
// the same chunk sequence and reaches the same barriers, also after it gave up on a copy (it
// then skips waits, math and global writes), so no warp can be left waiting here.
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// The cut of the chunk list into the ranges of the C CTAs that take part.
//   Plain (W == 0): equal chunk counts, range c = [floor(N c / C), floor(N (c + 1) / C)).
//   Weighted: chunk g of segment (s, h) sits at weight u g + e (E[s] + h), E[s] being the
//   non-empty segments before sequence s, so that every segment end weighs e on top of its
//   chunk's u; range c holds the chunks whose weight w has floor(w C / W) == c, W the total.
//   Used when a CTA finishes many segments (the cost of a segment's end then rivals that of
//   its chunks) and only while W >= (u + e) C, which leaves no range empty.
// Quotient of non-negative 64-bit integers, through the 32-bit divide when both fit (the
// partition's numbers nearly always do, and the 64-bit divide is a long software sequence).
__device__ __forceinline__ long long div_nn(long long x, long long y) {
    if (((unsigned long long)x | (unsigned long long)y) >> 32 == 0) return (long long)((uint32_t)x / (uint32_t)y);
    return x / y;
}

struct Cut {
    long long N;        // chunks
    int C;              // CTAs that take part
    long long W;        // total weight, 0 for the plain cut
    int u, e;
    const int32_t* P;   // [S + 1] first chunk of each sequence
    const int32_t* E;   // [S + 1] non-empty segments before each sequence (weighted cut)
};

// The cut as the prefix sums in shared memory define it (P[S] chunks; E follows Lc, i.e. starts
// at P + 2 S + 1).  Rebuilt where it is needed rather than kept live through the chunk loop.
// Kernels built without kManyEnds always cut plainly (their code carries none of the weighted cut).
template <bool kManyEnds>
__device__ __forceinline__ Cut make_cut(const DecodeArgs& a, const int32_t* P, int S) {
    Cut k;
    k.P = P;
    k.E = P + 2 * S + 1;
    k.N = P[S];
    k.C = k.N > 0 ? (int)min((long long)gridDim.x, k.N) : 0;
    k.u = a.cut_unit;
    k.e = a.cut_seg;
    k.W = 0;
    if (kManyEnds && a.cut_seg > 0 && k.C > 0) {
        const long long W = (long long)k.u * k.N + (long long)k.e * k.E[S];
        if (W >= (long long)(k.u + k.e) * k.C) k.W = W;
    }
    return k;
}

__device__ __forceinline__ long long cut_weight(const Cut& k, long long g, int s, int h) {
    return (long long)k.u * g + (long long)k.e * (k.E[s] + h);
}

// CTA of the weighted cut whose range holds the chunk of weight w.
__device__ __forceinline__ int cta_of_weight(const Cut& k, long long w) { return (int)div_nn(w * k.C, k.W); }

// CTA whose range holds chunk g of segment (s, h).
__device__ __forceinline__ int cta_of(const Cut& k, long long g, int s, int h) {
    if (!k.W) return (int)(((g + 1) * (long long)k.C - 1) / k.N);
    return cta_of_weight(k, cut_weight(k, g, s, h));
}

// Whether the segment (s, h), whose first chunk Pseg belongs to CTA c_first, starts that
// CTA's range (weighted: the chunk before it, a segment end, weighs u + e less).
__device__ __forceinline__ bool starts_range(const Cut& k, long long Pseg, int s, int h, int c_first) {
    if (!k.W) return Pseg == (k.N * c_first) / k.C;
    if (Pseg == 0) return true;
    return cta_of_weight(k, cut_weight(k, Pseg, s, h) - k.u - k.e) < c_first;
}

// First chunk of range c < C of the weighted cut.
__device__ __forceinline__ long long range_begin_weighted(const Cut& k, int c, int S, int Hkv) {
    const long long T = div_nn((long long)c * k.W + k.C - 1, k.C);   // the range's least weight
    // the last sequence whose first chunk weighs at most T
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)k.u * k.P[mid] + (long long)k.e * k.E[mid] <= T) lo = mid;
        else hi = mid - 1;
    }
    const int n = (k.P[lo + 1] - k.P[lo]) / Hkv;
    if (n == 0) return k.P[lo];
    const long long span = (long long)k.u * n + k.e;   // one segment of the sequence
    const long long off = T - ((long long)k.u * k.P[lo] + (long long)k.e * k.E[lo]);
    const long long h = div_nn(off, span);
    if (h >= Hkv) return k.P[lo + 1];
    const long long kk = div_nn(off - h * span + k.u - 1, k.u);
    if (kk >= n) return k.P[lo] + (h + 1) * n;
    return k.P[lo] + h * n + kk;
}

// First chunk of range c (N for c == C).
__device__ __forceinline__ long long range_begin(const Cut& k, int c, int S, int Hkv) {
    if (!k.W) return (k.N * c) / k.C;
    if (c >= k.C) return k.N;
    return range_begin_weighted(k, c, S, Hkv);
}

// Largest s in [0, S) with P[s] <= g (skips empty sequences because P repeats for them).
__device__ __forceinline__ int seq_of(const int32_t* P, int S, long long g) {
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)P[mid] <= g) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

struct SegPos {
    int s, h, k, n, L;  // sequence, kv head, chunk within the segment, chunks per segment, length
};

__device__ __forceinline__ SegPos locate(const int32_t* P, const int32_t* Lc, int S, int Hkv, long long g) {
    SegPos p;
    p.s = seq_of(P, S, g);
    p.n = (P[p.s + 1] - P[p.s]) / Hkv;
    const int r = (int)(g - P[p.s]);
    p.h = r / p.n;
    p.k = r - p.h * p.n;
    p.L = Lc[p.s];
    return p;
}

__device__ __forceinline__ void advance(SegPos& p, const int32_t* P, const int32_t* Lc, int S, int Hkv) {
    if (++p.k < p.n) return;
    p.k = 0;
    if (++p.h < Hkv) return;
    p.h = 0;
    do {
        ++p.s;
    } while (p.s < S && P[p.s + 1] == P[p.s]);
    if (p.s >= S) {   // past the last chunk: nothing left to read
        p.n = 0;
        p.L = 0;
        return;
    }
    p.n = (P[p.s + 1] - P[p.s]) / Hkv;
    p.L = Lc[p.s];
}

// Query span and q / out offsets, fixed at compile time for one query token per sequence.
template <bool kMulti>
__device__ __forceinline__ QSpan span_of(const DecodeArgs& a, int s, int L) {
    if constexpr (kMulti) return q_span(a, s, L);
    else return QSpan{s, 1};
}

template <bool kMulti>
__device__ __forceinline__ size_t out_offset(const DecodeArgs& a, const QSpan& q, int h, int G, int r) {
    if constexpr (kMulti) return q_offset(a, q, h, G, r);
    else return ((size_t)q.row0 * a.num_q_heads + (size_t)h * G + r) * kHeadDim;
}

// What the producer needs to issue one chunk's copies.
struct ChunkDesc {
    int s, h, t0, nblk, load_q;
    int q0, qn;   // the segment's query rows (first row, tokens), read when load_q
    int ids[4];   // physical blocks of the chunk (-1: none or outside the pool)
    int newblk;   // physical block of token L - 1 when this chunk holds it (-2: a bad id), else -1
};

template <bool kMulti>
__device__ __forceinline__ ChunkDesc describe(const DecodeArgs& a, const int32_t* P, const int32_t* Lc, int S,
                                              int Hkv, long long b_c, long long b_e, long long g) {
    ChunkDesc d;
    d.s = 0;
    d.h = 0;
    d.t0 = 0;
    d.nblk = 0;
    d.load_q = 0;
    d.ids[0] = d.ids[1] = d.ids[2] = d.ids[3] = -1;
    d.newblk = -1;
    d.q0 = 0;
    d.qn = 0;
    if (g >= b_e) return d;
    const SegPos p = locate(P, Lc, S, Hkv, g);
    const int B = a.block_size;
    d.s = p.s;
    d.h = p.h;
    d.t0 = p.k * kStageTokens;
    const int t1 = min(d.t0 + kStageTokens, p.L);
    const int first = d.t0 / B;
    d.nblk = (t1 - 1) / B - first + 1;   // <= 64 / 16
    d.load_q = (p.k == 0) || (g == b_c);
    if (d.load_q) {
        const QSpan q = span_of<kMulti>(a, p.s, p.L);
        d.q0 = q.row0;
        d.qn = q.n;
    }
    const int32_t* row = a.block_tables + (size_t)p.s * a.max_blocks_per_seq + first;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if (e < d.nblk) {
            const int id = row[e];
            if (id >= 0 && id < a.num_blocks) {
                d.ids[e] = id;
            } else {
                flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
            }
        }
    }
    if (t1 == p.L) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e == d.nblk - 1) d.newblk = d.ids[e] >= 0 ? d.ids[e] : -2;
    }
    return d;
}

// 64-token chunks of each kv head of sequence s: all of its L cached tokens, unless no query
// token of it is new (several-token mode), then none.
template <bool kMulti>
__device__ __forceinline__ int seq_chunks(const DecodeArgs& a, int s, int L) {
    if (kMulti && span_of<kMulti>(a, s, L).n == 0) return 0;
    return (L + kStageTokens - 1) / kStageTokens;
}

// Zero output rows of the empty sequences this CTA is responsible for (s = c, c + grid, ...).
// (Several query tokens per sequence: a sequence without chunks has no new token, so no row.)
template <bool kMulti>
__device__ __forceinline__ void zero_empty_rows(const DecodeArgs& a, const int32_t* P, int c, int t, int nthreads) {
    if (kMulti) return;
    const int Hq = a.num_q_heads;
    for (int s = c; s < a.num_seqs; s += (int)gridDim.x) {
        if (P[s + 1] == P[s]) {
            uint16_t* out = static_cast<uint16_t*>(a.out) + (size_t)s * Hq * kHeadDim;
            for (int e = t; e < Hq * kHeadDim; e += nthreads) out[e] = 0;
        }
    }
}

// Merge every piece (m, l, o) of the cut segment (s, h) -- chunks [Pseg, Pseg + n) of the list,
// cut by the CTA ranges -- into its normalised output rows.  Threads t = 0..nthreads-1 share the
// G x 16 (row, 8-column) items; one online pass over the pieces, a batch of loads in flight.
template <typename T, bool kMulti>
__device__ __forceinline__ void merge_pieces(const DecodeArgs& a, const QSpan& qsp, int s, int h, long long Pseg,
                                             int n, const Cut& cut, int t, int nthreads) {
    const int G = a.num_q_heads / a.num_kv_heads;
    const int rows = qsp.n * G;
    const int c_first = cta_of(cut, Pseg, s, h), c_last = cta_of(cut, Pseg + n - 1, s, h);
    // piece slot: 0 = the piece holding its CTA's first chunk; only the first CTA's piece can
    // start later than that
    const int first_slot = starts_range(cut, Pseg, s, h, c_first) ? 0 : 1;
    for (int e = t; e < rows * 16; e += nthreads) {
        const int row = e >> 4, d0 = (e & 15) * 8;
        // one online pass over the pieces, a few at a time, every load of a batch in flight
        float M = -INFINITY, den = 0.f;
        float num[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int cc0 = c_first; cc0 <= c_last; cc0 += kMergeBatch) {
            float2 ml[kMergeBatch];
            float4 x0[kMergeBatch], x1[kMergeBatch];
#pragma unroll
            for (int k = 0; k < kMergeBatch; ++k) {
                const int cc = cc0 + k;
                if (cc <= c_last) {
                    const size_t pc = (size_t)cc * 2 + (cc == c_first ? first_slot : 0);
                    const size_t row_idx = pc * kPieceRows + row;
                    ml[k] = ld_cg2(&a.part_ml[row_idx]);
                    x0[k] = ld_cg4(a.part_o + row_idx * kHeadDim + d0);
                    x1[k] = ld_cg4(a.part_o + row_idx * kHeadDim + d0 + 4);
                } else {
                    ml[k] = make_float2(-INFINITY, 0.f);
                    x0[k] = x1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            float bm = M;
#pragma unroll
            for (int k = 0; k < kMergeBatch; ++k) bm = fmaxf(bm, ml[k].x);
            // nothing seen yet (M = -inf): the running sums are 0 and stay so
            const float rescale = (kMulti && M == -INFINITY) ? 0.f : exp2f(M - bm);
            den *= rescale;
#pragma unroll
            for (int q = 0; q < 8; ++q) num[q] *= rescale;
#pragma unroll
            for (int k = 0; k < kMergeBatch; ++k) {
                // absent pieces, and rows a piece saw no token of (causal limit): weight 0
                const float f = (kMulti && ml[k].x == -INFINITY) ? 0.f : exp2f(ml[k].x - bm);
                den = fmaf(f, ml[k].y, den);
                num[0] = fmaf(f, x0[k].x, num[0]);
                num[1] = fmaf(f, x0[k].y, num[1]);
                num[2] = fmaf(f, x0[k].z, num[2]);
                num[3] = fmaf(f, x0[k].w, num[3]);
                num[4] = fmaf(f, x1[k].x, num[4]);
                num[5] = fmaf(f, x1[k].y, num[5]);
                num[6] = fmaf(f, x1[k].z, num[6]);
                num[7] = fmaf(f, x1[k].w, num[7]);
            }
            M = bm;
        }
        const float inv = 1.f / den;
        uint4 packed;
        packed.x = Elem<T>::pack2(num[0] * inv, num[1] * inv);
        packed.y = Elem<T>::pack2(num[2] * inv, num[3] * inv);
        packed.z = Elem<T>::pack2(num[4] * inv, num[5] * inv);
        packed.w = Elem<T>::pack2(num[6] * inv, num[7] * inv);
        *reinterpret_cast<uint4*>(static_cast<T*>(a.out) + out_offset<kMulti>(a, qsp, h, G, row) + d0) = packed;
    }
}

// Finish one segment piece at its last chunk in this CTA's range: merge the four consumer warps
// through the stage buffer they have just consumed (`scratch`, 32 KB), then write the normalised
// output (whole segment) or this CTA's partial (m, l, o).  A cut piece is then either handed to
// the epilogue warp (`handoff`: every consumer thread arrives on `pdone` after its stores) or
// finished here: count the arrival and, as the last CTA of the segment to arrive, merge all
// pieces.  Returns true if this call merged a cut segment.
template <typename T, int kNT, bool kMulti, bool kManyEnds>
__device__ __forceinline__ bool flush_segment(const DecodeArgs& a, unsigned char* scratch, const SegPos& pos,
                                              const int32_t* P, long long b_c, long long b_e,
                                              int c, const float (&o)[kNT][8][4], const float (&m_run)[kNT][2],
                                              const float (&l_run)[kNT][2], bool dead, volatile int* last_flag,
                                              bool handoff, uint64_t* pdone, const QSpan& qsp) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int Hkv = a.num_kv_heads, G = a.num_q_heads / Hkv;
    const int rows = qsp.n * G;   // query rows of the segment
    const long long Pseg = (long long)P[pos.s] + (long long)pos.h * pos.n;
    const bool whole = (Pseg >= b_c) && (Pseg + pos.n <= b_e);
    // row sums: each lane holds a partial over its own tokens; the 8 lanes of a row share tig
    float lr[kNT][2];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float v = l_run[nt][j];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            lr[nt][j] = v;
        }
    float* red_o = reinterpret_cast<float*>(scratch);                             // [4][8][kRedStride]
    float2* red_ml = reinterpret_cast<float2*>(red_o + kConsumerWarps * 8 * kRedStride);  // [4][8]
    const size_t piece = (size_t)c * 2 + ((Pseg <= b_c) ? 0 : 1);
    consumers_sync();   // every warp is past its reads of the stage
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        const int rg = nt * 8;   // query rows rg + 0..7 of the segment
        if (rg >= rows) break;
        // O^T fragment: o[nt][mt][j] = O[row tig*2 + j][dim mt*16 + gid], o[nt][mt][2 + j] the
        // same row at dim + 8; only the group's real query rows are written
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int row = tig * 2 + j;
            if (rg + row < rows) {
                float* dst = &red_o[(warp * 8 + row) * kRedStride + gid];
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    dst[mt * 16] = o[nt][mt][j];
                    dst[mt * 16 + 8] = o[nt][mt][2 + j];
                }
                if (gid == 0) red_ml[warp * 8 + row] = make_float2(m_run[nt][j], lr[nt][j]);
            }
        }
        consumers_sync();
        const int r = tid >> 4;            // row within the group of 8
        const int d0 = (tid & 15) * 8;     // 8 columns per thread
        const int row = rg + r;
        if (row < rows && !dead) {
            float M = -INFINITY;
#pragma unroll
            for (int w2 = 0; w2 < kConsumerWarps; ++w2) M = fmaxf(M, red_ml[w2 * 8 + r].x);
            float num[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            float den = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kConsumerWarps; ++w2) {
                const float2 ml = red_ml[w2 * 8 + r];
                // a warp without a valid token for the row: weight 0 (also when no warp has one,
                // which a cut piece can meet under a causal limit; its den stays 0)
                const float f = (kMulti && ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
                den = fmaf(f, ml.y, den);
                const float4 x0 = *reinterpret_cast<const float4*>(&red_o[(w2 * 8 + r) * kRedStride + d0]);
                const float4 x1 = *reinterpret_cast<const float4*>(&red_o[(w2 * 8 + r) * kRedStride + d0 + 4]);
                num[0] = fmaf(f, x0.x, num[0]);
                num[1] = fmaf(f, x0.y, num[1]);
                num[2] = fmaf(f, x0.z, num[2]);
                num[3] = fmaf(f, x0.w, num[3]);
                num[4] = fmaf(f, x1.x, num[4]);
                num[5] = fmaf(f, x1.y, num[5]);
                num[6] = fmaf(f, x1.z, num[6]);
                num[7] = fmaf(f, x1.w, num[7]);
            }
            if (whole) {
                const float inv = 1.f / den;
                uint4 packed;
                packed.x = Elem<T>::pack2(num[0] * inv, num[1] * inv);
                packed.y = Elem<T>::pack2(num[2] * inv, num[3] * inv);
                packed.z = Elem<T>::pack2(num[4] * inv, num[5] * inv);
                packed.w = Elem<T>::pack2(num[6] * inv, num[7] * inv);
                *reinterpret_cast<uint4*>(static_cast<T*>(a.out) + out_offset<kMulti>(a, qsp, pos.h, G, row) + d0) =
                    packed;
            } else {
                float* dst = a.part_o + (piece * kPieceRows + row) * kHeadDim + d0;
                *reinterpret_cast<float4*>(dst) = make_float4(num[0], num[1], num[2], num[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(num[4], num[5], num[6], num[7]);
                if ((tid & 15) == 0) a.part_ml[piece * kPieceRows + row] = make_float2(M, den);
            }
        }
        // The scratch is rewritten by the next column tile; a cut piece finished here also needs
        // every thread's partial stores ahead of thread 0's release.  Otherwise the stage goes
        // back to the producer only once every thread has arrived on its empty barrier.
        if (nt + 1 < kNT || (!whole && !handoff)) consumers_sync();
    }
    if (!whole && handoff) {
        mbar_arrive(pdone);   // release: this thread's partial stores precede the epilogue's arrival
        fence_proxy_async_smem();
        return false;
    }
    if (!whole) {
        // ---- pieces of a cut segment: the last CTA to arrive merges them ----
        // (the barrier that closed the loop above orders every thread's partial stores before
        // thread 0's release)
        const int sigma = pos.s * Hkv + pos.h;
        const Cut cut = make_cut<kManyEnds>(a, P, a.num_seqs);
        const int c_first = cta_of(cut, Pseg, pos.s, pos.h), c_last = cta_of(cut, Pseg + pos.n - 1, pos.s, pos.h);
        if (tid == 0) {
            *last_flag = 0;
            if (!dead) {
                const int prev = atom_add_acq_rel_gpu(&a.seg_counters[sigma], 1);
                *last_flag = (prev == c_last - c_first) ? 1 : 0;
            }
        }
        consumers_sync();
        const bool last = *last_flag != 0 && !dead;
        if (last) {
            merge_pieces<T, kMulti>(a, qsp, pos.s, pos.h, Pseg, pos.n, cut, tid, kConsumerThreads);
            if (tid == 0) a.seg_counters[sigma] = 0;   // ready for the next call
        }
        fence_proxy_async_smem();   // generic writes to the stage precede its next TMA fill
        return last;
    }
    fence_proxy_async_smem();
    return false;
}

// Exclusive prefix sums over the sequences, by the whole CTA: Lc[s] = the clamped length,
// P[s] = Hkv * (chunks of the sequences before s) and, with kSeqs, E[s] = Hkv * (sequences
// with chunks before s), both counted in one pass (chunks in the low 40 bits of a 64-bit
// count, sequences above).  P[S] (and E[S]) hold the totals.
template <bool kMulti, bool kSeqs>
__device__ __forceinline__ void chunk_prefix(const DecodeArgs& a, int S, int cap, int32_t* P, int32_t* Lc,
                                             int32_t* E, long long* bounds = nullptr) {
    using Acc = typename std::conditional<kSeqs, long long, int>::type;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hkv = a.num_kv_heads;
    auto count = [](int n) -> Acc {
        if constexpr (kSeqs) return (Acc)n + (n > 0 ? (1ll << 40) : 0ll);
        else return n;
    };
    const int per = (S + kThreads - 1) / kThreads;
    const int lo = min(S, tid * per), hi = min(S, lo + per);
    Acc local = 0;
    for (int s = lo; s < hi; ++s) {
        int L = a.context_lens[s];
        if (L < 0 || L > cap) {
            flag_status(a.status, PA_DEV_BAD_CONTEXT);
            L = L < 0 ? 0 : cap;
        }
        Lc[s] = L;
        if constexpr (kMulti) {
            const int n = a.q_start[s + 1] - a.q_start[s];
            const int r0 = a.q_start[s];
            if (n < 0 || n > L || n > a.max_q || r0 < 0 || r0 + n > a.q_rows) flag_status(a.status, PA_DEV_BAD_CONTEXT);
        }
        local += count(seq_chunks<kMulti>(a, s, L));
    }
    // exclusive scan of `local` over the CTA
    Acc incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const Acc v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    __shared__ Acc warp_tot[kThreads / 32];
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    Acc before = 0;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    Acc run = before + incl - local;
    auto put = [&](int s, Acc v) {
        if constexpr (kSeqs) {
            P[s] = (int32_t)(v & ((1ll << 40) - 1)) * Hkv;
            E[s] = (int32_t)(v >> 40) * Hkv;
        } else {
            P[s] = v * Hkv;
        }
    };
    Acc tot = 0;
    for (int w = 0; w < kThreads / 32; ++w) tot += warp_tot[w];
    // Weighted cut: the first chunks of this CTA's range and of the next (bounds[0], bounds[1];
    // the latter only when the next range exists), each written by the one thread whose
    // sequence holds the boundary weight (see Cut).  Nothing is written when the cut falls back
    // to the plain one (make_cut then gives W == 0 as well).
    long long W = 0, T[2] = {-1, -1};
    int C = 0;
    const int c = blockIdx.x;
    if constexpr (kSeqs) {
        const long long N = (tot & ((1ll << 40) - 1)) * Hkv, nseg = (tot >> 40) * Hkv;
        C = N > 0 ? (int)min((long long)gridDim.x, N) : 0;
        W = (long long)a.cut_unit * N + (long long)a.cut_seg * nseg;
        if (C == 0 || c >= C || W < (long long)(a.cut_unit + a.cut_seg) * C) W = 0;
        if (W)
            for (int j = 0; j < 2; ++j)
                if (c + j < C) T[j] = div_nn((long long)(c + j) * W + C - 1, C);   // the range's least weight
    }
    for (int s = lo; s < hi; ++s) {
        put(s, run);
        const int n = seq_chunks<kMulti>(a, s, Lc[s]);
        if constexpr (kSeqs) {
            if (W && n > 0) {
                const long long p0 = (run & ((1ll << 40) - 1)) * Hkv, e0 = (run >> 40) * Hkv;
                const long long w0 = (long long)a.cut_unit * p0 + (long long)a.cut_seg * e0;
                const long long span = (long long)a.cut_unit * n + a.cut_seg;   // one segment
                for (int j = 0; j < 2; ++j) {
                    const long long off = T[j] - w0;
                    if (T[j] < 0 || off < 0 || off >= span * Hkv) continue;
                    const long long h = div_nn(off, span);
                    const long long kk = div_nn(off - h * span + a.cut_unit - 1, a.cut_unit);
                    bounds[j] = kk >= n ? p0 + (h + 1) * n : p0 + h * n + kk;
                }
            }
        }
        run += count(n);
    }
    if (tid == kThreads - 1) put(S, tot);
}

// The weighted cut's prefix sums (only the kernel for many segment ends has them).
template <bool kMulti>
__device__ __forceinline__ void chunk_prefix_weighted(const DecodeArgs& a, int S, int cap, int32_t* P, int32_t* Lc,
                                                   int32_t* E, long long* bounds) {
    chunk_prefix<kMulti, true>(a, S, cap, P, Lc, E, bounds);
}

template <typename T, bool kG16, int kStages, bool kMulti, bool kManyEnds>
__global__ void __launch_bounds__(kThreads, (kStages > 3) ? 1 : 2)
    decode_persist_kernel(const DecodeArgs a, const __grid_constant__ MapsOf<kManyEnds> maps, const int R_log2) {
    using Lay = PLayout<kG16, kStages>;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;
    unsigned char* base_ptr = smem_raw + (ring - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(base_ptr + Lay::kBars);
    uint64_t* empty = full + kStages;
    uint64_t* qbar = empty + kStages;   // q rows of the first kStages chunks (fetched after the dependency wait)
    uint64_t* pdone = qbar + 1;         // the consumers have published the piece the epilogue warp finishes
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + Lay::kFlags);
    volatile int* issued_count = abort_flag + 1;
    volatile int* last_flag = abort_flag + 2;
    volatile int* epi_merges = abort_flag + 3;
    volatile int* new_phys = reinterpret_cast<volatile int*>(base_ptr + Lay::kNewPhys);
    volatile int* stage_q0 = new_phys + 2 * kStages;   // first q row of the segment a stage starts
    volatile int* stage_qn = new_phys + 3 * kStages;   // and its query tokens
    // One query token: s * Hkv + h of the new K/V row a deferred stage holds, or -1 (the slots of
    // stage_q0, which only the several-token mode uses).
    volatile int* stage_new = stage_q0;
    int32_t* P = reinterpret_cast<int32_t*>(base_ptr + Lay::kPrefix);   // [S + 1]
    const int S = a.num_seqs;
    int32_t* Lc = P + S + 1;                                              // [S], clamped lengths
    int32_t* E = Lc + S;   // [S + 1] non-empty segments before each sequence (weighted cut only)
    const bool weighted_layout = kManyEnds && a.cut_seg > 0;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads, G = Hq / Hkv, B = a.block_size;
    const int cap = a.max_blocks_per_seq * B;
    // Many segment ends per CTA, one query token per sequence and a group of at most kQRows - 2
    // heads: the producer copies a segment's new K and V rows into the last two q rows of the
    // stage holding its last chunk, so that the consumer finds them in shared memory rather than
    // waiting on a global load at every segment end.  (Kernels for few segment ends per CTA keep
    // the global load: there the extra producer work measured slower on a chain of launches.)
    const bool new_in_q = kManyEnds && !kMulti && a.k_new != nullptr && G <= Lay::kQRows - 2;
    constexpr uint32_t kNewRowK = (uint32_t)(Lay::kQRows - 2) * kHeadDim * 2u;   // offset in the q rows

    if (tid == 0) {
        trace(a.timeline, c, kTrEntry);
        prefetch_map(&maps.k);
        prefetch_map(&maps.v);
        if constexpr (kManyEnds) {
            prefetch_map(&maps.k2);
            prefetch_map(&maps.v2);
            prefetch_map(&maps.k4);
            prefetch_map(&maps.v4);
        }
#pragma unroll
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerThreads);
        }
        mbar_init(qbar, 1);
        mbar_init(pdone, kConsumerThreads);
        *abort_flag = 0;
        *issued_count = 0;
        *last_flag = 0;
        *epi_merges = 0;
        fence_mbar_init();
    }
    // Without the early contract every input may come from the preceding kernel: wait now.
    // With it, lengths, tables and the cached rows are read first and the wait comes later.
    if (!a.early) {
        grid_dependency_wait();
        if (tid == 0) trace(a.timeline, c, kTrDeps);
    }

    // ---- prefix sums of chunk counts: P[s] = Hkv * sum_{s' < s} ceil(L_s' / 64) (and E) ----
    __shared__ long long cut_bounds[2];   // weighted cut: this range's first chunk and the next's
    if (weighted_layout) chunk_prefix_weighted<kMulti>(a, S, cap, P, Lc, E, cut_bounds);
    else chunk_prefix<kMulti, false>(a, S, cap, P, Lc, E);
    __syncthreads();
    if (tid == 0) trace(a.timeline, c, kTrScan);

    const long long N = P[S];
    // C <= N CTAs take part, so that every one of them owns at least one chunk
    const int C = N > 0 ? (int)min((long long)gridDim.x, N) : 0;
    if (c >= C) {
        if (a.early) grid_dependency_wait();
        grid_launch_dependents();
        zero_empty_rows<kMulti>(a, P, c, tid, kThreads);
        return;
    }
    long long b_c, b_e;
    {
        const Cut cut = make_cut<kManyEnds>(a, P, S);
        if (weighted_layout && cut.W) {
            // found with the prefix sums (the cut range_begin would search for)
            b_c = cut_bounds[0];
            b_e = c + 1 < C ? cut_bounds[1] : N;
        } else {
            b_c = range_begin(cut, c, S, Hkv);
            b_e = range_begin(cut, c + 1, S, Hkv);
        }
    }
    if (!a.early) grid_launch_dependents();

    if (warp == kProducerWarp) {
        // ================= producer warp =================
        // Lane j describes chunk gbase + j (segment position and physical block ids); the next
        // group's descriptors are loaded while this group's copies are issued, so the ring is
        // refilled as soon as a stage frees up.
        ChunkDesc cur = describe<kMulti>(a, P, Lc, S, Hkv, b_c, b_e, b_c + lane);
        unsigned long long wait_empty_ns = 0;
        if (a.timeline && lane == 0 && cur.ids[0] != INT_MIN) trace(a.timeline, c, kTrIds);
        volatile int* qdef = new_phys + kStages;   // [kStages]: q rows the first stages still need
        const bool append = a.k_new != nullptr;
        bool deps_done = false;
        // After the preceding kernel has finished (early mode), fetch the q rows of the first
        // stages onto their own barrier: they may be that kernel's output.
        auto dependency_point = [&](int issued) {
            if (a.early) {
                grid_dependency_wait();
                grid_launch_dependents();
            }
            if (lane == 0) {
                const int n = min(issued, kStages);
                const uint32_t group_bytes = (uint32_t)G * kHeadDim * 2u;
                uint32_t bytes = 0;
                for (int e = 0; e < n; ++e) {
                    if (qdef[e] >= 0) bytes += (uint32_t)(kMulti ? stage_qn[e] : 1) * group_bytes;
                    if (new_in_q && stage_new[e] >= 0) bytes += 4u * kHeadDim;
                }
                mbar_arrive_expect_tx(qbar, bytes);
                for (int e = 0; e < n; ++e) {
                    const int sh = new_in_q ? stage_new[e] : -1;
                    if (sh >= 0) {
                        const uint32_t nd = ring + (uint32_t)e * Lay::kStageBytes + kKVBytes + kNewRowK;
                        bulk_g2s(nd, static_cast<const T*>(a.k_new) + (size_t)sh * kHeadDim, 2u * kHeadDim, qbar);
                        bulk_g2s(nd + 2u * kHeadDim, static_cast<const T*>(a.v_new) + (size_t)sh * kHeadDim,
                                 2u * kHeadDim, qbar);
                    }
                }
                for (int e = 0; e < n; ++e) {
                    const int sh = qdef[e];
                    if (sh >= 0) {
                        // query token r of the segment: its group's G rows, contiguous in q
                        // the segment's query rows: its span (several tokens) or row s (one token;
                        // the stage metadata is written in several-token mode only)
                        const int nq = kMulti ? stage_qn[e] : 1;
                        const int row0 = kMulti ? stage_q0[e] : sh / Hkv;
                        for (int r = 0; r < nq; ++r) {
                            const T* qsrc = static_cast<const T*>(a.q) +
                                            ((size_t)(row0 + r) * Hq + (sh % Hkv) * G) * kHeadDim;
                            bulk_g2s(ring + (uint32_t)e * Lay::kStageBytes + kKVBytes + (uint32_t)r * group_bytes, qsrc,
                                     group_bytes, qbar);
                        }
                    }
                }
            }
            __syncwarp();
        };
        int i = 0;
        bool ok = true;
        for (long long gbase = b_c; gbase < b_e && ok; gbase += 32) {
            const ChunkDesc nxt = describe<kMulti>(a, P, Lc, S, Hkv, b_c, b_e, gbase + 32 + lane);
            const int cnt = (int)min(32LL, b_e - gbase);
            for (int j = 0; j < cnt; ++j, ++i) {
                const int st = i % kStages;
                if (i == kStages && !deps_done) {
                    dependency_point(i);
                    deps_done = true;
                }
                if (i >= kStages) {
                    bool w = true;
                    if (lane == 0) {
                        const unsigned long long t0 = a.timeline ? global_timer_ns() : 0ull;
                        w = mbar_wait_bounded(&empty[st], (uint32_t)((i / kStages) - 1) & 1u);
                        if (a.timeline) wait_empty_ns += global_timer_ns() - t0;
                    }
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
                const int s_j = __shfl_sync(0xffffffffu, cur.s, j);
                const int h_j = __shfl_sync(0xffffffffu, cur.h, j);
                const int t0_j = __shfl_sync(0xffffffffu, cur.t0, j);
                const int nblk_j = __shfl_sync(0xffffffffu, cur.nblk, j);
                const int loadq_j = __shfl_sync(0xffffffffu, cur.load_q, j);
                const int newblk_j = __shfl_sync(0xffffffffu, cur.newblk, j);
                const int q0_j = kMulti ? __shfl_sync(0xffffffffu, cur.q0, j) : s_j;
                const int qn_j = kMulti ? __shfl_sync(0xffffffffu, cur.qn, j) : 1;
                int ids[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) ids[e] = __shfl_sync(0xffffffffu, cur.ids[e], j);
                if (lane == 0) {
                    if (*abort_flag) {
                        ok = false;
                    } else {
                        const int R = 1 << R_log2;
                        const uint32_t dst = ring + (uint32_t)st * Lay::kStageBytes;
                        const int within = (B > kStageTokens) ? (t0_j % B) : 0;
                        const bool defer_q = i < kStages;   // fetched at the dependency point
                        const uint32_t group_bytes = (uint32_t)G * kHeadDim * 2u;
                        if (defer_q) qdef[i] = loadq_j ? s_j * Hkv + h_j : -1;
                        new_phys[st] = append ? newblk_j : -1;
                        const bool new_row = new_in_q && newblk_j != -1;   // this chunk holds token L - 1
                        if (new_in_q && defer_q) stage_new[i] = new_row ? s_j * Hkv + h_j : -1;
                        if (kMulti) {
                            stage_q0[st] = q0_j;
                            stage_qn[st] = qn_j;
                        }
                        const int nq = kMulti ? qn_j : 1;
                        uint32_t bytes = (loadq_j && !defer_q) ? (uint32_t)nq * group_bytes : 0u;
                        if (new_row && !defer_q) bytes += 4u * kHeadDim;
                        // box height of block e: the lowest of R, R / 2, R / 4 rows that covers its
                        // valid rows (shift 0, 1 or 2); rows past them are never read
                        auto box_shift = [&](int e) {
                            if constexpr (!kManyEnds) return 0;
                            const int rows = min(kStageTokens, Lc[s_j] - t0_j) - e * R;   // valid rows
                            return rows <= (R >> 2) ? 2 : (rows <= (R >> 1) ? 1 : 0);
                        };
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (e < nblk_j && ids[e] >= 0) bytes += 4u * (uint32_t)(R >> box_shift(e)) * 128u;
                        if (i >= kStages) fence_proxy_async_smem();
                        mbar_arrive_expect_tx(&full[st], bytes);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (e < nblk_j && ids[e] >= 0) {
                                const int row = (ids[e] * Hkv + h_j) * B + within;
                                const uint32_t box = dst + (uint32_t)(e * 2 * R) * 128u;
                                const CUtensorMap* mk = &maps.k;
                                const CUtensorMap* mv = &maps.v;
                                if constexpr (kManyEnds) {
                                    const int sh = box_shift(e);
                                    if (sh) {
                                        mk = sh == 1 ? &maps.k2 : &maps.k4;
                                        mv = sh == 1 ? &maps.v2 : &maps.v4;
                                    }
                                }
                                tma_load_2d(box, mk, 0, row, &full[st]);
                                tma_load_2d(box + (uint32_t)R * 128u, mk, 64, row, &full[st]);
                                tma_load_2d(box + kKBytes, mv, 0, row, &full[st]);
                                tma_load_2d(box + kKBytes + (uint32_t)R * 128u, mv, 64, row, &full[st]);
                            }
                        }
                        if (i == 0) trace(a.timeline, c, kTrIssue);
                        if (loadq_j && !defer_q) {
                            for (int r = 0; r < nq; ++r) {
                                const T* qsrc =
                                    static_cast<const T*>(a.q) + ((size_t)(q0_j + r) * Hq + h_j * G) * kHeadDim;
                                bulk_g2s(dst + kKVBytes + (uint32_t)r * group_bytes, qsrc, group_bytes, &full[st]);
                            }
                        }
                        if (new_row && !defer_q) {
                            const size_t sh = (size_t)s_j * Hkv + h_j;
                            bulk_g2s(dst + kKVBytes + kNewRowK, static_cast<const T*>(a.k_new) + sh * kHeadDim,
                                     2u * kHeadDim, &full[st]);
                            bulk_g2s(dst + kKVBytes + kNewRowK + 2u * kHeadDim,
                                     static_cast<const T*>(a.v_new) + sh * kHeadDim, 2u * kHeadDim, &full[st]);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            cur = nxt;
        }
        if (!deps_done) dependency_point(i);
        if (lane == 0) {
            *issued_count = i;
            trace_put(a.timeline, c, kTrWaitEmpty, wait_empty_ns);
        }
    } else if (warp == kEpilogueWarp) {
        // ================= epilogue warp =================
        // The range's first segment, when it began in an earlier range and ends before this one
        // does: count this CTA's arrival and, if it is the last, merge the segment's pieces.
        const SegPos p0 = locate(P, Lc, S, Hkv, b_c);
        const long long Pseg = (long long)P[p0.s] + (long long)p0.h * p0.n;
        if (Pseg < b_c && Pseg + p0.n - 1 < b_e - 1) {
            if (a.early) grid_dependency_wait();   // counters and outputs are written after it
            bool ok = true;
            if (lane == 0) ok = mbar_wait_bounded(pdone, 0u);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    flag_status(a.status, PA_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
            } else if (*abort_flag == 0) {
                // acquired through pdone: the consumers' partial stores; the release publishes them
                const int sigma = p0.s * Hkv + p0.h;
                const Cut cut = make_cut<kManyEnds>(a, P, S);
                const int c_first = cta_of(cut, Pseg, p0.s, p0.h), c_last = cta_of(cut, Pseg + p0.n - 1, p0.s, p0.h);
                int last = 0;
                if (lane == 0) last = atom_add_acq_rel_gpu(&a.seg_counters[sigma], 1) == c_last - c_first;
                last = __shfl_sync(0xffffffffu, last, 0);
                __syncwarp();   // the lanes' merge reads come after lane 0's acquire
                if (last) {
                    merge_pieces<T, kMulti>(a, span_of<kMulti>(a, p0.s, p0.L), p0.s, p0.h, Pseg, p0.n, cut, lane,
                                            32);
                    if (lane == 0) {
                        a.seg_counters[sigma] = 0;   // ready for the next call
                        *epi_merges = 1;
                    }
                }
            }
        }
    } else {
        // ================= consumer warps =================
        constexpr int kNT = kG16 ? 2 : 1;   // 8-row column tiles of the GQA group
        const int gid = lane >> 2, tig = lane & 3;
        const int t_warp = warp * 16;
        // ldmatrix row addresses: K tile as the A operand (tokens x dims), V tile transposed as
        // the A operand (dims x tokens)
        const int tokA = t_warp + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int chA = lane >> 4;
        const int tokV = t_warp + (lane & 7) + ((lane >> 4) << 3);
        const int chV = (lane >> 3) & 1;
        float m_run[kNT][2], l_run[kNT][2];
        float o[kNT][8][4];
        uint32_t qb[8][kNT][2];   // Q^T as the B operand: [k-step][column tile][2 registers]
        int lim[kNT][2];          // newest position each of the lane's query rows attends to
        QSpan qsp{0, 0};          // the current segment's query tokens
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            m_run[nt][0] = m_run[nt][1] = -INFINITY;
            l_run[nt][0] = l_run[nt][1] = 0.f;
        }
        if (a.early) {
            grid_dependency_wait();   // q, the new rows and every output belong after this point
            grid_launch_dependents();
            if (tid == 0) trace(a.timeline, c, kTrDeps);
        }
        unsigned long long wait_full_ns = 0, flush_ns = 0, merges = 0, flushes = 0;
        zero_empty_rows<kMulti>(a, P, c, tid, kConsumerThreads);
        const bool append = a.k_new != nullptr;
        SegPos pos = locate(P, Lc, S, Hkv, b_c);
        // A warp that gave up on a wait (or sees that another did) is "dead": it keeps walking
        // the same chunk sequence, so that every consumer warp reaches the same barriers, but
        // waits for nothing and writes no result.
        bool dead = false;
        int i = 0;
        for (long long g = b_c; g < b_e; ++g, ++i) {
            const int st = i % kStages;
            dead = dead || __any_sync(0xffffffffu, *abort_flag != 0);
            const unsigned long long tw = (a.timeline && tid == 0) ? global_timer_ns() : 0ull;
            if (!dead && !__all_sync(0xffffffffu, mbar_wait_bounded(&full[st], (uint32_t)(i / kStages) & 1u))) {
                if (lane == 0) {
                    flag_status(a.status, PA_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
                dead = true;
            }
            __syncwarp();
            if (a.timeline && tid == 0) {
                const unsigned long long now = global_timer_ns();
                wait_full_ns += now - tw;
                if (i == 0) trace_put(a.timeline, c, kTrFirst, now);
                if (g == b_e - 1) trace_put(a.timeline, c, kTrLastLanded, now);
            }
            const uint32_t kbase = ring + (uint32_t)st * Lay::kStageBytes;
            const uint32_t vbase = kbase + kKBytes;
            const bool seg_begin = (pos.k == 0) || (g == b_c);
            const bool seg_end = (pos.k == pos.n - 1) || (g == b_e - 1);
            if (!dead && seg_begin && i < kStages) {
                // the first stages' q rows arrive on their own barrier
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(qbar, 0u))) {
                    if (lane == 0) {
                        flag_status(a.status, PA_DEV_TIMEOUT);
                        *abort_flag = 1;
                    }
                    dead = true;
                }
            }
            if (seg_begin) qsp = kMulti ? QSpan{stage_q0[st], stage_qn[st]} : QSpan{pos.s, 1};
            if (seg_begin && !dead) {
                // B fragments of Q^T: register 0 = Q[row][ks*16 + tig*2 + {0,1}], register 1 the
                // same at + 8, row = nt*8 + gid = token (row / G) x group member (row % G);
                // rows past the segment's are zero
                const int rows = qsp.n * G;
                const uint32_t* qs = reinterpret_cast<const uint32_t*>(base_ptr + (size_t)st * Lay::kStageBytes +
                                                                       kKVBytes);
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    const int row = nt * 8 + gid;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int wcol = (ks * 16 + tig * 2) >> 1;
                        qb[ks][nt][0] = (row < rows) ? qs[row * 64 + wcol] : 0u;
                        qb[ks][nt][1] = (row < rows) ? qs[row * 64 + wcol + 4] : 0u;
                    }
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int r = nt * 8 + tig * 2 + j;   // a column of S^T this lane holds
                        lim[nt][j] = (kMulti && r < rows) ? pos.L - qsp.n + r / G : -1;
                    }
                    m_run[nt][0] = m_run[nt][1] = -INFINITY;
                    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
                }
            }
            const int nvalid = min(kStageTokens, pos.L - pos.k * kStageTokens);

            if (t_warp < nvalid && !dead) {
                if (nvalid < t_warp + 16) {
                    uint4* vz = reinterpret_cast<uint4*>(base_ptr + (size_t)st * Lay::kStageBytes + kKBytes);
                    for (int idx = lane; idx < (t_warp + 16 - nvalid) * 16; idx += 32) {
                        const int t = nvalid + (idx >> 4);
                        const int cc = idx & 15;
                        vz[line_of(t, cc >> 3, R_log2) * 8 + (cc & 7)] = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (kMulti && append) {
                    // the segment's new tokens (positions L - n .. L - 1) in this warp's 16 rows:
                    // their K/V rows go into the staged tile and into their cache slots
                    const int c0 = pos.k * kStageTokens + t_warp;
                    const int p_lo = max(pos.L - qsp.n, c0), p_hi = min(pos.L, c0 + 16);
                    const int cc = lane & 15;
                    const bool isv = lane >= 16;
                    for (int p = p_lo; p < p_hi; ++p) {
                        const int i_new = p - (pos.L - qsp.n);
                        const size_t src_off = ((size_t)(qsp.row0 + i_new) * Hkv + pos.h) * kHeadDim + cc * 8;
                        const uint4 val = *reinterpret_cast<const uint4*>(
                            static_cast<const T*>(isv ? a.v_new : a.k_new) + src_off);
                        st_shared_v4(chunk_addr(isv ? vbase : kbase, p - pos.k * kStageTokens, cc, R_log2), val);
                        const int phys = a.block_tables[(size_t)pos.s * a.max_blocks_per_seq + p / B];
                        if (phys >= 0 && phys < a.num_blocks) {
                            const size_t row = ((size_t)phys * Hkv + pos.h) * B + (size_t)(p % B);
                            T* cache = const_cast<T*>(static_cast<const T*>(isv ? a.v_cache : a.k_cache));
                            *reinterpret_cast<uint4*>(cache + row * kHeadDim + cc * 8) = val;
                        }
                    }
                    if (p_lo < p_hi) {
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                }
                const int tn = nvalid - 1;   // the newest token, when this is the segment's last chunk
                if (!kMulti && append && pos.k == pos.n - 1 && (tn >> 4) == warp) {
                    // append: the new K/V row goes into the staged tile and into its cache slot
                    const int cc = lane & 15;
                    const bool isv = lane >= 16;
                    uint4 val;
                    if (new_in_q) {
                        // staged by the producer with the chunk (or, in the first stages, with q)
                        val = *reinterpret_cast<const uint4*>(base_ptr + (size_t)st * Lay::kStageBytes + kKVBytes +
                                                              kNewRowK + (isv ? 2u * kHeadDim : 0u) + cc * 16);
                    } else {
                        const size_t src_off = ((size_t)pos.s * Hkv + pos.h) * kHeadDim + cc * 8;
                        val = *reinterpret_cast<const uint4*>(static_cast<const T*>(isv ? a.v_new : a.k_new) + src_off);
                    }
                    st_shared_v4(chunk_addr(isv ? vbase : kbase, tn, cc, R_log2), val);
                    const int phys = new_phys[st];
                    if (phys >= 0) {
                        const size_t row = ((size_t)phys * Hkv + pos.h) * B + (size_t)((pos.L - 1) % B);
                        T* cache = const_cast<T*>(static_cast<const T*>(isv ? a.v_cache : a.k_cache));
                        *reinterpret_cast<uint4*>(cache + row * kHeadDim + cc * 8) = val;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                // S^T = K Q^T over the warp's 16 tokens: two accumulator chains (even / odd k-steps)
                float sc[kNT][4], sc2[kNT][4];
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[nt][e] = sc2[nt][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(chunk_addr(kbase, tokA, 2 * ks + chA, R_log2), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < kNT; ++nt) {
                        if (ks & 1) mma16816<T>(sc2[nt], a0, a1, a2, a3, qb[ks][nt][0], qb[ks][nt][1]);
                        else mma16816<T>(sc[nt], a0, a1, a2, a3, qb[ks][nt][0], qb[ks][nt][1]);
                    }
                }
                // online softmax per query row: lane holds rows tig*2 + j at tokens gid and gid + 8;
                // the 8 lanes of a row (same tig) reduce with xor 4, 8, 16
                // position of the lane's first token; one query token per sequence sees every valid
                // token of the chunk, several see up to their own positions (lim)
                const int tok0 = pos.k * kStageTokens + t_warp + gid;
                const bool in0 = t_warp + gid < nvalid, in1 = t_warp + gid + 8 < nvalid;
                // bf16 keeps 8 significant bits: P goes in as a high and a low bf16 part (two PV
                // products), so that rows attending to few tokens keep fp32-like weights
                constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
                // Exponent base per row: m_run, moved only when a score exceeds it by more than
                // kLazyLog2 (then to the exact running max, rescaling O and l).  Weights stay below
                // 2^kLazyLog2, and most chunks skip the cross-lane max and the rescale.
                float xs[kNT][4];
                bool move = false;
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const bool ok0 = kMulti ? tok0 <= lim[nt][j] : in0;
                        const bool ok1 = kMulti ? tok0 + 8 <= lim[nt][j] : in1;
                        xs[nt][j] = ok0 ? (sc[nt][j] + sc2[nt][j]) * a.scale_log2 : -INFINITY;
                        xs[nt][2 + j] = ok1 ? (sc[nt][2 + j] + sc2[nt][2 + j]) * a.scale_log2 : -INFINITY;
                        // (m_run = -inf: any visible token moves the base)
                        move = move || xs[nt][j] > m_run[nt][j] + kLazyLog2 ||
                               xs[nt][2 + j] > m_run[nt][j] + kLazyLog2;
                    }
                if (__any_sync(0xffffffffu, move)) {
                    float alpha[kNT][2];
#pragma unroll
                    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            // the 8 lanes of a row (same tig) reduce with xor 4, 8, 16
                            float mx = fmaxf(xs[nt][j], xs[nt][2 + j]);
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                            const float m_new = fmaxf(m_run[nt][j], mx);
                            alpha[nt][j] = (m_new == -INFINITY) ? 1.f : exp2f(m_run[nt][j] - m_new);
                            m_run[nt][j] = m_new;
                            l_run[nt][j] *= alpha[nt][j];
                        }
#pragma unroll
                    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            o[nt][mt][0] *= alpha[nt][0];
                            o[nt][mt][1] *= alpha[nt][1];
                            o[nt][mt][2] *= alpha[nt][0];
                            o[nt][mt][3] *= alpha[nt][1];
                        }
                }
                uint32_t pb[kNT][2], pl[kNT][2];
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    float pv[4];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float m_use = (m_run[nt][j] == -INFINITY) ? 0.f : m_run[nt][j];
                        pv[j] = exp2f(xs[nt][j] - m_use);
                        pv[2 + j] = exp2f(xs[nt][2 + j] - m_use);
                        l_run[nt][j] += pv[j] + pv[2 + j];
                    }
                    // P^T as the B operand: the C fragment (tokens x rows) transposed per 8x8 block
                    const uint32_t h0 = Elem<T>::pack2(pv[0], pv[1]), h1 = Elem<T>::pack2(pv[2], pv[3]);
                    pb[nt][0] = movmatrix_trans(h0);
                    pb[nt][1] = movmatrix_trans(h1);
                    if (kSplitP) {
                        const float2 r0 = Elem<T>::to_float2(h0), r1 = Elem<T>::to_float2(h1);
                        pl[nt][0] = movmatrix_trans(Elem<T>::pack2(pv[0] - r0.x, pv[1] - r0.y));
                        pl[nt][1] = movmatrix_trans(Elem<T>::pack2(pv[2] - r1.x, pv[3] - r1.y));
                    }
                }
                // O^T += V^T P^T, one 16-dim tile of V^T at a time
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(chunk_addr(vbase, tokV, 2 * mt + chV, R_log2), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < kNT; ++nt) {
                        mma16816<T>(o[nt][mt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                        if (kSplitP) mma16816<T>(o[nt][mt], a0, a1, a2, a3, pl[nt][0], pl[nt][1]);
                    }
                }
            }

            if (seg_end) {
                const unsigned long long tf = (a.timeline && tid == 0) ? global_timer_ns() : 0ull;
                const bool merged = flush_segment<T, kNT, kMulti, kManyEnds>(a, base_ptr + (size_t)st * Lay::kStageBytes, pos, P, b_c, b_e,
                                                     c, o, m_run, l_run, dead, last_flag, g != b_e - 1, pdone,
                                                     qsp);
                if (a.timeline && tid == 0) {
                    flush_ns += global_timer_ns() - tf;
                    merges += merged ? 1 : 0;
                    ++flushes;
                }
            }
            mbar_arrive(&empty[st]);   // this thread is done with the stage's buffers
            advance(pos, P, Lc, S, Hkv);
        }
        if (tid == 0 && a.timeline) {
            trace(a.timeline, c, kTrLoopEnd);
            trace_put(a.timeline, c, kTrWaitFull, wait_full_ns);
            trace_put(a.timeline, c, kTrFlush, flush_ns);
            trace_put(a.timeline, c, kTrMerges, merges);   // the epilogue warp's merge is added at exit
            trace_put(a.timeline, c, kTrFlushes, flushes);
        }
    }

    __syncthreads();
    if (tid == 0 && a.timeline) {
        trace(a.timeline, c, kTrExit);
        unsigned int smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        trace_put(a.timeline, c, kTrChunks, (unsigned long long)(b_e - b_c));
        trace_put(a.timeline, c, kTrSm, smid);
        a.timeline[(size_t)c * kTimelineSlots + kTrMerges] += (unsigned long long)*epi_merges;
    }
    if (*abort_flag && tid == 0) {
        // let every copy still in flight land before the CTA's shared memory is released
        const int n = *issued_count;
        for (int st = 0; st < kStages; ++st) {
            int last = -1;
            for (int i = st; i < n; i += kStages) last = i;
            if (last >= 0) (void)mbar_wait_bounded(&full[st], (uint32_t)(last / kStages) & 1u);
        }
    }
}

// ---- host side ----

bool encode_map(const void* base, unsigned long long rows, int box_rows, CUtensorMap* out) {
    return encode_pool_map(base, rows, box_rows, out);
}

template <typename T, bool kG16, int kStages, bool kMulti, bool kManyEnds = false>
cudaError_t launch_impl(const DecodeArgs& a, const MmaMapsTails& all, int R_log2, cudaStream_t stream) {
    MapsOf<kManyEnds> maps;
    if constexpr (kManyEnds) maps = all;
    else maps = MmaMaps{all.k, all.v};
    static std::atomic<unsigned long long> configured{0};
    auto kernel = decode_persist_kernel<T, kG16, kStages, kMulti, kManyEnds>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)PLayout<kG16, kStages>::total(kPersistMaxSeqs));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = PLayout<kG16, kStages>::total(a.num_seqs, a.cut_seg > 0);
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

template <bool kMulti>
cudaError_t dispatch(const DecodeArgs& a, const MmaMapsTails& maps, int R_log2, int dtype, bool g16, bool deep,
                     cudaStream_t stream) {
    if (dtype == PA_BF16) {
        if (g16) return deep ? launch_impl<__nv_bfloat16, true, 6, kMulti>(a, maps, R_log2, stream)
                             : launch_impl<__nv_bfloat16, true, 3, kMulti>(a, maps, R_log2, stream);
        if constexpr (!kMulti)
            if (!deep && a.cut_seg > 0) return launch_impl<__nv_bfloat16, false, 3, false, true>(a, maps, R_log2, stream);
        return deep ? launch_impl<__nv_bfloat16, false, 6, kMulti>(a, maps, R_log2, stream)
                    : launch_impl<__nv_bfloat16, false, 3, kMulti>(a, maps, R_log2, stream);
    }
    if (g16) return deep ? launch_impl<__half, true, 6, kMulti>(a, maps, R_log2, stream)
                         : launch_impl<__half, true, 3, kMulti>(a, maps, R_log2, stream);
    if constexpr (!kMulti)
        if (!deep && a.cut_seg > 0) return launch_impl<__half, false, 3, false, true>(a, maps, R_log2, stream);
    return deep ? launch_impl<__half, false, 6, kMulti>(a, maps, R_log2, stream)
                : launch_impl<__half, false, 3, kMulti>(a, maps, R_log2, stream);
}

}  // namespace

// Two CTAs per SM (the 3-stage ring) unless 9 to 16 query rows per segment and so many sequences
// that two CTAs' shared memory (their prefix arrays included) no longer fits one SM.
int persist_ctas_per_sm(int rows, int num_seqs) {
    if (rows <= 8) return 2;
    return 2 * (PLayout<true, 3>::total(num_seqs) + 1024) <= 228u * 1024u ? 2 : 1;
}

cudaError_t launch_decode_persist(const DecodeArgs& a, int dtype, cudaStream_t stream) {
    const int R = a.block_size < kStageTokens ? a.block_size : kStageTokens;
    int R_log2 = 0;
    while ((1 << R_log2) < R) ++R_log2;
    const unsigned long long rows = (unsigned long long)a.num_blocks * a.num_kv_heads * a.block_size;
    if (rows == 0 || rows > 0x7fffffffull) return cudaErrorInvalidValue;
    MmaMapsTails maps;
    if (!encode_map(a.k_cache, rows, R, &maps.k) || !encode_map(a.v_cache, rows, R, &maps.v))
        return cudaErrorInvalidValue;
    const bool g16 = a.max_q * (a.num_q_heads / a.num_kv_heads) > 8;   // query rows per segment
    // as many CTAs as SMs (or fewer): one CTA per SM with the deep ring
    const bool deep = a.num_ctas <= sm_count_current();
    DecodeArgs b = a;
    // Many segments per CTA (short contexts, many kv heads): a segment's end then costs about
    // half a chunk's share of the stream, and the cut weighs it so (measured best of 1:1, 2:1,
    // 3:2, 3:4, 1:2, 1:3 on 256 sequences x 32 kv heads; the third prefix array fits beside two
    // CTAs per SM up to 512 sequences).
    // Only the one-token kernel with two CTAs per SM and at most 8 query rows is built with it.
    const bool many_ends = a.num_seqs <= 512 && (long long)a.num_seqs * a.num_kv_heads >= 4ll * a.num_ctas;
    b.cut_unit = 2;
    b.cut_seg = (many_ends && !g16 && !deep && !a.q_start) ? 1 : 0;
    if (b.cut_seg > 0 &&
        (!encode_map(a.k_cache, rows, R / 2, &maps.k2) || !encode_map(a.v_cache, rows, R / 2, &maps.v2) ||
         !encode_map(a.k_cache, rows, R / 4, &maps.k4) || !encode_map(a.v_cache, rows, R / 4, &maps.v4)))
        return cudaErrorInvalidValue;
    if (a.q_start) return dispatch<true>(b, maps, R_log2, dtype, g16, deep, stream);
    return dispatch<false>(b, maps, R_log2, dtype, g16, deep, stream);
}

}  // namespace pa
