// Paged decode attention, split pass, tensor-core path.
//
// Same computation as the CUDA-core split pass ("显存虚拟化革命：PagedAttention 内存池管理与
// 显存碎片终结", §五.1: per sequence and head, walk the logical blocks through block_tables,
// q.k per token, running-max softmax, weight V, normalise at the end), with the two small
// products of every staged tile on the tensor cores:
//   S (16 x 16 per warp)  = Q_group (16 rows: the G query heads of the kv head, zero padded)
//                           x K_tile^T                          mma.sync m16n8k16, fp32 accum
//   O (16 x 128 per warp) += P (S after the online softmax, rounded to the input type)
//                           x V_tile                            mma.sync m16n8k16, fp32 accum
// G <= 16 query heads share each tile, so one tile read from HBM serves the whole group.
//
// Staging: 64-token stages in a 3-deep shared-memory ring.  Each (block, kv-head) tile is
// fetched by 2-D TMA tensor loads (one per 64-column half of the 128-wide rows) with the
// 128-byte swizzle, so the ldmatrix reads of 8 consecutive tokens at one column touch 8
// distinct bank groups.  One thread issues the loads after checking the block id against
// the pool; an mbarrier with a transaction count tracks each stage.
//
// Work split: warp w of the CTA owns tokens [16w, 16w+16) of every stage and keeps its own
// running max / sum / output; the four warps are merged once at the end of the split.
#include "pa_internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

namespace pa {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;          // + one TMA producer warp
constexpr int kStages = 3;
constexpr int kStageKBytes = kStageTokens * kHeadDim * 2;   // 16 KB of K per stage (V the same)
constexpr int kStageBytes = 2 * kStageKBytes;
constexpr size_t kRingBytes = (size_t)kStages * kStageBytes;
constexpr size_t kBarOff = kRingBytes;                        // full[kStages], empty[kStages]
constexpr size_t kFlagOff = kBarOff + 2 * kStages * sizeof(uint64_t);  // abort flag, issued count
constexpr size_t kTblOff = kFlagOff + 16;                     // block-table slice of the split
constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kTblOff + kMaxTableSlice * sizeof(int32_t);
constexpr int kRedStride = kHeadDim + 8;                      // padded rows of the warp-merge buffer
static_assert((size_t)kConsumerWarps * 16 * kRedStride * 4 + kConsumerWarps * 16 * 8 <= kRingBytes,
              "merge buffers must fit in the ring");

struct MmaMaps {
    CUtensorMap k;
    CUtensorMap v;
};

template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1);

template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
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

// Shared-memory line (128 bytes) of token t (0..63 in the stage), column half h.
// Rows of one staged box are R = min(block_size, 64) lines; a stage holds 64 / R boxes,
// each [2 halves][R rows][64 columns].
__device__ __forceinline__ uint32_t line_of(int t, int h, int R_log2) {
    const int R = 1 << R_log2;
    return (uint32_t)(((t >> R_log2) << (R_log2 + 1)) + h * R + (t & (R - 1)));
}

// Byte address of the 16-byte chunk `c` (0..15 over the 128 columns) of token t.
__device__ __forceinline__ uint32_t chunk_addr(uint32_t base, int t, int c, int R_log2) {
    return base + line_of(t, c >> 3, R_log2) * 128u + ((uint32_t)((c & 7) ^ (t & 7)) << 4);
}

template <typename T>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi) {
    return Elem<T>::pack2(lo, hi);
}

template <typename T>
__device__ __forceinline__ uint16_t out_bits(float x);
template <>
__device__ __forceinline__ uint16_t out_bits<__half>(float x) {
    return __half_as_ushort(__float2half_rn(x));
}
template <>
__device__ __forceinline__ uint16_t out_bits<__nv_bfloat16>(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Issue the TMA loads of one stage: tokens [base, min(base + 64, tok_end)).
__device__ __forceinline__ void issue_stage(const DecodeArgs& a, const MmaMaps& maps, const int32_t* tbl, int tbl0,
                                            int hk, int base, int tok_end, uint32_t kdst, uint64_t* bar,
                                            int R_log2) {
    const int B = a.block_size;
    const int R = 1 << R_log2;                   // rows per box: min(B, 64)
    const int first = base / B;
    const int last = (min(base + kStageTokens, tok_end) - 1) / B;
    const int within = (B > kStageTokens) ? (base % B) : 0;
    int phys[4];
    uint32_t bytes = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        phys[j] = -1;
        if (first + j <= last) {
            const int p = tbl[first + j - tbl0];
            if (p >= 0 && p < a.num_blocks) {
                phys[j] = p;
                bytes += 2u * 2u * (uint32_t)R * 128u;   // K and V, two 64-column halves
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
            const uint32_t box = kdst + (uint32_t)(j * 2 * R) * 128u;
            tma_load_2d(box, &maps.k, 0, row, bar);
            tma_load_2d(box + (uint32_t)R * 128u, &maps.k, 64, row, bar);
            tma_load_2d(box + kStageKBytes, &maps.v, 0, row, bar);
            tma_load_2d(box + kStageKBytes + (uint32_t)R * 128u, &maps.v, 64, row, bar);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_mma_kernel(const DecodeArgs a, const __grid_constant__ MmaMaps maps, const int R_log2) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;                  // 1024-aligned for the swizzle
    unsigned char* base_ptr = smem_raw + (ring - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(base_ptr + kBarOff);
    uint64_t* empty = full + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + kFlagOff);
    volatile int* issued_count = abort_flag + 1;
    int32_t* tbl = reinterpret_cast<int32_t*>(base_ptr + kTblOff);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, hk = blockIdx.y, s = blockIdx.z;
    const int Hq = a.num_q_heads;
    const int G = Hq / a.num_kv_heads;
    const int B = a.block_size;

    if (tid == 0) {
        prefetch_map(&maps.k);
        prefetch_map(&maps.v);
#pragma unroll
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        *abort_flag = 0;
        *issued_count = 0;
        fence_mbar_init();
    }
    grid_dependency_wait();

    // the split's slice of the block table and the context length, loaded together
    const int tps = a.tokens_per_split;
    const int tok0 = split * tps;
    const int tbl0 = tok0 / B;
    const int ntbl = min(tps / B, a.max_blocks_per_seq - tbl0);
    {
        const int32_t* row = a.block_tables + (size_t)s * a.max_blocks_per_seq + tbl0;
        for (int j = tid; j < ntbl; j += kThreads) tbl[j] = row[j];
    }
    int Lctx = a.context_lens[s];
    const int cap = a.max_blocks_per_seq * B;
    if (Lctx < 0 || Lctx > cap) {
        if (tid == 0 && split == 0 && hk == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
        Lctx = Lctx < 0 ? 0 : cap;
    }
    __syncthreads();
    if (Lctx == 0) {
        if (split == 0 && tid < kHeadDim) {
            uint16_t* out = static_cast<uint16_t*>(a.out);
            for (int g = 0; g < G; ++g) out[((size_t)s * Hq + hk * G + g) * kHeadDim + tid] = 0;
        }
        return;
    }
    if (tok0 >= Lctx) return;
    const int tok1 = min(Lctx, tok0 + tps);
    const int nsplit_s = (Lctx + tps - 1) / tps;
    const int nst = (tok1 - tok0 + kStageTokens - 1) / kStageTokens;
    grid_launch_dependents();

    const int qr = lane >> 2, qc = (lane & 3) * 2;
    float m_run[2] = {-INFINITY, -INFINITY};   // rows qr and qr + 8, log2 units
    float l_run[2] = {0.f, 0.f};               // this thread's columns only
    float o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

    if (warp == kConsumerWarps) {
        // ---------------- producer warp: one lane keeps the ring full ----------------
        if (lane == 0) {
            int i = 0;
            for (; i < nst; ++i) {
                const int st = i % kStages;
                if (i >= kStages) {
                    if (!mbar_wait_bounded(&empty[st], (uint32_t)((i / kStages) - 1) & 1u)) {
                        flag_status(a.status, PA_DEV_TIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                    fence_proxy_async_smem();   // consumers' reads of this buffer precede the overwrite
                }
                if (*abort_flag) break;
                issue_stage(a, maps, tbl, tbl0, hk, tok0 + i * kStageTokens, tok1, ring + (uint32_t)st * kStageBytes,
                            &full[st], R_log2);
            }
            *issued_count = i;
        }
    } else {
        // ---------------- consumer warps: tokens [16w, 16w + 16) of every stage ----------------
        uint32_t qa[8][4];
        {
            const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
            const size_t row0 = ((size_t)s * Hq + hk * G + qr) * kHeadDim;
            const size_t row1 = row0 + 8 * kHeadDim;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int d = ks * 16 + qc;
                qa[ks][0] = (qr < G) ? q32[(row0 + d) >> 1] : 0u;
                qa[ks][1] = (qr + 8 < G) ? q32[(row1 + d) >> 1] : 0u;
                qa[ks][2] = (qr < G) ? q32[(row0 + d + 8) >> 1] : 0u;
                qa[ks][3] = (qr + 8 < G) ? q32[(row1 + d + 8) >> 1] : 0u;
            }
        }
        const int t_warp = warp * 16;
        const int tk = t_warp + (lane & 7) + ((lane >> 4) << 3);   // ldmatrix rows: K tile
        const int ck = (lane >> 3) & 1;
        const int tv = t_warp + (lane & 7) + (((lane >> 3) & 1) << 3);   // V tile (transposed)
        const int cv = lane >> 4;

        for (int i = 0; i < nst; ++i) {
            const int st = i % kStages;
            if (!mbar_wait_bounded(&full[st], (uint32_t)(i / kStages) & 1u)) {
                flag_status(a.status, PA_DEV_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            if (*abort_flag) break;
            const uint32_t kbase = ring + (uint32_t)st * kStageBytes;
            const uint32_t vbase = kbase + kStageKBytes;
            const int nvalid = min(kStageTokens, tok1 - (tok0 + i * kStageTokens));

            if (t_warp < nvalid) {
                if (nvalid < t_warp + 16) {
                    // rows past the context may hold stale or unwritten data: zero this warp's
                    // V rows there so that P = 0 never meets a non-finite value in P.V
                    uint4* vz = reinterpret_cast<uint4*>(base_ptr + (size_t)st * kStageBytes + kStageKBytes);
                    for (int idx = lane; idx < (t_warp + 16 - nvalid) * 16; idx += 32) {
                        const int t = nvalid + (idx >> 4);
                        const int c = idx & 15;
                        vz[line_of(t, c >> 3, R_log2) * 8 + (c & 7)] = make_uint4(0, 0, 0, 0);
                    }
                    __syncwarp();
                }
                // ---- S = Q K^T for this warp's 16 tokens ----
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(chunk_addr(kbase, tk, 2 * ks + ck, R_log2), b0, b1, b2, b3);
                    mma16816<T>(sc[0], qa[ks], b0, b1);
                    mma16816<T>(sc[1], qa[ks], b2, b3);
                }
                // ---- online softmax over the 16 columns, rows qr and qr + 8 ----
                float p[2][4];
                float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = t_warp + n * 8 + qc + (e & 1);
                        const float x = sc[n][e] * a.scale_log2;
                        p[n][e] = (col < nvalid) ? x : -INFINITY;
                        mx[e >> 1] = fmaxf(mx[e >> 1], p[n][e]);
                    }
                float alpha[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                    const float m_new = fmaxf(m_run[r], mx[r]);
                    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                    alpha[r] = exp2f(m_run[r] - m_use);
                    m_run[r] = m_new;
                    mx[r] = m_use;
                }
                float rs[2] = {0.f, 0.f};
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        p[n][e] = exp2f(p[n][e] - mx[e >> 1]);
                        rs[e >> 1] += p[n][e];
                    }
                l_run[0] = l_run[0] * alpha[0] + rs[0];
                l_run[1] = l_run[1] * alpha[1] + rs[1];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    o[j][0] *= alpha[0];
                    o[j][1] *= alpha[0];
                    o[j][2] *= alpha[1];
                    o[j][3] *= alpha[1];
                }
                // ---- O += P V ----
                uint32_t pa_[4];
                pa_[0] = pack_pair<T>(p[0][0], p[0][1]);
                pa_[1] = pack_pair<T>(p[0][2], p[0][3]);
                pa_[2] = pack_pair<T>(p[1][0], p[1][1]);
                pa_[3] = pack_pair<T>(p[1][2], p[1][3]);
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(chunk_addr(vbase, tv, 2 * np + cv, R_log2), b0, b1, b2, b3);
                    mma16816<T>(o[2 * np], pa_, b0, b1);
                    mma16816<T>(o[2 * np + 1], pa_, b2, b3);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);   // this warp is done with the stage's buffers
        }
    }

    __syncthreads();
    if (*abort_flag) {
        if (tid == 0) {
            // let every copy still in flight land before the CTA's shared memory is released
            const int n = *issued_count;
            for (int st = 0; st < kStages; ++st) {
                int last = -1;
                for (int i = st; i < n; i += kStages) last = i;
                if (last >= 0) (void)mbar_wait_bounded(&full[st], (uint32_t)(last / kStages) & 1u);
            }
        }
        return;
    }

    // ---- merge the four consumer warps: per row, M = max m_w, o = sum 2^(m_w - M) o_w ----
    float* red_o = reinterpret_cast<float*>(base_ptr);        // [4][16][kRedStride]
    float2* red_ml = reinterpret_cast<float2*>(base_ptr + (size_t)kConsumerWarps * 16 * kRedStride * 4);
    if (warp < kConsumerWarps) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int d = j * 8 + qc;
            *reinterpret_cast<float2*>(&red_o[(warp * 16 + qr) * kRedStride + d]) = make_float2(o[j][0], o[j][1]);
            *reinterpret_cast<float2*>(&red_o[(warp * 16 + qr + 8) * kRedStride + d]) =
                make_float2(o[j][2], o[j][3]);
        }
        if ((lane & 3) == 0) {
            red_ml[warp * 16 + qr] = make_float2(m_run[0], l_run[0]);
            red_ml[warp * 16 + qr + 8] = make_float2(m_run[1], l_run[1]);
        }
    }
    __syncthreads();
    if (tid >= kHeadDim) return;
    const int d = tid;
    for (int g = 0; g < G; ++g) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_ml[w * 16 + g].x);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float2 ml = red_ml[w * 16 + g];
            const float sc = exp2f(ml.x - M);   // warps without a valid token: 2^-inf = 0
            num = fmaf(sc, red_o[(w * 16 + g) * kRedStride + d], num);
            den = fmaf(sc, ml.y, den);
        }
        const int h = hk * G + g;
        if (nsplit_s == 1) {
            static_cast<uint16_t*>(a.out)[((size_t)s * Hq + h) * kHeadDim + d] = out_bits<T>(num / den);
        } else {
            const size_t pidx = ((size_t)s * Hq + h) * a.max_splits + split;
            a.part_o[pidx * kHeadDim + d] = num;
            if (d == 0) a.part_ml[pidx] = make_float2(M, den);
        }
    }
}

// ---- host side: tensor maps (cached per cache pointer) and launch ----

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

struct MapKey {
    const void* ptr;
    unsigned long long rows;
    int box_rows;
};

struct MapCacheEntry {
    MapKey key;
    CUtensorMap map;
    bool used;
};

constexpr int kMapCacheSize = 128;
MapCacheEntry g_maps[kMapCacheSize];
int g_map_next = 0;
std::mutex g_map_mutex;

bool make_map(const void* base, unsigned long long rows, int box_rows, CUtensorMap* out) {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (auto& e : g_maps)
        if (e.used && e.key.ptr == base && e.key.rows == rows && e.key.box_rows == box_rows) {
            *out = e.map;
            return true;
        }
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUtensorMap m;
    CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    MapCacheEntry& e = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCacheSize;
    e.key = MapKey{base, rows, box_rows};
    e.map = m;
    e.used = true;
    *out = m;
    return true;
}

template <typename T>
cudaError_t launch_split_mma(const DecodeArgs& a, const MmaMaps& maps, int R_log2, cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    auto kernel = decode_split_mma_kernel<T>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.max_splits, a.num_kv_heads, a.num_seqs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
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

bool mma_supports_group(int group) { return group >= 1 && group <= 16; }

cudaError_t launch_decode_split_mma(const DecodeArgs& a, int dtype, cudaStream_t stream) {
    const int R = a.block_size < kStageTokens ? a.block_size : kStageTokens;
    int R_log2 = 0;
    while ((1 << R_log2) < R) ++R_log2;
    const unsigned long long rows = (unsigned long long)a.num_blocks * a.num_kv_heads * a.block_size;
    if (rows == 0 || rows > 0x7fffffffull) return cudaErrorInvalidValue;
    MmaMaps maps;
    if (!make_map(a.k_cache, rows, R, &maps.k) || !make_map(a.v_cache, rows, R, &maps.v))
        return cudaErrorInvalidValue;
    return dtype == PA_BF16 ? launch_split_mma<__nv_bfloat16>(a, maps, R_log2, stream)
                            : launch_split_mma<__half>(a, maps, R_log2, stream);
}

}  // namespace pa
