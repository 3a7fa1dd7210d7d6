// Several new query tokens per sequence, any number of them: tensor-core tiles of 64 query rows.
//
// What it computes (the same as the persistent kernel's several-token mode): sequence s owns
// query rows q_start[s] .. q_start[s+1]-1, its n newest tokens, the last n of its L cached ones;
// token i sits at position L - n + i and attends causally over positions 0 .. L - n + i:
// "显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结", §五.1 (walk the logical blocks
// through block_tables, q.k, running-max softmax, weight V, normalise), for the chunked prefill
// its closing section points to.
//
// Decomposition: one CTA per (64-row tile, kv head, sequence).  A segment's query rows are
// r = i * G + g (new token i, member g of the GQA group); consumer warp w owns rows
// [16 w, 16 w + 16) of the tile and every token of every stage:
//   S (16 x 64)   = Q (16 x 128) K_stage^T        mma.sync m16n8k16, fp32 accumulation
//   O (16 x 128) += P (16 x 64, from S's C fragments) V_stage
// with a running max / sum per row and each row's causal limit in the mask.  One producer warp
// streams 64-token stages of K and V (2-D TMA, 128-byte swizzle, as the decode kernels) up to
// the tile's last position into a 3-deep ring; full / empty mbarriers, every wait bounded.
// No warp shares rows with another, so nothing is merged: each warp normalises and writes its
// rows.  bf16 weights enter the PV product as a high and a low part.
#include "pa_internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <type_traits>

namespace pa {

namespace {

constexpr int kWarps = 4;                                   // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;                 // + one TMA producer warp
constexpr int kRows = kWarps * 16;                          // query rows per tile
constexpr int kStages = 3;
constexpr int kStageKBytes = kStageTokens * kHeadDim * 2;   // 16 KB of K per stage (V the same)
constexpr int kStageBytes = 2 * kStageKBytes;
constexpr size_t kRingBytes = (size_t)kStages * kStageBytes;
constexpr size_t kBarOff = kRingBytes;                      // full[kStages], empty[kStages]
constexpr size_t kFlagOff = kBarOff + 2 * kStages * sizeof(uint64_t);  // abort flag, issued count
constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kFlagOff + 16;

struct Maps {
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

// Named barrier of the four consumer warps.
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
}

// Shared-memory line (128 bytes) of token t (0..63 of the stage), column half h: a stage holds
// 64 / R boxes of [2 halves][R rows][64 columns], R = min(block_size, 64).
__device__ __forceinline__ uint32_t line_of(int t, int h, int R_log2) {
    const int R = 1 << R_log2;
    return (uint32_t)(((t >> R_log2) << (R_log2 + 1)) + h * R + (t & (R - 1)));
}

// Byte address of 16-byte chunk c (0..15 over the 128 columns) of token t, 128-byte swizzle.
__device__ __forceinline__ uint32_t chunk_addr(uint32_t base, int t, int c, int R_log2) {
    return base + line_of(t, c >> 3, R_log2) * 128u + ((uint32_t)((c & 7) ^ (t & 7)) << 4);
}

// Issue the TMA loads of one stage: the blocks holding tokens [base, min(base + 64, tok_end)).
__device__ __forceinline__ void issue_stage(const DecodeArgs& a, const Maps& maps, const int32_t* table_row, int hk,
                                            int base, int tok_end, uint32_t kdst, uint64_t* bar, int R_log2) {
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
    prefill_mma_kernel(const DecodeArgs a, const __grid_constant__ Maps maps, const int R_log2) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;   // 1024-aligned for the swizzle
    unsigned char* base_ptr = smem_raw + (ring - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(base_ptr + kBarOff);
    uint64_t* empty = full + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + kFlagOff);
    volatile int* issued_count = abort_flag + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, hk = blockIdx.y, s = blockIdx.z;
    const int G = a.num_q_heads / a.num_kv_heads;
    const int cap = a.max_blocks_per_seq * a.block_size;

    grid_dependency_wait();
    int L = a.context_lens[s];
    if (L < 0 || L > cap) {
        if (tid == 0 && tile == 0 && hk == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
        L = L < 0 ? 0 : cap;
    }
    if (tid == 0 && tile == 0 && hk == 0) {
        const int n_raw = a.q_start[s + 1] - a.q_start[s];
        const int r0_raw = a.q_start[s];
        if (n_raw < 0 || n_raw > L || n_raw > a.max_q || r0_raw < 0 || r0_raw + n_raw > a.q_rows)
            flag_status(a.status, PA_DEV_BAD_CONTEXT);
    }
    const QSpan qs = q_span(a, s, L);
    const int rows = qs.n * G;
    const int r0 = tile * kRows;
    if (r0 >= rows) return;   // uniform for the CTA
    // tokens the tile needs: up to the position of its last row
    const int r_last = min(r0 + kRows, rows) - 1;
    const int t_end = L - qs.n + r_last / G + 1;
    const int nst = (t_end + kStageTokens - 1) / kStageTokens;

    if (tid == 0) {
        prefetch_map(&maps.k);
        prefetch_map(&maps.v);
#pragma unroll
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarps);
        }
        *abort_flag = 0;
        *issued_count = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_launch_dependents();

    if (warp == kWarps) {
        // ---------------- producer warp: one lane keeps the ring full ----------------
        if (lane == 0) {
            const int32_t* table_row = a.block_tables + (size_t)s * a.max_blocks_per_seq;
            int i = 0;
            for (; i < nst; ++i) {
                const int st = i % kStages;
                if (i >= kStages) {
                    if (!mbar_wait_bounded(&empty[st], (uint32_t)((i / kStages) - 1) & 1u)) {
                        flag_status(a.status, PA_DEV_TIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                    fence_proxy_async_smem();   // consumers' generic accesses precede the overwrite
                }
                if (*abort_flag) break;
                issue_stage(a, maps, table_row, hk, i * kStageTokens, t_end, ring + (uint32_t)st * kStageBytes,
                            &full[st], R_log2);
            }
            *issued_count = i;
        }
    } else {
        // ---------------- consumer warps: rows [16 w, 16 w + 16) of the tile ----------------
        const int gid = lane >> 2, tig = lane & 3;
        const int ra = r0 + warp * 16 + gid, rb = ra + 8;   // this lane's two rows
        // newest position each row attends to (-1: no such row)
        const int lim_a = (ra < rows) ? L - qs.n + ra / G : -1;
        const int lim_b = (rb < rows) ? L - qs.n + rb / G : -1;
        const int warp_lim = __reduce_max_sync(0xffffffffu, max(lim_a, lim_b));
        // Q rows as A fragments: row ra (registers 0, 2) and rb (1, 3), dims ks*16 + tig*2 (+8)
        uint32_t qa[8][4];
        {
            const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
            const size_t oa = (ra < rows) ? q_offset(a, qs, hk, G, ra) : 0;
            const size_t ob = (rb < rows) ? q_offset(a, qs, hk, G, rb) : 0;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int d = ks * 16 + tig * 2;
                qa[ks][0] = (ra < rows) ? q32[(oa + d) >> 1] : 0u;
                qa[ks][1] = (rb < rows) ? q32[(ob + d) >> 1] : 0u;
                qa[ks][2] = (ra < rows) ? q32[(oa + d + 8) >> 1] : 0u;
                qa[ks][3] = (rb < rows) ? q32[(ob + d + 8) >> 1] : 0u;
            }
        }
        constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
        float m_run[2] = {-INFINITY, -INFINITY};   // rows ra, rb, log2 units
        float l_run[2] = {0.f, 0.f};               // this lane's columns only
        float o[16][4];
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        // ldmatrix row addresses: K (B of S = Q K^T, tokens 16 tg + ...) and V (B of O += P V)
        const int tk = (lane & 7) + ((lane >> 4) << 3);
        const int ck = (lane >> 3) & 1;
        const int tv = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int cv = lane >> 4;
        bool dead = false;

        for (int i = 0; i < nst; ++i) {
            const int st = i % kStages;
            const int base = i * kStageTokens;
            dead = dead || __any_sync(0xffffffffu, *abort_flag != 0);
            if (!dead && !__all_sync(0xffffffffu, mbar_wait_bounded(&full[st], (uint32_t)(i / kStages) & 1u))) {
                if (lane == 0) {
                    flag_status(a.status, PA_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
                dead = true;
            }
            const uint32_t kbase = ring + (uint32_t)st * kStageBytes;
            const uint32_t vbase = kbase + kStageKBytes;
            if (i == nst - 1) {
                // the last stage: rows from t_end on are masked, but they can hold pool slots past
                // the context or stale data; zero them so that P = 0 never meets a non-finite V
                const int nvalid = t_end - base;
                uint4* vz = reinterpret_cast<uint4*>(base_ptr + (size_t)st * kStageBytes + kStageKBytes);
                if (!dead)
                    for (int idx = tid; idx < (kStageTokens - nvalid) * 16; idx += kWarps * 32) {
                        const int t = nvalid + (idx >> 4);
                        const int cc = idx & 15;
                        vz[line_of(t, cc >> 3, R_log2) * 8 + (cc & 7)] = make_uint4(0, 0, 0, 0);
                    }
                consumers_sync();   // every warp reads every V row of the stage
            }
            if (!dead && base <= warp_lim) {
                // ---- S = Q K^T over the stage's 64 tokens: 8 column tiles of 8 tokens ----
                float sc[8][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                    for (int tg = 0; tg < 4; ++tg) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(chunk_addr(kbase, tg * 16 + tk, 2 * ks + ck, R_log2), b0, b1, b2, b3);
                        mma16816<T>(sc[2 * tg], qa[ks], b0, b1);
                        mma16816<T>(sc[2 * tg + 1], qa[ks], b2, b3);
                    }
                }
                // ---- online softmax, rows ra (elements 0, 1) and rb (2, 3), causal limits ----
                float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = base + j * 8 + tig * 2 + (e & 1);
                        const float x = (t <= ((e < 2) ? lim_a : lim_b)) ? sc[j][e] * a.scale_log2 : -INFINITY;
                        sc[j][e] = x;
                        mx[e >> 1] = fmaxf(mx[e >> 1], x);
                    }
                float alpha[2], m_use[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                    const float m_new = fmaxf(m_run[r], mx[r]);
                    m_use[r] = (m_new == -INFINITY) ? 0.f : m_new;
                    alpha[r] = exp2f(m_run[r] - m_use[r]);
                    m_run[r] = m_new;
                }
                float rs[2] = {0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        sc[j][e] = exp2f(sc[j][e] - m_use[e >> 1]);
                        rs[e >> 1] += sc[j][e];
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
                // ---- O += P V: P's C fragments of column tiles 2kt, 2kt + 1 are the A fragment
                // of k-step kt (16 tokens) ----
#pragma unroll
                for (int kt = 0; kt < 4; ++kt) {
                    uint32_t ph[4], pl[4];
                    ph[0] = Elem<T>::pack2(sc[2 * kt][0], sc[2 * kt][1]);
                    ph[1] = Elem<T>::pack2(sc[2 * kt][2], sc[2 * kt][3]);
                    ph[2] = Elem<T>::pack2(sc[2 * kt + 1][0], sc[2 * kt + 1][1]);
                    ph[3] = Elem<T>::pack2(sc[2 * kt + 1][2], sc[2 * kt + 1][3]);
                    if (kSplitP) {
                        const float2 h0 = Elem<T>::to_float2(ph[0]), h1 = Elem<T>::to_float2(ph[1]);
                        const float2 h2 = Elem<T>::to_float2(ph[2]), h3 = Elem<T>::to_float2(ph[3]);
                        pl[0] = Elem<T>::pack2(sc[2 * kt][0] - h0.x, sc[2 * kt][1] - h0.y);
                        pl[1] = Elem<T>::pack2(sc[2 * kt][2] - h1.x, sc[2 * kt][3] - h1.y);
                        pl[2] = Elem<T>::pack2(sc[2 * kt + 1][0] - h2.x, sc[2 * kt + 1][1] - h2.y);
                        pl[3] = Elem<T>::pack2(sc[2 * kt + 1][2] - h3.x, sc[2 * kt + 1][3] - h3.y);
                    }
#pragma unroll
                    for (int np = 0; np < 8; ++np) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(chunk_addr(vbase, kt * 16 + tv, 2 * np + cv, R_log2), b0, b1, b2, b3);
                        mma16816<T>(o[2 * np], ph, b0, b1);
                        mma16816<T>(o[2 * np + 1], ph, b2, b3);
                        if (kSplitP) {
                            mma16816<T>(o[2 * np], pl, b0, b1);
                            mma16816<T>(o[2 * np + 1], pl, b2, b3);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);   // this warp is done with the stage's buffers
        }
        // ---- normalise and write this lane's two rows ----
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
        }
        if (!dead) {
            T* out = static_cast<T*>(a.out);
            if (ra < rows) {
                const float inv = 1.f / l_run[0];
                uint32_t* dst = reinterpret_cast<uint32_t*>(out + q_offset(a, qs, hk, G, ra));
#pragma unroll
                for (int j = 0; j < 16; ++j) dst[(j * 8 + tig * 2) >> 1] = Elem<T>::pack2(o[j][0] * inv, o[j][1] * inv);
            }
            if (rb < rows) {
                const float inv = 1.f / l_run[1];
                uint32_t* dst = reinterpret_cast<uint32_t*>(out + q_offset(a, qs, hk, G, rb));
#pragma unroll
                for (int j = 0; j < 16; ++j) dst[(j * 8 + tig * 2) >> 1] = Elem<T>::pack2(o[j][2] * inv, o[j][3] * inv);
            }
        }
    }

    __syncthreads();
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool encode_map(const void* base, unsigned long long rows, int box_rows, CUtensorMap* out) {
    auto fn = encode_fn();
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
cudaError_t launch_impl(const DecodeArgs& a, const Maps& maps, int R_log2, cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    auto kernel = prefill_mma_kernel<T>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    const int G = a.num_q_heads / a.num_kv_heads;
    const long long tiles = ((long long)a.max_q * G + kRows - 1) / kRows;
    if (tiles > 0x7fffffffLL || a.num_kv_heads > 65535 || a.num_seqs > 65535) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, a.num_kv_heads, a.num_seqs);
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

cudaError_t launch_prefill_mma(const DecodeArgs& a, int dtype, cudaStream_t stream) {
    const int R = a.block_size < kStageTokens ? a.block_size : kStageTokens;
    int R_log2 = 0;
    while ((1 << R_log2) < R) ++R_log2;
    const unsigned long long rows = (unsigned long long)a.num_blocks * a.num_kv_heads * a.block_size;
    if (rows == 0 || rows > 0x7fffffffull) return cudaErrorInvalidValue;
    Maps maps;
    if (!encode_map(a.k_cache, rows, R, &maps.k) || !encode_map(a.v_cache, rows, R, &maps.v))
        return cudaErrorInvalidValue;
    return dtype == PA_BF16 ? launch_impl<__nv_bfloat16>(a, maps, R_log2, stream)
                            : launch_impl<__half>(a, maps, R_log2, stream);
}

}  // namespace pa
