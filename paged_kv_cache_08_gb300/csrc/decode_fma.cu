// Paged decode attention, split pass, CUDA-core path.
//
// What it computes ("显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结", §五.1 kernel
// sketch): for one sequence and one kv head, loop over the logical blocks, look up each
// physical block in block_tables, stage its K and V rows in shared memory, take q.k for every
// token, keep a running max and sum (the "local rescaled accumulation"), weight V, and
// normalise at the end.  Address rule: "端侧 SLM 显存保活术：在 4GB 内存板卡上实现轻量
// PagedAttention 与 KV 缓存分块", section "注意力寻址：非连续物理块的间接寻址内核".
//
// GB300 design (differs from the page's one-CTA-per-(head, sequence) sketch):
//  * one CTA per (token split, kv head, sequence); the G query heads of the kv head's GQA
//    group share every staged K/V tile, so each byte of cache is read from HBM once;
//  * a (block, kv-head) tile is one contiguous run of block_size*128 elements, fetched
//    whole by one bulk TMA copy (cp.async.bulk) into a 3-stage shared-memory ring of
//    64-token stages, completion tracked by mbarrier transaction counts; a single thread
//    issues the copies and checks every block id against the pool before using it;
//  * scores: a half-warp per token, 8 dimensions per lane, fp32 FMAs against q held in
//    registers (pre-multiplied by scale*log2 e), xor-shuffle reduction over the 16 lanes;
//  * softmax: one warp per query head per stage, running max / sum in base 2;
//  * P.V: a lane owns 8 output dimensions of all G heads for 8 of the stage's tokens; the
//    eight token groups are summed through shared memory once, at the end of the split;
//  * a split that covers the whole sequence writes the normalised output directly; other
//    splits write (m, l, unnormalised o) partials for the combine pass.
#include "pa_internal.cuh"

#include <atomic>

namespace pa {

namespace {

constexpr int kThreads = 128;
constexpr int kStages = 3;
constexpr int kTileElems = kStageTokens * kHeadDim;  // one stage of K (or of V)

template <int G>
struct FmaSmem {
    static constexpr size_t kStageBytes = 2ull * kTileElems * 2;  // K and V, 16-bit elements
    static constexpr size_t kRing = kStages * kStageBytes;
    static constexpr size_t kScores = kRing;                                  // float [G][64]
    static constexpr size_t kMl = kScores + sizeof(float) * G * kStageTokens;  // float2 [G]
    static constexpr size_t kAlpha = kMl + sizeof(float2) * G;                 // float [G]
    static constexpr size_t kBars = (kAlpha + sizeof(float) * G + 7) & ~size_t(7);
    static constexpr size_t kTotal = kBars + sizeof(uint64_t) * kStages;
    static_assert(8ull * G * kHeadDim * sizeof(float) <= kRing, "reduction buffer must fit the ring");
};

template <typename T>
__device__ __forceinline__ uint16_t to_bits(float x);
template <>
__device__ __forceinline__ uint16_t to_bits<__half>(float x) {
    return __half_as_ushort(__float2half_rn(x));
}
template <>
__device__ __forceinline__ uint16_t to_bits<__nv_bfloat16>(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Issue the bulk copies of stage `stage` (tokens [base, min(base+64, tok_end))) into `kdst`
// and `vdst`.  Shared-memory row r holds token base + r.  Only block ids inside the pool
// are fetched; the barrier expects exactly the bytes of the copies issued.
template <typename T>
__device__ __forceinline__ void issue_stage(const DecodeArgs& a, const int32_t* table, int hk, int base,
                                            int tok_end, T* kdst, T* vdst, uint64_t* bar) {
    const int B = a.block_size;
    const T* kc = static_cast<const T*>(a.k_cache);
    const T* vc = static_cast<const T*>(a.v_cache);
    const int last = min(base + kStageTokens, tok_end) - 1;
    if (B >= kStageTokens) {
        // one block holds the whole stage: rows [base % B, base % B + 64) of block base / B
        const int phys = table[base / B];
        const bool ok = phys >= 0 && phys < a.num_blocks;
        const uint32_t bytes = kTileElems * sizeof(T);
        mbar_arrive_expect_tx(bar, ok ? 2u * bytes : 0u);
        if (ok) {
            const size_t src = (((size_t)phys * a.num_kv_heads + hk) * B + (base % B)) * kHeadDim;
            bulk_copy_g2s(kdst, kc + src, bytes, bar);
            bulk_copy_g2s(vdst, vc + src, bytes, bar);
        } else {
            flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
        }
        return;
    }
    const int first_blk = base / B;
    const int nblk = last / B - first_blk + 1;  // <= 64 / 16
    int phys[kStageTokens / 16];
    uint32_t total = 0;
    const uint32_t tile_bytes = (uint32_t)B * kHeadDim * sizeof(T);
#pragma unroll
    for (int j = 0; j < kStageTokens / 16; ++j) {
        phys[j] = -1;
        if (j < nblk) {
            const int p = table[first_blk + j];
            if (p >= 0 && p < a.num_blocks) {
                phys[j] = p;
                total += 2u * tile_bytes;
            } else {
                flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
            }
        }
    }
    mbar_arrive_expect_tx(bar, total);
#pragma unroll
    for (int j = 0; j < kStageTokens / 16; ++j) {
        if (phys[j] >= 0) {
            const size_t src = ((size_t)phys[j] * a.num_kv_heads + hk) * B * kHeadDim;
            bulk_copy_g2s(kdst + (size_t)j * B * kHeadDim, kc + src, tile_bytes, bar);
            bulk_copy_g2s(vdst + (size_t)j * B * kHeadDim, vc + src, tile_bytes, bar);
        }
    }
}

// Slotted mode: position in a sequence's run list (run r, rows already taken from it).
struct RunCursor {
    int r;
    int in_run;
};

// Issue the bulk copies of tokens [base, min(base + 64, tok_end)) read through runs: each piece
// of a run is one contiguous group of rows of its (block, kv head) tile, copied to shared rows
// t - base.  The cursor stands at token base and is left at the stage's end.
template <typename T>
__device__ __forceinline__ void issue_stage_runs(const DecodeArgs& a, RunCursor& cur, int r_end, int hk, int base,
                                                 int tok_end, T* kdst, T* vdst, uint64_t* bar) {
    const T* kc = static_cast<const T*>(a.k_cache);
    const T* vc = static_cast<const T*>(a.v_cache);
    const int end = min(base + kStageTokens, tok_end);
    const uint32_t row_bytes = kHeadDim * sizeof(T);
    // pass 1: bytes of the stage's pieces; pass 2: the copies
    uint32_t total = 0;
    {
        RunCursor c = cur;
        for (int t = base; t < end && c.r < r_end;) {
            const int take = min(run_len(a, c.r) - c.in_run, end - t);
            total += 2u * (uint32_t)max(take, 0) * row_bytes;
            t += max(take, 0);
            c.in_run += max(take, 0);
            if (c.in_run >= run_len(a, c.r)) {
                ++c.r;
                c.in_run = 0;
            }
        }
    }
    mbar_arrive_expect_tx(bar, total);
    for (int t = base; t < end && cur.r < r_end;) {
        const int len = run_len(a, cur.r);
        const int take = min(len - cur.in_run, end - t);
        if (take > 0) {
            const int blk = a.runs[3 * cur.r], off = a.runs[3 * cur.r + 1];
            const size_t src = (((size_t)blk * a.num_kv_heads + hk) * a.block_size + off + cur.in_run) * kHeadDim;
            bulk_copy_g2s(kdst + (size_t)(t - base) * kHeadDim, kc + src, (uint32_t)take * row_bytes, bar);
            bulk_copy_g2s(vdst + (size_t)(t - base) * kHeadDim, vc + src, (uint32_t)take * row_bytes, bar);
            t += take;
            cur.in_run += take;
        }
        if (cur.in_run >= len) {
            ++cur.r;
            cur.in_run = 0;
        }
    }
}

template <typename T, int G>
__global__ void __launch_bounds__(kThreads, 2) decode_split_fma_kernel(const DecodeArgs a) {
    using L = FmaSmem<G>;
    extern __shared__ __align__(128) unsigned char smem[];
    T* ring = reinterpret_cast<T*>(smem);
    float* sc = reinterpret_cast<float*>(smem + L::kScores);
    float2* ml = reinterpret_cast<float2*>(smem + L::kMl);
    float* alpha_s = reinterpret_cast<float*>(smem + L::kAlpha);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = lane >> 4, l16 = lane & 15;
    const int split = blockIdx.x, hk = blockIdx.y, s = blockIdx.z;
    const int Hq = a.num_q_heads;

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    grid_dependency_wait();  // the cache and q may come from the preceding kernel

    const int cap = a.max_blocks_per_seq * a.block_size;
    int Lctx;
    RunCursor cur{0, 0};
    int r_end = 0;
    if (a.runs) {
        // slotted mode: the context is the runs' total length; a run that leaves its block or
        // the pool counts as empty and is flagged; the total is capped at the planned capacity
        const int r0 = a.seq_runs[s];
        r_end = a.seq_runs[s + 1];
        int* total_s = reinterpret_cast<int*>(alpha_s);   // scratch before the first stage
        if (tid == 0) *total_s = 0;
        __syncthreads();
        int part = 0;
        for (int r = r0 + tid; r < r_end; r += kThreads) {
            const int len = run_len(a, r);
            if (len != a.runs[3 * r + 2] && split == 0 && hk == 0) flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
            part += len;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) atomicAdd(total_s, part);
        __syncthreads();
        Lctx = *total_s;
        __syncthreads();
        if (Lctx > cap) {
            if (tid == 0 && split == 0 && hk == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
            Lctx = cap;
        }
        cur.r = r0;
    } else {
        Lctx = a.context_lens[s];
        if (Lctx < 0 || Lctx > cap) {
            if (tid == 0 && split == 0 && hk == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
            Lctx = Lctx < 0 ? 0 : cap;
        }
    }
    const int tps = a.tokens_per_split;
    const int tok0 = split * tps;
    if (Lctx == 0) {
        if (split == 0) {
            uint16_t* out = static_cast<uint16_t*>(a.out);
#pragma unroll
            for (int g = 0; g < G; ++g) out[((size_t)s * Hq + hk * G + g) * kHeadDim + tid] = 0;
        }
        return;
    }
    if (tok0 >= Lctx) return;
    const int tok1 = min(Lctx, tok0 + tps);
    const int nsplit_s = (Lctx + tps - 1) / tps;
    const int nst = (tok1 - tok0 + kStageTokens - 1) / kStageTokens;
    const int32_t* table = a.block_tables ? a.block_tables + (size_t)s * a.max_blocks_per_seq : nullptr;

    __syncthreads();  // barriers initialised
    if (tid == 0) {
        if (a.runs) {
            // move the cursor to the split's first token
            for (int t = 0; t < tok0 && cur.r < r_end;) {
                const int take = min(run_len(a, cur.r) - cur.in_run, tok0 - t);
                t += take;
                cur.in_run += take;
                if (cur.in_run >= run_len(a, cur.r)) {
                    ++cur.r;
                    cur.in_run = 0;
                }
            }
        }
        const int pre = min(kStages, nst);
        for (int i = 0; i < pre; ++i) {
            T* kd = ring + (size_t)i * 2 * kTileElems;
            if (a.runs)
                issue_stage_runs<T>(a, cur, r_end, hk, tok0 + i * kStageTokens, tok1, kd, kd + kTileElems, &bars[i]);
            else
                issue_stage<T>(a, table, hk, tok0 + i * kStageTokens, tok1, kd, kd + kTileElems, &bars[i]);
        }
    }
    grid_launch_dependents();

    // q of the G heads, 8 dimensions per lane, pre-scaled so that exp becomes exp2
    float qf[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) +
                                                          ((size_t)s * Hq + hk * G + g) * kHeadDim + l16 * 8);
        unpack8<T>(raw, qf[g]);
#pragma unroll
        for (int j = 0; j < 8; ++j) qf[g][j] *= a.scale_log2;
    }
    float o[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < 8; ++j) o[g][j] = 0.f;
    if (tid < G) {
        ml[tid] = make_float2(-INFINITY, 0.f);
    }

    const int tg = warp * 2 + half;  // token group of this half-warp in the P.V step
    int i = 0;
    bool timed_out = false;
    for (; i < nst; ++i) {
        const int st = i % kStages;
        const uint32_t parity = (uint32_t)(i / kStages) & 1u;
        const bool ok = mbar_wait_bounded(&bars[st], parity);
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        const T* Ks = ring + (size_t)st * 2 * kTileElems;
        const T* Vs = Ks + kTileElems;
        const int base = tok0 + i * kStageTokens;
        const int nvalid = min(kStageTokens, tok1 - base);

        // ---- scores: s[g][t] = (scale log2e) q_g . k_t ----
#pragma unroll 2
        for (int it = 0; it < 8; ++it) {
            const int t = warp * 16 + it * 2 + half;
            const uint4 kr = *reinterpret_cast<const uint4*>(Ks + t * kHeadDim + l16 * 8);
            float kf[8];
            unpack8<T>(kr, kf);
            float acc[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float x = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) x = fmaf(qf[g][j], kf[j], x);
                acc[g] = x;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], off);
            }
            if (l16 == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) sc[g * kStageTokens + t] = (t < nvalid) ? acc[g] : -INFINITY;
            }
        }
        __syncthreads();

        // ---- online softmax, one warp per head ----
        for (int g = warp; g < G; g += kThreads / 32) {
            const float x0 = sc[g * kStageTokens + lane];
            const float x1 = sc[g * kStageTokens + 32 + lane];
            const float mx = warp_max(fmaxf(x0, x1));
            const float2 prev = ml[g];
            const float m_new = fmaxf(prev.x, mx);
            const float p0 = exp2f(x0 - m_new), p1 = exp2f(x1 - m_new);
            sc[g * kStageTokens + lane] = p0;
            sc[g * kStageTokens + 32 + lane] = p1;
            const float sum = warp_sum(p0 + p1);
            const float alpha = exp2f(prev.x - m_new);
            if (lane == 0) {
                ml[g] = make_float2(m_new, prev.y * alpha + sum);
                alpha_s[g] = alpha;
            }
        }
        __syncthreads();

        // ---- o = alpha o + P V ----
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float al = alpha_s[g];
#pragma unroll
            for (int j = 0; j < 8; ++j) o[g][j] *= al;
        }
#pragma unroll 2
        for (int r = 0; r < 8; ++r) {
            const int t = tg * 8 + r;
            if (t < nvalid) {
                const uint4 vr = *reinterpret_cast<const uint4*>(Vs + t * kHeadDim + l16 * 8);
                float vf[8];
                unpack8<T>(vr, vf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float p = sc[g * kStageTokens + t];
#pragma unroll
                    for (int j = 0; j < 8; ++j) o[g][j] = fmaf(p, vf[j], o[g][j]);
                }
            }
        }
        __syncthreads();  // stage buffer and scores free again
        if (tid == 0 && i + kStages < nst) {
            fence_proxy_async_smem();
            T* kd = ring + (size_t)st * 2 * kTileElems;
            if (a.runs)
                issue_stage_runs<T>(a, cur, r_end, hk, tok0 + (i + kStages) * kStageTokens, tok1, kd, kd + kTileElems,
                                    &bars[st]);
            else
                issue_stage<T>(a, table, hk, tok0 + (i + kStages) * kStageTokens, tok1, kd, kd + kTileElems,
                               &bars[st]);
        }
    }

    if (timed_out) {
        if (tid == 0) flag_status(a.status, PA_DEV_TIMEOUT);
        // let every copy still in flight land before the CTA's shared memory is released
        for (int j = i; j < min(nst, i + kStages); ++j)
            (void)mbar_wait_bounded(&bars[j % kStages], (uint32_t)(j / kStages) & 1u);
        return;
    }

    // ---- sum the eight token groups' partial outputs through shared memory ----
    float* red = reinterpret_cast<float*>(smem);  // [8][G][128]; every copy has landed
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float4* dst = reinterpret_cast<float4*>(red + ((size_t)tg * G + g) * kHeadDim + l16 * 8);
        dst[0] = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
        dst[1] = make_float4(o[g][4], o[g][5], o[g][6], o[g][7]);
    }
    __syncthreads();
    const int d = tid;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc += red[((size_t)k * G + g) * kHeadDim + d];
        const float2 st = ml[g];
        const int h = hk * G + g;
        if (nsplit_s == 1) {
            static_cast<uint16_t*>(a.out)[((size_t)s * Hq + h) * kHeadDim + d] = to_bits<T>(acc / st.y);
        } else {
            const size_t p = ((size_t)s * Hq + h) * a.max_splits + split;
            a.part_o[p * kHeadDim + d] = acc;
            if (d == 0) a.part_ml[p] = st;
        }
    }
}

// ---- combine: out = sum_j 2^(m_j - M) o_j / sum_j 2^(m_j - M) l_j ----
template <typename T>
__global__ void __launch_bounds__(kHeadDim) decode_combine_kernel(const DecodeArgs a) {
    grid_dependency_wait();  // partials come from the split pass
    const int h = blockIdx.x, s = blockIdx.y, d = threadIdx.x;
    const int cap = a.max_blocks_per_seq * a.block_size;
    int Lctx = 0;
    if (a.runs) {
        for (int r = a.seq_runs[s]; r < a.seq_runs[s + 1]; ++r) Lctx += run_len(a, r);   // as the split pass
    } else {
        Lctx = a.context_lens[s];
    }
    Lctx = Lctx < 0 ? 0 : (Lctx > cap ? cap : Lctx);
    const int n = (Lctx + a.tokens_per_split - 1) / a.tokens_per_split;
    if (n <= 1) return;
    const size_t base = ((size_t)s * a.num_q_heads + h) * a.max_splits;
    float M = -INFINITY;
    for (int j = 0; j < n; ++j) M = fmaxf(M, a.part_ml[base + j].x);
    float lsum = 0.f, acc = 0.f;
    for (int j = 0; j < n; ++j) {
        const float2 mlj = a.part_ml[base + j];
        const float w = exp2f(mlj.x - M);
        lsum = fmaf(w, mlj.y, lsum);
        acc = fmaf(w, a.part_o[(base + j) * kHeadDim + d], acc);
    }
    static_cast<uint16_t*>(a.out)[((size_t)s * a.num_q_heads + h) * kHeadDim + d] = to_bits<T>(acc / lsum);
}

template <typename K>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const DecodeArgs& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <typename T, int G>
cudaError_t launch_split(const DecodeArgs& a, cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    auto kernel = decode_split_fma_kernel<T, G>;
    const size_t smem = FmaSmem<G>::kTotal;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    dim3 grid(a.max_splits, a.num_kv_heads, a.num_seqs);
    e = launch_pdl(kernel, grid, dim3(kThreads), smem, stream, a);
    if (e == cudaSuccess) note_launches(1);
    return e;
}

template <typename T>
cudaError_t split_for_group(const DecodeArgs& a, int group, cudaStream_t stream) {
    switch (group) {
        case 1: return launch_split<T, 1>(a, stream);
        case 2: return launch_split<T, 2>(a, stream);
        case 3: return launch_split<T, 3>(a, stream);
        case 4: return launch_split<T, 4>(a, stream);
        case 6: return launch_split<T, 6>(a, stream);
        case 8: return launch_split<T, 8>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool fma_supports_group(int group) {
    return group == 1 || group == 2 || group == 3 || group == 4 || group == 6 || group == 8;
}

cudaError_t launch_decode_split_fma(const DecodeArgs& a, int dtype, int group, cudaStream_t stream) {
    return dtype == PA_BF16 ? split_for_group<__nv_bfloat16>(a, group, stream)
                            : split_for_group<__half>(a, group, stream);
}

cudaError_t launch_decode_combine(const DecodeArgs& a, int dtype, cudaStream_t stream) {
    dim3 grid(a.num_q_heads, a.num_seqs);
    cudaError_t e = dtype == PA_BF16
                        ? launch_pdl(decode_combine_kernel<__nv_bfloat16>, grid, dim3(kHeadDim), 0, stream, a)
                        : launch_pdl(decode_combine_kernel<__half>, grid, dim3(kHeadDim), 0, stream, a);
    if (e == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace pa
