/*
 * pa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct fp64 CPU statement of what the paged KV
 * cache write and paged decode attention compute.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg load this file's library.
 * It shares no code, header, table or helper with the CUDA library; it is
 * compiled by the host C compiler alone.
 *
 * What it follows:
 *   [A] "端侧 SLM 显存保活术：在 4GB 内存板卡上实现轻量 PagedAttention 与 KV 缓存分块",
 *       section "注意力寻址：非连续物理块的间接寻址内核": a token t lives in logical
 *       block t / B at offset t % B; the physical block is block_table[t / B].
 *       Section "KV Cache 的物理膨胀账本": bytes of K and V per token per layer =
 *       2 x kv_heads x head_dim x bytes per element.
 *   [B] "显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结",
 *       section 三 (sequence diagram of the decode loop): the new token is written at
 *       the next offset of the sequence's last block, or at offset 0 of a freshly
 *       appended block when the last one is full; then attention runs.
 *       Section 四: a sequence about to write into a shared, unfilled block first gets a
 *       deep copy of that block in a fresh one.  FAQ on preemption: a request's blocks move
 *       to host memory and back (the same whole-block copy between two pools).
 *       Section 五.1 (kernel sketch): per (sequence, head) loop over the logical
 *       blocks, look up the physical block, take q.k for every cached token,
 *       softmax, weight V, normalise at the end.
 *
 * Readings where the pages are silent (each one listed in the design notes):
 *   - context_lens[s] counts the new token; decode attends over all of them.
 *   - Query head h reads kv head h / (num_q_heads / num_kv_heads) (contiguous GQA groups).
 *   - Pools are [num_blocks][num_kv_heads][block_size][head_dim]; one (block, kv-head)
 *     tile is contiguous.
 *   - A negative slot means "skip this row"; a zero-length context gives a zero output.
 *
 * Decode is the plain definition: gather the cached rows through the block table
 * into contiguous fp64 K and V, then out = softmax(scale * q K^T) V, with the
 * maximum subtracted before exp and the sum divided at the end.
 *
 * PAO_MUTANT (compile-time, tests only) plants one known mistake so that the test
 * suite can show each of its pins notices it; ordinary builds leave it undefined.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef PAO_MUTANT
#define PAO_MUTANT 0
#endif

/* ---- element decoding: IEEE 754 binary16, and bfloat16 (upper half of binary32) ---- */

double pao_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);                /* subnormal: m * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25);    /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

double pao_bf16_to_f64(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int m = b & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -133);               /* subnormal: m * 2^-126 * 2^-7 */
    } else if (e == 255) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + m), e - 134);    /* (1 + m/128) * 2^(e-127) */
    }
    return sign ? -v : v;
}

static double elem(const uint16_t* p, int is_bf16) {
    return is_bf16 ? pao_bf16_to_f64(*p) : pao_f16_to_f64(*p);
}

void pao_decode_elems(const uint16_t* src, int64_t n, int is_bf16, double* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = elem(src + i, is_bf16);
}

/* ---- [A] byte ledger ---- */

int64_t pao_kv_bytes_per_token(int num_kv_heads, int head_dim, int elem_bytes) {
    return (int64_t)2 * num_kv_heads * head_dim * elem_bytes;   /* K and V */
}

/* ---- [A] address of a token: (physical block, offset) and the flat slot ---- */

void pao_locate(const int32_t* table_row, int64_t t, int block_size, int32_t* phys, int32_t* off) {
    int64_t logical = t / block_size;
#if PAO_MUTANT == 3
    *off = (int32_t)((t + 1) % block_size);                     /* planted: wrong offset */
#else
    *off = (int32_t)(t % block_size);
#endif
    *phys = table_row[logical];
}

int64_t pao_slot_of_token(const int32_t* table_row, int64_t t, int block_size) {
    int32_t phys, off;
    pao_locate(table_row, t, block_size, &phys, &off);
    return (int64_t)phys * block_size + off;
}

/* [B] the new token is the last of context_lens[s]; an empty context writes nothing. */
void pao_slot_mapping(const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                      int num_seqs, int block_size, int64_t* slots) {
    for (int s = 0; s < num_seqs; ++s) {
        int32_t L = context_lens[s];
#if PAO_MUTANT == 6
        int64_t last = L;                                        /* planted: one past the new token */
#else
        int64_t last = (int64_t)L - 1;
#endif
        slots[s] = (L > 0) ? pao_slot_of_token(block_tables + (int64_t)s * max_blocks, last, block_size)
                           : -1;
    }
}

/* ---- [B] cache write: a byte copy of each (token, kv-head) row into its slot ---- */

void pao_cache_write(const uint16_t* k, const uint16_t* v, const int64_t* slots,
                     uint16_t* k_cache, uint16_t* v_cache,
                     int num_tokens, int num_kv_heads, int head_dim, int block_size) {
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slots[i];
        if (slot < 0) continue;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
#if PAO_MUTANT == 7
            int64_t dst = ((blk * block_size + off) * num_kv_heads + h) * head_dim; /* planted: [NB][B][H][D] */
#else
            int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim;
#endif
            int64_t src = ((int64_t)i * num_kv_heads + h) * head_dim;
            memcpy(k_cache + dst, k + src, sizeof(uint16_t) * (size_t)head_dim);
            memcpy(v_cache + dst, v + src, sizeof(uint16_t) * (size_t)head_dim);
        }
    }
}

/* ---- [B] section 四: copy-on-write deep copy of whole physical blocks; its FAQ on
 * preemption: the same copy moves a request's blocks to a host pool and back ---- */

/* For each pair i in order, every kv head's rows of block src_ids[i] of (src_k, src_v) are
 * copied to block dst_ids[i] of (dst_k, dst_v).  A pair with an id outside its pool is left
 * out.  Returns the number of pairs left out. */
int pao_copy_blocks(const uint16_t* src_k, const uint16_t* src_v, int src_blocks,
                    uint16_t* dst_k, uint16_t* dst_v, int dst_blocks,
                    const int32_t* src_ids, const int32_t* dst_ids, int num_pairs,
                    int num_kv_heads, int block_size, int head_dim) {
    const int64_t per_block = (int64_t)num_kv_heads * block_size * head_dim;   /* elements */
#if PAO_MUTANT == 8
    const int64_t copied = (int64_t)block_size * head_dim;                      /* planted: kv head 0 only */
#else
    const int64_t copied = per_block;
#endif
    int left_out = 0;
    for (int i = 0; i < num_pairs; ++i) {
        const int32_t s = src_ids[i], d = dst_ids[i];
        if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
            ++left_out;
            continue;
        }
        memcpy(dst_k + d * per_block, src_k + s * per_block, sizeof(uint16_t) * (size_t)copied);
        memcpy(dst_v + d * per_block, src_v + s * per_block, sizeof(uint16_t) * (size_t)copied);
    }
    return left_out;
}

/* ---- [B] decode attention over the paged cache, fp64 ---- */

/* Gather the L cached rows of (sequence, kv head hk) into contiguous fp64 arrays. */
static void gather(const uint16_t* cache, const int32_t* table_row, int L, int hk,
                   int num_kv_heads, int head_dim, int block_size, int is_bf16, double* dst) {
    for (int t = 0; t < L; ++t) {
        int32_t phys, off;
        pao_locate(table_row, t, block_size, &phys, &off);
        const uint16_t* row = cache + (((int64_t)phys * num_kv_heads + hk) * block_size + off) * head_dim;
        for (int d = 0; d < head_dim; ++d) dst[(int64_t)t * head_dim + d] = elem(row + d, is_bf16);
    }
}

/* out[s][h][:] = sum_t p_t V[t][:],  p = softmax_t(scale * q[s][h] . K[t]).
 * Returns 0, or -1 when the arguments cannot describe a valid problem. */
int pao_decode(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
               const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
               double scale, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
               int block_size, int is_bf16, int num_threads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0)
        return -1;
    const int G = num_q_heads / num_kv_heads;
    const int64_t pairs = (int64_t)num_seqs * num_kv_heads;
    int bad = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(| : bad)
#endif
    for (int64_t pr = 0; pr < pairs; ++pr) {
        const int s = (int)(pr / num_kv_heads);
        const int hk = (int)(pr % num_kv_heads);
        const int L = context_lens[s];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks * block_size) { bad = 1; continue; }
        const int32_t* row = block_tables + (int64_t)s * max_blocks;
        double* K = (double*)malloc(sizeof(double) * ((size_t)L * head_dim + 1));
        double* V = (double*)malloc(sizeof(double) * ((size_t)L * head_dim + 1));
        double* z = (double*)malloc(sizeof(double) * ((size_t)L + 1));
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        gather(k_cache, row, L, hk, num_kv_heads, head_dim, block_size, is_bf16, K);
        gather(v_cache, row, L, hk, num_kv_heads, head_dim, block_size, is_bf16, V);
        for (int g = 0; g < G; ++g) {
#if PAO_MUTANT == 1
            const int h = g * num_kv_heads + hk;                 /* planted: strided GQA groups */
#else
            const int h = hk * G + g;
#endif
            double* o = out + ((int64_t)s * num_q_heads + h) * head_dim;
            const uint16_t* qr = q + ((int64_t)s * num_q_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) qv[d] = elem(qr + d, is_bf16);
            if (L == 0) {
                for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
                continue;
            }
            double zmax = -INFINITY;
            for (int t = 0; t < L; ++t) {
                double acc = 0.0;
                for (int d = 0; d < head_dim; ++d) acc += qv[d] * K[(int64_t)t * head_dim + d];
#if PAO_MUTANT == 2
                z[t] = acc;                                      /* planted: scale dropped */
#else
                z[t] = scale * acc;
#endif
                if (z[t] > zmax) zmax = z[t];
            }
            double denom = 0.0;
            for (int t = 0; t < L; ++t) {
                z[t] = exp(z[t] - zmax);
                denom += z[t];
            }
            for (int d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int t = 0; t < L; ++t) {
#if PAO_MUTANT == 4
                    acc += z[t] * K[(int64_t)t * head_dim + d];  /* planted: K in place of V */
#else
                    acc += z[t] * V[(int64_t)t * head_dim + d];
#endif
                }
#if PAO_MUTANT == 5
                o[d] = acc;                                      /* planted: no normalisation */
#else
                o[d] = acc / denom;
#endif
            }
        }
        free(K); free(V); free(z); free(qv);
    }
    return bad ? -1 : 0;
}

/* ---- several new query tokens per sequence (chunked prefill, speculative verification) ----
 * Sequence s owns query rows query_start[s] .. query_start[s+1]-1: its n_s newest tokens,
 * which are the last n_s of its context_lens[s] = L_s cached tokens.  Query token i sits at
 * position L_s - n_s + i and attends causally, over the cached tokens t = 0 .. L_s - n_s + i.
 * With n_s = 1 this is pao_decode.  q, out: [num_q_tokens][num_q_heads][head_dim].
 * Returns 0, or -1 when the arguments cannot describe a valid problem (n_s < 0 or > L_s). */
int pao_multi_query(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                    const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                    const int32_t* query_start, double scale, int num_seqs, int num_q_heads,
                    int num_kv_heads, int head_dim, int block_size, int is_bf16, int num_threads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0)
        return -1;
    const int G = num_q_heads / num_kv_heads;
    const int64_t pairs = (int64_t)num_seqs * num_kv_heads;
    int bad = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(| : bad)
#endif
    for (int64_t pr = 0; pr < pairs; ++pr) {
        const int s = (int)(pr / num_kv_heads);
        const int hk = (int)(pr % num_kv_heads);
        const int L = context_lens[s];
        const int n = query_start[s + 1] - query_start[s];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks * block_size || n < 0 || n > L) { bad = 1; continue; }
        const int32_t* row = block_tables + (int64_t)s * max_blocks;
        double* K = (double*)malloc(sizeof(double) * ((size_t)L * head_dim + 1));
        double* V = (double*)malloc(sizeof(double) * ((size_t)L * head_dim + 1));
        double* z = (double*)malloc(sizeof(double) * ((size_t)L + 1));
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        gather(k_cache, row, L, hk, num_kv_heads, head_dim, block_size, is_bf16, K);
        gather(v_cache, row, L, hk, num_kv_heads, head_dim, block_size, is_bf16, V);
        for (int i = 0; i < n; ++i) {
#if PAO_MUTANT == 9
            const int last = L - n + i - 1;                      /* planted: a query misses itself */
#else
            const int last = L - n + i;                          /* newest position query i sees */
#endif
            const int64_t qrow = query_start[s] + i;
            for (int g = 0; g < G; ++g) {
                const int h = hk * G + g;
                double* o = out + (qrow * num_q_heads + h) * head_dim;
                const uint16_t* qr = q + (qrow * num_q_heads + h) * head_dim;
                for (int d = 0; d < head_dim; ++d) qv[d] = elem(qr + d, is_bf16);
                double zmax = -INFINITY;
                for (int t = 0; t <= last; ++t) {
                    double acc = 0.0;
                    for (int d = 0; d < head_dim; ++d) acc += qv[d] * K[(int64_t)t * head_dim + d];
                    z[t] = scale * acc;
                    if (z[t] > zmax) zmax = z[t];
                }
                double denom = 0.0;
                for (int t = 0; t <= last; ++t) {
                    z[t] = exp(z[t] - zmax);
                    denom += z[t];
                }
                for (int d = 0; d < head_dim; ++d) {
                    double acc = 0.0;
                    for (int t = 0; t <= last; ++t) acc += z[t] * V[(int64_t)t * head_dim + d];
                    o[d] = (last >= 0) ? acc / denom : 0.0;
                }
            }
        }
        free(K); free(V); free(z); free(qv);
    }
    return bad ? -1 : 0;
}

/* ---- slotted blocks (the radix-tree fragmentation page, "Slotted Block 分槽与微块共享架构"):
 * a sequence's context is a list of runs (block_id, slot_offset, length), read in order;
 * token t of the sequence is row slot_offset + (t - run start) of block block_id. ---- */

/* Gather the cached rows of (sequence, kv head hk) given by runs[r0 .. r1) into contiguous fp64
 * rows; returns the number of rows, or -1 if a run leaves its block or the pool. */
static int gather_runs(const uint16_t* cache, const int32_t* runs, int r0, int r1, int hk, int num_kv_heads,
                       int head_dim, int block_size, int num_blocks, int is_bf16, double* dst) {
    int t = 0;
    for (int r = r0; r < r1; ++r) {
        const int32_t blk = runs[3 * r], off = runs[3 * r + 1], len = runs[3 * r + 2];
        if (blk < 0 || blk >= num_blocks || off < 0 || len < 0 || off + len > block_size) return -1;
        for (int k = 0; k < len; ++k, ++t) {
#if PAO_MUTANT == 10
            const int64_t row = ((int64_t)blk * num_kv_heads + hk) * block_size + k;          /* planted: offset dropped */
#else
            const int64_t row = ((int64_t)blk * num_kv_heads + hk) * block_size + off + k;
#endif
            if (dst)
                for (int d = 0; d < head_dim; ++d) dst[(int64_t)t * head_dim + d] = elem(cache + row * head_dim + d, is_bf16);
        }
    }
    return t;
}

/* One query token per sequence over a context given by runs: sequence s owns runs
 * seq_runs[s] .. seq_runs[s+1]-1; its length is the sum of their lengths.  out as pao_decode. */
int pao_decode_runs(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                    const int32_t* runs, const int32_t* seq_runs, double scale, int num_seqs, int num_q_heads,
                    int num_kv_heads, int head_dim, int block_size, int num_blocks, int is_bf16, int num_threads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0) return -1;
    const int G = num_q_heads / num_kv_heads;
    const int64_t pairs = (int64_t)num_seqs * num_kv_heads;
    int bad = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(| : bad)
#endif
    for (int64_t pr = 0; pr < pairs; ++pr) {
        const int s = (int)(pr / num_kv_heads);
        const int hk = (int)(pr % num_kv_heads);
        const int L = gather_runs(k_cache, runs, seq_runs[s], seq_runs[s + 1], hk, num_kv_heads, head_dim,
                                  block_size, num_blocks, is_bf16, NULL);
        if (L < 0) { bad = 1; continue; }
        double* K = (double*)malloc(sizeof(double) * ((size_t)L * head_dim + 1));
        double* V = (double*)malloc(sizeof(double) * ((size_t)L * head_dim + 1));
        double* z = (double*)malloc(sizeof(double) * ((size_t)L + 1));
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        gather_runs(k_cache, runs, seq_runs[s], seq_runs[s + 1], hk, num_kv_heads, head_dim, block_size, num_blocks,
                    is_bf16, K);
        gather_runs(v_cache, runs, seq_runs[s], seq_runs[s + 1], hk, num_kv_heads, head_dim, block_size, num_blocks,
                    is_bf16, V);
        for (int g = 0; g < G; ++g) {
            const int h = hk * G + g;
            double* o = out + ((int64_t)s * num_q_heads + h) * head_dim;
            const uint16_t* qr = q + ((int64_t)s * num_q_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) qv[d] = elem(qr + d, is_bf16);
            double zmax = -INFINITY;
            for (int t = 0; t < L; ++t) {
                double acc = 0.0;
                for (int d = 0; d < head_dim; ++d) acc += qv[d] * K[(int64_t)t * head_dim + d];
                z[t] = scale * acc;
                if (z[t] > zmax) zmax = z[t];
            }
            double denom = 0.0;
            for (int t = 0; t < L; ++t) {
                z[t] = exp(z[t] - zmax);
                denom += z[t];
            }
            for (int d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int t = 0; t < L; ++t) acc += z[t] * V[(int64_t)t * head_dim + d];
                o[d] = (L > 0) ? acc / denom : 0.0;
            }
        }
        free(K); free(V); free(z); free(qv);
    }
    return bad ? -1 : 0;
}

/* Online defragmentation (same page): move runs of rows.  moves[m] = (src_block, src_off,
 * length, dst_block, dst_off); every kv head's rows src_off .. src_off+length-1 of src_block
 * are copied to dst_off .. of dst_block, moves applied in order.  A move leaving a block or a
 * pool is left out; returns how many were. */
int pao_gather_runs(const uint16_t* src_k, const uint16_t* src_v, int src_blocks, uint16_t* dst_k, uint16_t* dst_v,
                    int dst_blocks, const int32_t* moves, int num_moves, int num_kv_heads, int block_size,
                    int head_dim) {
    int left_out = 0;
    for (int m = 0; m < num_moves; ++m) {
        const int32_t sb = moves[5 * m], so = moves[5 * m + 1], len = moves[5 * m + 2];
        const int32_t db = moves[5 * m + 3], dof = moves[5 * m + 4];
        if (sb < 0 || sb >= src_blocks || db < 0 || db >= dst_blocks || len < 0 || so < 0 || dof < 0 ||
            so + len > block_size || dof + len > block_size) {
            ++left_out;
            continue;
        }
        for (int h = 0; h < num_kv_heads; ++h) {
            const int64_t s_row = ((int64_t)sb * num_kv_heads + h) * block_size + so;
            const int64_t d_row = ((int64_t)db * num_kv_heads + h) * block_size + dof;
            memmove(dst_k + d_row * head_dim, src_k + s_row * head_dim, sizeof(uint16_t) * (size_t)len * head_dim);
            memmove(dst_v + d_row * head_dim, src_v + s_row * head_dim, sizeof(uint16_t) * (size_t)len * head_dim);
        }
    }
    return left_out;
}

int pao_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
