/*
 * oracle.c -- plain float64 CPU reference for the paged KV-cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no header, table or helper with the
 * CUDA code: every format decoder and every loop below is written out from
 * the definitions it cites.
 *
 * What it computes (sources, by page title and section):
 *  - Ultralytics glossary "PagedAttention", section "How paging works":
 *    a request's keys are scattered into a shared pool of fixed-size blocks
 *    (position pos goes to block_table[pos // block_size], offset
 *    pos % block_size) and the attention kernel reads them back block by
 *    block through the table.
 *  - OptiVerse "Paged KV cache", section "Block table and non-contiguous
 *    allocation": logical block i covers tokens [16 i, 16 i + 15]; the
 *    kernel looks the physical block up in the table for every block.
 *  - iThome "how to store the KV cache", section "Copy-on-Write": a
 *    diverging writer gets a new block holding a copy of the old contents.
 *  - Attention itself is the textbook decode step for one new query:
 *    s_j = scale * <q, k_j>, p = softmax(s), out = sum_j p_j v_j, with
 *    query head h reading KV head h / (Hq / Hkv) (grouped-query attention,
 *    Ultralytics glossary, section "Related techniques").
 *
 * Cache layout: k_cache, v_cache are [num_blocks][Hkv][block_size][D] with
 * elements of the cache type.  Queries are [B][Hq][D].
 *
 * Element types (codes): 0 = IEEE binary16, 1 = bfloat16, 2 = OCP FP8 E4M3
 * ("E4M3FN": bias 7, no infinities, S.1111.111 is NaN, largest finite 448).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F16 0
#define ORC_BF16 1
#define ORC_E4M3 2

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133); /* subnormal: f * 2^-7 * 2^-126 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + (double)f / 128.0, e - 127);
    }
    return sign ? -v : v;
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign, 4 exponent (bias 7),
 * 3 fraction bits; exponent field 15 is still a normal binade except for
 * fraction 7, which encodes NaN; there is no infinity. */
double oracle_e4m3_to_double(uint8_t x) {
    int sign = (x >> 7) & 1;
    int e = (x >> 3) & 0xf;
    int f = x & 0x7;
    double v;
    if (e == 15 && f == 7) {
        return NAN;
    } else if (e == 0) {
        v = ldexp((double)f, -9); /* subnormal: f * 2^-3 * 2^-6 */
    } else {
        v = ldexp(1.0 + (double)f / 8.0, e - 7);
    }
    return sign ? -v : v;
}

/* Encode a binary32 value as E4M3 with round-to-nearest, ties to an even
 * fraction, saturating to +-448 (values of larger magnitude and infinities
 * map to the largest finite code of their sign; NaN maps to the NaN code).
 * Written as a search over every finite code so that it can be checked by
 * eye: the nearest representable value wins; on a tie the code whose lowest
 * bit is 0 wins. */
uint8_t oracle_e4m3_from_float(float y) {
    if (isnan(y)) return 0x7f;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);
    int best = 0;
    double best_err = a; /* distance to +0 (code 0) */
    for (int c = 1; c <= 0x7e; ++c) {
        double err = fabs(oracle_e4m3_to_double((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

static double load_elem(const void* base, int dtype, size_t idx) {
    switch (dtype) {
        case ORC_F16: return oracle_f16_to_double(((const uint16_t*)base)[idx]);
        case ORC_BF16: return oracle_bf16_to_double(((const uint16_t*)base)[idx]);
        case ORC_E4M3: return oracle_e4m3_to_double(((const uint8_t*)base)[idx]);
        default: return NAN;
    }
}

static size_t elem_size(int dtype) { return dtype == ORC_E4M3 ? 1 : 2; }

/*
 * Paged decode attention, float64.
 *
 * For every sequence b (context length L = context_lens[b] tokens) and query
 * head h, gather the contiguous keys and values of KV head kvh = h / (Hq/Hkv)
 * through the block table (token j lives in physical block
 * block_tables[b][j / bs] at offset j % bs), dequantise (E4M3 elements are
 * multiplied by their per-tensor scale), and evaluate
 *     s_j   = scale * sum_d q[b][h][d] * K[j][d]
 *     p_j   = exp(s_j - max_i s_i) / sum_i exp(s_i - max_i s_i)
 *     out_d = sum_j p_j * V[j][d]
 * out is [B][Hq][D] float64.  Returns 0, or -1 on an argument that the
 * definition does not cover (L < 1 or beyond the table, a block id outside
 * the pool, Hq not a multiple of Hkv).
 */
int oracle_paged_decode(const void* q, int q_dtype,
                        const void* k_cache, const void* v_cache, int cache_dtype,
                        double k_scale, double v_scale,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens,
                        int B, int Hq, int Hkv, int bs, int D, int num_blocks,
                        double scale, double* out) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int L = context_lens[b];
        if (L < 1 || L > max_blocks_per_seq * bs) return -1;
        for (int j = 0; j < (L + bs - 1) / bs; ++j) {
            int blk = block_tables[(size_t)b * max_blocks_per_seq + j];
            if (blk < 0 || blk >= num_blocks) return -1;
        }
    }
    int status = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            int L = context_lens[b];
            int kvh = h / G;
            const int32_t* table = block_tables + (size_t)b * max_blocks_per_seq;
            double* s = (double*)malloc(sizeof(double) * (size_t)L);
            double* qv = (double*)malloc(sizeof(double) * (size_t)D);
            if (!s || !qv) {
                free(s);
                free(qv);
#pragma omp atomic write
                status = -2;
                continue;
            }
            for (int d = 0; d < D; ++d) qv[d] = load_elem(q, q_dtype, ((size_t)b * Hq + h) * D + d);
            double kmul = cache_dtype == ORC_E4M3 ? k_scale : 1.0;
            double vmul = cache_dtype == ORC_E4M3 ? v_scale : 1.0;
            double m = -INFINITY;
            for (int j = 0; j < L; ++j) {
                size_t row = (((size_t)table[j / bs] * Hkv + kvh) * bs + (j % bs)) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qv[d] * (load_elem(k_cache, cache_dtype, row + d) * kmul);
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            double z = 0.0;
            for (int j = 0; j < L; ++j) {
                s[j] = exp(s[j] - m);
                z += s[j];
            }
            double* o = out + ((size_t)b * Hq + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int j = 0; j < L; ++j) {
                size_t row = (((size_t)table[j / bs] * Hkv + kvh) * bs + (j % bs)) * D;
                double p = s[j] / z;
                for (int d = 0; d < D; ++d) o[d] += p * (load_elem(v_cache, cache_dtype, row + d) * vmul);
            }
            free(s);
            free(qv);
        }
    }
    return status;
}

/*
 * Slot-mapped KV append (Ultralytics glossary "PagedAttention", section
 * "How paging works": key_pool[table[pos // bs], pos % bs] = key; OptiVerse
 * "Paged KV cache": the 42nd token lands at position 10 of block 12).
 *
 * For each new token t and KV head h, the K and V vectors k[t][h][:],
 * v[t][h][:] (element type act_dtype) are written to slot
 * s = slot_mapping[t], i.e. block s / bs, offset s % bs.  A negative slot
 * means "no token" and is skipped.  When the cache type equals the
 * activation type the bytes are copied unchanged; for an E4M3 cache each
 * element x is stored as e4m3(x / scale), the division done in binary32
 * (float) arithmetic.  Returns 0, or -1 if a slot lies outside the pool.
 */
int oracle_append(const void* k, const void* v, int act_dtype,
                  const int64_t* slot_mapping, int T,
                  void* k_cache, void* v_cache, int cache_dtype,
                  int num_blocks, int Hkv, int bs, int D,
                  float k_scale, float v_scale) {
    size_t ae = elem_size(act_dtype);
    size_t ce = elem_size(cache_dtype);
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * bs) return -1;
        int64_t blk = slot / bs, off = slot % bs;
        for (int h = 0; h < Hkv; ++h) {
            size_t src = ((size_t)t * Hkv + h) * D;
            size_t dst = (((size_t)blk * Hkv + h) * bs + (size_t)off) * D;
            if (cache_dtype == act_dtype) {
                memcpy((char*)k_cache + dst * ce, (const char*)k + src * ae, (size_t)D * ae);
                memcpy((char*)v_cache + dst * ce, (const char*)v + src * ae, (size_t)D * ae);
            } else if (cache_dtype == ORC_E4M3) {
                for (int d = 0; d < D; ++d) {
                    float xk = (float)load_elem(k, act_dtype, src + d);
                    float xv = (float)load_elem(v, act_dtype, src + d);
                    float yk = xk / k_scale;
                    float yv = xv / v_scale;
                    ((uint8_t*)k_cache)[dst + d] = oracle_e4m3_from_float(yk);
                    ((uint8_t*)v_cache)[dst + d] = oracle_e4m3_from_float(yv);
                }
            } else {
                return -1;
            }
        }
    }
    return 0;
}

/*
 * Copy-on-write block copy (iThome "how to store the KV cache", section
 * "Copy-on-Write": the diverging branch gets a fresh block and the old
 * block's contents are copied into it).  For every pair (src, dst) the
 * whole physical block -- all KV heads, all slots, K and V -- is copied.
 * block_bytes is the size of one physical block of one of the two caches.
 * Returns 0, or -1 on a block id outside the pool.
 */
int oracle_block_copy(void* k_cache, void* v_cache, const int32_t* src_dst_pairs,
                      int num_pairs, int num_blocks, size_t block_bytes) {
    for (int i = 0; i < num_pairs; ++i) {
        int src = src_dst_pairs[2 * i], dst = src_dst_pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return -1;
        memmove((char*)k_cache + (size_t)dst * block_bytes, (char*)k_cache + (size_t)src * block_bytes, block_bytes);
        memmove((char*)v_cache + (size_t)dst * block_bytes, (char*)v_cache + (size_t)src * block_bytes, block_bytes);
    }
    return 0;
}

/* Preemption by swapping (the PagedAttention notes page, section on
 * preemption): the blocks of a preempted sequence are copied out of the pool
 * and later copied back into the blocks it is given.  Staging entry i holds
 * block ids[i] of the K cache, then the same block of the V cache.
 * direction 0: staging[i] = (K[ids[i]], V[ids[i]]); 1: the reverse. */
int oracle_block_swap(void* k_cache, void* v_cache, const int32_t* ids, int num_ids, int num_blocks,
                      size_t block_bytes, void* staging, int direction) {
    for (int i = 0; i < num_ids; ++i) {
        int b = ids[i];
        if (b < 0 || b >= num_blocks) return -1;
        char* st = (char*)staging + (size_t)i * 2 * block_bytes;
        char* kb = (char*)k_cache + (size_t)b * block_bytes;
        char* vb = (char*)v_cache + (size_t)b * block_bytes;
        if (direction == 0) {
            memcpy(st, kb, block_bytes);
            memcpy(st + block_bytes, vb, block_bytes);
        } else {
            memcpy(kb, st, block_bytes);
            memcpy(vb, st + block_bytes, block_bytes);
        }
    }
    return 0;
}

/* Number of OpenMP threads the attention oracle runs with. */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Decode n elements of the given type to float64 (E4M3 without scale). */
void oracle_decode_array(const void* src, int dtype, size_t n, double* out) {
    for (size_t i = 0; i < n; ++i) out[i] = load_elem(src, dtype, i);
}

/* Encode n binary32 values to E4M3 with oracle_e4m3_from_float. */
void oracle_e4m3_encode_array(const float* x, size_t n, uint8_t* out) {
    for (size_t i = 0; i < n; ++i) out[i] = oracle_e4m3_from_float(x[i]);
}

/*
 * QUEST query-aware block selection (Tencent Cloud "LLMs serving challenges",
 * section "Query-sparsity attention / QUEST"):
 *  1. for every block, the channel-wise minimum and maximum of its keys;
 *  2. for the query, an upper bound of q.k over the block's keys:
 *     U = sum_c max(q_c * min_c, q_c * max_c)  (a negative q_c pairs with the
 *     minimum, a positive one with the maximum);
 *  3. keep the K blocks with the largest bounds and attend only to them.
 * Readings: the keys are the stored (dequantised) cache values of the block's
 * filled slots; for grouped heads one selection serves the kv head, ranked by
 * the largest bound over its query heads; ties go to the lower logical block;
 * no block is forced in; with K >= the number of blocks every block is kept.
 * Output, per (sequence, kv head): the selected physical blocks in logical
 * order (sel_tables [B][Hkv][budget_blocks]) and their token count (sel_lens
 * [B][Hkv]: full blocks plus the filled part of the sequence's last block if
 * selected).  bounds [B][Hkv][max_blocks] (may be NULL) receives U.
 */
int oracle_quest_select(const void* q, int q_dtype, const void* k_cache, int cache_dtype, double k_scale,
                        const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                        int B, int Hq, int Hkv, int bs, int D, int num_blocks, int budget_blocks,
                        int32_t* sel_tables, int32_t* sel_lens, double* bounds) {
    if (Hkv <= 0 || Hq % Hkv != 0 || budget_blocks < 1) return -1;
    int G = Hq / Hkv;
    double kmul = cache_dtype == ORC_E4M3 ? k_scale : 1.0;
    for (int b = 0; b < B; ++b) {
        int L = context_lens[b];
        if (L < 1 || L > max_blocks_per_seq * bs) return -1;
        int nblk = (L + bs - 1) / bs;
        const int32_t* table = block_tables + (size_t)b * max_blocks_per_seq;
        for (int j = 0; j < nblk; ++j)
            if (table[j] < 0 || table[j] >= num_blocks) return -1;
        for (int kvh = 0; kvh < Hkv; ++kvh) {
            double* U = (double*)malloc(sizeof(double) * (size_t)nblk);
            char* taken = (char*)calloc((size_t)nblk, 1);
            double* mn = (double*)malloc(sizeof(double) * (size_t)D);
            double* mx = (double*)malloc(sizeof(double) * (size_t)D);
            if (!U || !taken || !mn || !mx) {
                free(U); free(taken); free(mn); free(mx);
                return -2;
            }
            for (int j = 0; j < nblk; ++j) {
                int filled = (j == nblk - 1) ? L - j * bs : bs;
                for (int d = 0; d < D; ++d) {
                    mn[d] = INFINITY;
                    mx[d] = -INFINITY;
                }
                for (int t = 0; t < filled; ++t) {
                    size_t row = (((size_t)table[j] * Hkv + kvh) * bs + t) * D;
                    for (int d = 0; d < D; ++d) {
                        double x = load_elem(k_cache, cache_dtype, row + d) * kmul;
                        if (x < mn[d]) mn[d] = x;
                        if (x > mx[d]) mx[d] = x;
                    }
                }
                double best = -INFINITY;
                for (int g = 0; g < G; ++g) {
                    double u = 0.0;
                    for (int d = 0; d < D; ++d) {
                        double qd = load_elem(q, q_dtype, ((size_t)b * Hq + kvh * G + g) * D + d);
                        double a = qd * mn[d], c = qd * mx[d];
                        u += a > c ? a : c;
                    }
                    if (u > best) best = u;
                }
                U[j] = best;
                if (bounds) bounds[((size_t)b * Hkv + kvh) * max_blocks_per_seq + j] = best;
            }
            int keep = nblk < budget_blocks ? nblk : budget_blocks;
            for (int r = 0; r < keep; ++r) {  /* repeated arg-max; the first maximum wins ties */
                int arg = -1;
                for (int j = 0; j < nblk; ++j)
                    if (!taken[j] && (arg < 0 || U[j] > U[arg])) arg = j;
                taken[arg] = 1;
            }
            int32_t* out_row = sel_tables + ((size_t)b * Hkv + kvh) * budget_blocks;
            int n = 0, tokens = 0;
            for (int j = 0; j < nblk; ++j) {
                if (!taken[j]) continue;
                out_row[n++] = table[j];
                tokens += (j == nblk - 1) ? L - j * bs : bs;
            }
            for (int i = n; i < budget_blocks; ++i) out_row[i] = 0;
            sel_lens[(size_t)b * Hkv + kvh] = tokens;
            free(U); free(taken); free(mn); free(mx);
        }
    }
    return 0;
}

/*
 * Attention over per-(sequence, kv head) block lists: the same definition as
 * oracle_paged_decode, with the keys and values of kv head kvh of sequence b
 * gathered through tables[b][kvh][.] over lens[b][kvh] tokens.
 */
int oracle_sparse_decode(const void* q, int q_dtype, const void* k_cache, const void* v_cache, int cache_dtype,
                         double k_scale, double v_scale, const int32_t* tables, int max_blocks, const int32_t* lens,
                         int B, int Hq, int Hkv, int bs, int D, int num_blocks, double scale, double* out) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    int G = Hq / Hkv;
    double kmul = cache_dtype == ORC_E4M3 ? k_scale : 1.0;
    double vmul = cache_dtype == ORC_E4M3 ? v_scale : 1.0;
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            int kvh = h / G;
            int L = lens[(size_t)b * Hkv + kvh];
            const int32_t* table = tables + ((size_t)b * Hkv + kvh) * max_blocks;
            if (L < 1 || L > max_blocks * bs) return -1;
            double* s = (double*)malloc(sizeof(double) * (size_t)L);
            if (!s) return -2;
            double m = -INFINITY;
            for (int j = 0; j < L; ++j) {
                int blk = table[j / bs];
                if (blk < 0 || blk >= num_blocks) {
                    free(s);
                    return -1;
                }
                size_t row = (((size_t)blk * Hkv + kvh) * bs + (j % bs)) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += load_elem(q, q_dtype, ((size_t)b * Hq + h) * D + d) *
                           (load_elem(k_cache, cache_dtype, row + d) * kmul);
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            double z = 0.0;
            for (int j = 0; j < L; ++j) {
                s[j] = exp(s[j] - m);
                z += s[j];
            }
            double* o = out + ((size_t)b * Hq + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int j = 0; j < L; ++j) {
                size_t row = (((size_t)table[j / bs] * Hkv + kvh) * bs + (j % bs)) * D;
                double p = s[j] / z;
                for (int d = 0; d < D; ++d) o[d] += p * (load_elem(v_cache, cache_dtype, row + d) * vmul);
            }
            free(s);
        }
    }
    return 0;
}

/* QUEST metadata alone: channel-wise minimum and maximum of the keys of each
 * (sequence, logical block, kv head) over the block's filled slots, float64
 * [B][max_blocks][Hkv][D] (entries of blocks past the context are NaN). */
int oracle_quest_block_minmax(const void* k_cache, int cache_dtype, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* context_lens, int B, int Hkv, int bs, int D,
                              int num_blocks, double* out_min, double* out_max) {
    for (int b = 0; b < B; ++b) {
        int L = context_lens[b];
        if (L < 1 || L > max_blocks_per_seq * bs) return -1;
        for (int j = 0; j < max_blocks_per_seq; ++j) {
            for (int h = 0; h < Hkv; ++h) {
                double* mn = out_min + (((size_t)b * max_blocks_per_seq + j) * Hkv + h) * D;
                double* mx = out_max + (((size_t)b * max_blocks_per_seq + j) * Hkv + h) * D;
                if (j * bs >= L) {
                    for (int d = 0; d < D; ++d) mn[d] = mx[d] = NAN;
                    continue;
                }
                int blk = block_tables[(size_t)b * max_blocks_per_seq + j];
                if (blk < 0 || blk >= num_blocks) return -1;
                int filled = L - j * bs < bs ? L - j * bs : bs;
                for (int d = 0; d < D; ++d) {
                    mn[d] = INFINITY;
                    mx[d] = -INFINITY;
                }
                for (int t = 0; t < filled; ++t) {
                    size_t row = (((size_t)blk * Hkv + h) * bs + t) * D;
                    for (int d = 0; d < D; ++d) {
                        double x = load_elem(k_cache, cache_dtype, row + d);
                        if (x < mn[d]) mn[d] = x;
                        if (x > mx[d]) mx[d] = x;
                    }
                }
            }
        }
    }
    return 0;
}
