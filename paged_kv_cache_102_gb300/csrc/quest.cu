// QUEST query-aware block selection (Tencent Cloud "LLMs serving
// challenges", section "Query-sparsity attention / QUEST"): per block the
// channel-wise minimum and maximum of its keys; for a query, the upper bound
//     U = sum_c max(q_c * min_c, q_c * max_c)
// of q.k over the block's keys; attention then reads only the K blocks with
// the largest bounds.
//
// Metadata layout: kmeta [num_blocks][Hkv][2][D] in the cache's 16-bit type
// (row 0 = min, row 1 = max over the block's filled slots; min and max of
// 16-bit values are themselves exact 16-bit values).
#include <cfloat>

#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

namespace {

template <int T>
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
    Vec16<T>::to_float(u, f);
}

template <int T>
__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 u;
    uint16_t* e = reinterpret_cast<uint16_t*>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = float_to_act<T>(f[i]);  // exact: f holds 16-bit values
    return u;
}

}  // namespace

// Full recompute: one thread per (sequence, logical block, kv head, 8-channel
// chunk) over the block's filled slots.
template <int T>
__global__ void __launch_bounds__(256) quest_minmax_kernel(QuestMetaParams p) {
    const int chunks = p.head_dim / 8;
    const int64_t per_seq = static_cast<int64_t>(p.max_blocks_per_seq) * p.num_kv_heads * chunks;
    const int64_t total = per_seq * p.num_seqs;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int seq = static_cast<int>(i / per_seq);
        int64_t r = i % per_seq;
        const int j = static_cast<int>(r / (p.num_kv_heads * chunks));
        r %= p.num_kv_heads * chunks;
        const int kvh = static_cast<int>(r / chunks);
        const int c = static_cast<int>(r % chunks);
        const int L = p.context_lens[seq];
        if (L < 1 || L > p.max_blocks_per_seq * p.block_size) {
            if (j == 0 && kvh == 0 && c == 0) atomicOr(p.err, kErrBadLen);
            continue;
        }
        if (j * p.block_size >= L) continue;
        const int blk = p.block_tables[static_cast<int64_t>(seq) * p.max_blocks_per_seq + j];
        if (blk < 0 || blk >= p.num_blocks) {
            atomicOr(p.err, kErrBadBlock);
            continue;
        }
        const int filled = min(p.block_size, L - j * p.block_size);
        float mn[8], mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            mn[e] = FLT_MAX;
            mx[e] = -FLT_MAX;
        }
        const uint16_t* base = static_cast<const uint16_t*>(p.k_cache) +
                               ((static_cast<int64_t>(blk) * p.num_kv_heads + kvh) * p.block_size) * p.head_dim +
                               c * 8;
        for (int t = 0; t < filled; ++t) {
            float f[8];
            unpack8<T>(*reinterpret_cast<const uint4*>(base + static_cast<int64_t>(t) * p.head_dim), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                mn[e] = fminf(mn[e], f[e]);
                mx[e] = fmaxf(mx[e], f[e]);
            }
        }
        uint16_t* meta = static_cast<uint16_t*>(p.kmeta) + ((static_cast<int64_t>(blk) * p.num_kv_heads + kvh) * 2) * p.head_dim;
        *reinterpret_cast<uint4*>(meta + c * 8) = pack8<T>(mn);
        *reinterpret_cast<uint4*>(meta + p.head_dim + c * 8) = pack8<T>(mx);
    }
}

// Incremental update with newly appended keys: the first slot of a block
// starts its metadata, later slots widen it.  At most one new token per block
// per call (as one decode step gives).
template <int T>
__global__ void __launch_bounds__(256) quest_append_minmax_kernel(QuestAppendParams p) {
    const int chunks = p.head_dim / 8;
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * chunks;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i % chunks);
        const int64_t th = i / chunks;
        const int kvh = static_cast<int>(th % p.num_kv_heads);
        const int64_t t = th / p.num_kv_heads;
        const int64_t slot = p.slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= static_cast<int64_t>(p.num_blocks) * p.block_size) {
            atomicOr(p.err, kErrBadSlot);
            continue;
        }
        const int64_t blk = slot / p.block_size;
        const bool first = slot % p.block_size == 0;
        float k[8];
        unpack8<T>(*reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k_new) + th * p.head_dim + c * 8), k);
        uint16_t* meta = static_cast<uint16_t*>(p.kmeta) + ((blk * p.num_kv_heads + kvh) * 2) * p.head_dim + c * 8;
        float mn[8], mx[8];
        if (first) {
#pragma unroll
            for (int e = 0; e < 8; ++e) mn[e] = mx[e] = k[e];
        } else {
            unpack8<T>(*reinterpret_cast<const uint4*>(meta), mn);
            unpack8<T>(*reinterpret_cast<const uint4*>(meta + p.head_dim), mx);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                mn[e] = fminf(mn[e], k[e]);
                mx[e] = fmaxf(mx[e], k[e]);
            }
        }
        *reinterpret_cast<uint4*>(meta) = pack8<T>(mn);
        *reinterpret_cast<uint4*>(meta + p.head_dim) = pack8<T>(mx);
    }
}

// Packed float pairs (Blackwell's two-wide fp32 FMA).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float f2_sum(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Two 16-bit elements (one 32-bit word) -> a packed float pair.
template <int T>
__device__ __forceinline__ uint64_t word_to_pair(uint32_t w) {
    if constexpr (T == kBF16) {
        return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w));
        return f2_pack(t.x, t.y);
    }
}

// N (4 or 8) 16-bit elements at a 2N-byte aligned address -> N/2 float pairs.
template <int T, int N>
__device__ __forceinline__ void load_pairs(const void* src, uint64_t* f2) {
    if constexpr (N == 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(src);
        f2[0] = word_to_pair<T>(u.x);
        f2[1] = word_to_pair<T>(u.y);
        f2[2] = word_to_pair<T>(u.z);
        f2[3] = word_to_pair<T>(u.w);
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(src);
        f2[0] = word_to_pair<T>(u.x);
        f2[1] = word_to_pair<T>(u.y);
    }
}

// Sum v[0..N) over the lanes of an aligned group of LPB lanes, leaving lane l
// with the sum of one value: at each halving step a lane keeps the half of
// the values picked by its lane bit and receives its partner's copy of that
// half, so N values need log2(N) exchanges of shrinking width before the
// plain butterfly finishes the sum.  Afterwards lanes that differ only in the
// bits LPB/2, LPB/4, ... (the first log2(N) of them) hold different values.
template <int N, int OFF>
struct SplitSum {
    __device__ __forceinline__ static float run(float* v, int lane) {
        if constexpr (OFF == 0) {
            return v[0];
        } else if constexpr (N == 1) {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
            return SplitSum<1, OFF / 2>::run(v, lane);
        } else {
            const bool upper = lane & OFF;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float send = upper ? v[i] : v[i + N / 2];
                const float keep = upper ? v[i + N / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
            }
            return SplitSum<N / 2, OFF / 2>::run(v, lane);
        }
    }
};

// Selection, step 1: the bound of every (sequence, kv head, logical block).
// For channel c the larger of q*min and q*max is q+ * max + q- * min, with q+
// and q- the positive and negative parts of q, so a bound is two fused
// multiply-adds per channel and head.
//
// Persistent CTAs walk a contiguous range of items; an item is 32 logical
// blocks of one (sequence, kv head) row, items ordered (sequence, kv head,
// chunk) so a CTA mostly stays on one row and keeps its query registers.
// Warp 0 reads the item's block ids and bulk-copies each block's min and max
// rows (4*D contiguous bytes) into a ring of shared-memory stages; warps 1..4
// compute from shared memory, D/8 lanes per block (D/4 for a group of 8),
// lane c holding q+ and q- of its 8 (or 4) channels of the group's query
// heads.  Bounds go to the workspace
// [B][Hkv][max_blocks] (-inf past the context).
constexpr int kBItem = 32;
constexpr int kBConsumerWarps = 4;
constexpr int kBThreads = 32 * (1 + kBConsumerWarps);

template <int D>
struct BoundsCfg {
    static constexpr int kSlotBytes = 4 * D;  // min row then max row
    static constexpr int kStageBytes = kBItem * kSlotBytes;
    static constexpr int kStages = 65536 / kStageBytes < 4 ? 4 : (65536 / kStageBytes > 8 ? 8 : 65536 / kStageBytes);
    static constexpr int kSmem = kStages * kStageBytes;
};

template <int T, int D, int G>
__global__ void __launch_bounds__(kBThreads, 3) quest_bounds_kernel(QuestSelectParams p, int64_t num_items) {
    using Cfg = BoundsCfg<D>;
    constexpr int S = Cfg::kStages;
    constexpr int CPL = G >= 8 ? 4 : 8;                    // channels per lane
    constexpr int LPB = D / CPL;                           // lanes per block
    constexpr int PER_PASS = 32 * kBConsumerWarps / LPB;   // blocks per consumer pass
    static_assert(G <= LPB, "the split sum leaves one head per lane");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full_bar[S], empty_bar[S];
    __shared__ unsigned valid_mask[S];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunks = (p.max_blocks_per_seq + kBItem - 1) / kBItem;
    const int64_t begin = num_items * blockIdx.x / gridDim.x;
    const int64_t end = num_items * (blockIdx.x + 1) / gridDim.x;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], kBConsumerWarps);
        }
        abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    auto item_coords = [&](int64_t it, int& seq, int& kvh, int& j0) {
        j0 = static_cast<int>(it % chunks) * kBItem;
        const int64_t r = it / chunks;
        kvh = static_cast<int>(r % p.num_kv_heads);
        seq = static_cast<int>(r / p.num_kv_heads);
    };
    if (warp == 0) {
        // Block ids (and context lengths) are fetched S items ahead, one
        // register slot per stage, so the table reads overlap the copies.
        const uint64_t policy = l2_policy_evict_first();
        auto fetch = [&](int64_t it, int& len, int& blk) {
            len = 0;
            blk = -1;
            if (it >= end) return;
            int seq, kvh, j0;
            item_coords(it, seq, kvh, j0);
            len = p.context_lens[seq];
            if (j0 + lane < p.max_blocks_per_seq)
                blk = p.block_tables[static_cast<int64_t>(seq) * p.max_blocks_per_seq + j0 + lane];
        };
        int pf_len[S], pf_blk[S];
#pragma unroll
        for (int k = 0; k < S; ++k) fetch(begin + k, pf_len[k], pf_blk[k]);
        int n = 0;
        bool stop = false;
        for (int64_t base = begin; base < end && !stop; base += S) {
#pragma unroll
            for (int k = 0; k < S; ++k) {
                const int64_t it = base + k;
                if (it >= end) break;
                if (n >= S && !mbar_wait(&empty_bar[k], ((n / S) - 1) & 1)) {
                    if (lane == 0) {
                        atomicOr(p.err, kErrTimeout);
                        abort_flag = 1;
                    }
                    stop = true;
                    break;
                }
                int seq, kvh, j0;
                item_coords(it, seq, kvh, j0);
                const int L = pf_len[k];
                const bool len_ok = L >= 1 && L <= p.max_blocks_per_seq * p.block_size;
                const int nblk = len_ok ? (L + p.block_size - 1) / p.block_size : 0;
                int blk = -1;
                if (j0 + lane < nblk) {
                    blk = pf_blk[k];
                    if (blk < 0 || blk >= p.num_blocks) {
                        atomicOr(p.err, kErrBadBlock);
                        blk = -1;
                    }
                }
                fetch(it + S, pf_len[k], pf_blk[k]);
                const unsigned m = __ballot_sync(0xffffffffu, blk >= 0);
                if (lane == 0) {
                    valid_mask[k] = m;
                    mbar_arrive_expect_tx(&full_bar[k], __popc(m) * Cfg::kSlotBytes);
                }
                __syncwarp();
                if (blk >= 0)
                    bulk_copy_g2s(smem + k * Cfg::kStageBytes + lane * Cfg::kSlotBytes,
                                  static_cast<const uint16_t*>(p.kmeta) +
                                      (static_cast<int64_t>(blk) * p.num_kv_heads + kvh) * 2 * D,
                                  Cfg::kSlotBytes, &full_bar[k], policy);
                ++n;
            }
        }
        // let every copy this warp issued land before the CTA can exit
        for (int k = n - 1; k >= 0 && k >= n - S; --k)
            if (!mbar_wait(&full_bar[k % S], (k / S) & 1) && lane == 0) atomicOr(p.err, kErrTimeout);
        return;
    }
    const int ct = threadIdx.x - 32;
    const int c = ct % LPB, grp = ct / LPB;
    uint64_t qp[G][CPL / 2], qn[G][CPL / 2];
    int64_t q_row = -1;
    int n = 0;
    for (int64_t it = begin; it < end; ++it, ++n) {
        const int s = n % S;
        if (!mbar_wait(&full_bar[s], (n / S) & 1)) {
            if (lane == 0) atomicOr(p.err, kErrTimeout);
            break;
        }
        if (abort_flag) break;
        int seq, kvh, j0;
        item_coords(it, seq, kvh, j0);
        const int64_t row = static_cast<int64_t>(seq) * p.num_kv_heads + kvh;
        if (row != q_row) {
            q_row = row;
            const uint16_t* qsrc = static_cast<const uint16_t*>(p.q) +
                                   (static_cast<int64_t>(seq) * p.num_q_heads + kvh * G) * D + c * CPL;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                uint64_t f2[CPL / 2];
                load_pairs<T, CPL>(qsrc + g * D, f2);
#pragma unroll
                for (int i = 0; i < CPL / 2; ++i) {
                    float lo, hi;
                    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(f2[i]));
                    qp[g][i] = f2_pack(fmaxf(lo, 0.f), fmaxf(hi, 0.f));
                    qn[g][i] = f2_pack(fminf(lo, 0.f), fminf(hi, 0.f));
                }
            }
        }
        const unsigned m = valid_mask[s];
        float* out = p.bounds + row * p.max_blocks_per_seq;
        const unsigned char* stage = smem + s * Cfg::kStageBytes;
#pragma unroll
        for (int pass = 0; pass < kBItem / PER_PASS; ++pass) {
            const int slot = pass * PER_PASS + grp;
            float best = -INFINITY;
            if (m != 0) {  // uniform over the CTA
                const bool live = (m >> slot) & 1u;
                uint64_t a[CPL / 2], b[CPL / 2];
                const unsigned char* src = stage + (live ? slot : 0) * Cfg::kSlotBytes + c * CPL * 2;
                load_pairs<T, CPL>(src, a);
                load_pairs<T, CPL>(src + 2 * D, b);
                float v[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    uint64_t acc = f2_fma(qp[g][0], b[0], 0ull);
                    acc = f2_fma(qn[g][0], a[0], acc);
#pragma unroll
                    for (int i = 1; i < CPL / 2; ++i) {
                        acc = f2_fma(qp[g][i], b[i], acc);
                        acc = f2_fma(qn[g][i], a[i], acc);
                    }
                    v[g] = f2_sum(acc);
                }
                best = SplitSum<G, LPB / 2>::run(v, lane);
#pragma unroll
                for (int off = LPB / 2; off > LPB / 2 / G; off >>= 1)
                    best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, off));
                if (!live) best = -INFINITY;
            }
            const int j = j0 + slot;
            if (c == 0 && j < p.max_blocks_per_seq) out[j] = best;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
}

// Order-preserving map of a float bound to an unsigned key (larger bound,
// larger key).
__device__ __forceinline__ uint32_t bound_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Selection, step 2: one CTA of 256 threads per (kv head, sequence) finds the
// budget_blocks largest bounds of its row by radix selection: four passes of
// 8-bit digit histograms in shared memory give the key of the K-th largest
// bound.  Blocks above that key are kept, and blocks equal to it are kept in
// ascending logical order until K are chosen.  One block-wide scan over
// contiguous per-thread ranges places the chosen blocks in logical order.
constexpr int kTopkThreads = 256;

__global__ void __launch_bounds__(kTopkThreads) quest_topk_kernel(QuestSelectParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int hist[256];
    __shared__ uint32_t warp_scan[kTopkThreads / 32];
    __shared__ int warp_tokens[kTopkThreads / 32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_remaining;
    const int kvh = blockIdx.x;
    const int seq = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = p.context_lens[seq];
    const int32_t* table = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq;
    int32_t* out_row = p.sel_tables + (static_cast<int64_t>(seq) * p.num_kv_heads + kvh) * p.budget_blocks;
    int32_t* out_len = p.sel_lens + static_cast<int64_t>(seq) * p.num_kv_heads + kvh;
    if (L < 1 || L > p.max_blocks_per_seq * p.block_size) {
        if (tid == 0) {
            if (kvh == 0) atomicOr(p.err, kErrBadLen);
            *out_len = 0;
        }
        return;
    }
    const int nblk = (L + p.block_size - 1) / p.block_size;
    if (nblk <= p.budget_blocks) {
        for (int j = tid; j < p.budget_blocks; j += kTopkThreads) out_row[j] = j < nblk ? table[j] : 0;
        if (tid == 0) *out_len = L;
        return;
    }
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);               // [max_blocks]
    int32_t* blocks = reinterpret_cast<int32_t*>(keys + p.max_blocks_per_seq);  // [max_blocks]
    const float* row = p.bounds + (static_cast<int64_t>(seq) * p.num_kv_heads + kvh) * p.max_blocks_per_seq;
    for (int j = tid; j < nblk; j += kTopkThreads) {
        keys[j] = bound_key(row[j]);
        blocks[j] = table[j];
    }
    if (tid == 0) {
        s_prefix = 0;
        s_remaining = p.budget_blocks;
    }
    __syncthreads();
    uint32_t mask = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        hist[tid] = 0;  // kTopkThreads == 256 bins
        __syncthreads();
        const uint32_t prefix = s_prefix;
        for (int b0 = 0; b0 < nblk; b0 += kTopkThreads) {  // uniform trip count
            const int j = b0 + tid;
            const uint32_t k = j < nblk ? keys[j] : 0u;
            const bool in = j < nblk && (k & mask) == prefix;
            const int digit = in ? static_cast<int>((k >> shift) & 255u) : 256;
            const unsigned same = __match_any_sync(0xffffffffu, digit);
            if (in && lane == __ffs(same) - 1) atomicAdd(&hist[digit], __popc(same));
        }
        __syncthreads();
        if (warp == 0) {
            // digits from the top: lane l owns digits 255-8l .. 248-8l
            int cnt[8], tot = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                cnt[e] = hist[255 - 8 * lane - e];
                tot += cnt[e];
            }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            const int remaining = s_remaining;
            const int excl = incl - tot;
            if (excl < remaining && remaining <= incl) {  // exactly one lane
                int cum = excl;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (cum + cnt[e] >= remaining) {
                        s_prefix = prefix | (static_cast<uint32_t>(255 - 8 * lane - e) << shift);
                        s_remaining = remaining - cum;
                        break;
                    }
                    cum += cnt[e];
                }
            }
        }
        mask |= 255u << shift;
        __syncthreads();
    }
    const uint32_t kth = s_prefix;  // key of the K-th largest bound
    const int ties = s_remaining;   // how many blocks with exactly that key to keep
    // thread t owns logical blocks [t*C, t*C + C); counts of keys above kth
    // (low 16 bits) and equal to it (high 16 bits) are scanned together
    const int C = (nblk + kTopkThreads - 1) / kTopkThreads;
    const int lo = min(nblk, tid * C), hi = min(nblk, lo + C);
    uint32_t packed = 0;
    for (int j = lo; j < hi; ++j) packed += keys[j] > kth ? 1u : (keys[j] == kth ? 0x10000u : 0u);
    uint32_t incl = packed;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_scan[warp] = incl;
    __syncthreads();
    uint32_t before = incl - packed;
    for (int w = 0; w < warp; ++w) before += warp_scan[w];
    int gt = static_cast<int>(before & 0xffffu), eq = static_cast<int>(before >> 16);
    int tokens = 0;
    for (int j = lo; j < hi; ++j) {
        const uint32_t k = keys[j];
        if (k > kth || (k == kth && eq < ties)) {
            out_row[gt + min(eq, ties)] = blocks[j];
            tokens += j == nblk - 1 ? L - j * p.block_size : p.block_size;
        }
        if (k > kth) ++gt;
        else if (k == kth) ++eq;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) tokens += __shfl_xor_sync(0xffffffffu, tokens, off);
    if (lane == 0) warp_tokens[warp] = tokens;
    __syncthreads();
    if (tid == 0) {
        int total = 0;
        for (int w = 0; w < kTopkThreads / 32; ++w) total += warp_tokens[w];
        *out_len = total;
    }
}

cudaError_t launch_quest_minmax(const QuestMetaParams& p, int dtype, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(p.num_seqs) * p.max_blocks_per_seq * p.num_kv_heads * (p.head_dim / 8);
    if (total == 0) return cudaSuccess;
    const int blocks = static_cast<int>(total / 256 + 1 < 152 * 32 ? total / 256 + 1 : 152 * 32);
    if (dtype == kBF16)
        quest_minmax_kernel<kBF16><<<blocks, 256, 0, s>>>(p);
    else
        quest_minmax_kernel<kF16><<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_quest_append_minmax(const QuestAppendParams& p, int dtype, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * (p.head_dim / 8);
    if (total == 0) return cudaSuccess;
    const int blocks = static_cast<int>(total / 256 + 1 < 152 * 16 ? total / 256 + 1 : 152 * 16);
    if (dtype == kBF16)
        quest_append_minmax_kernel<kBF16><<<blocks, 256, 0, s>>>(p);
    else
        quest_append_minmax_kernel<kF16><<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

namespace {
template <int T, int D, int G>
cudaError_t bounds_one(const QuestSelectParams& p, cudaStream_t s) {
    const int64_t items = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads *
                          ((p.max_blocks_per_seq + kBItem - 1) / kBItem);
    constexpr int smem = BoundsCfg<D>::kSmem;
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || !configured[dev]) {
        e = cudaFuncSetAttribute(quest_bounds_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) configured[dev] = true;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t want = static_cast<int64_t>(sms) * 3;
    const int grid = static_cast<int>(items < want ? items : want);
    quest_bounds_kernel<T, D, G><<<grid, kBThreads, smem, s>>>(p, items);
    return cudaGetLastError();
}
template <int T, int D>
cudaError_t bounds_g(const QuestSelectParams& p, int G, cudaStream_t s) {
    switch (G) {
        case 1: return bounds_one<T, D, 1>(p, s);
        case 2: return bounds_one<T, D, 2>(p, s);
        case 4: return bounds_one<T, D, 4>(p, s);
        case 8: return bounds_one<T, D, 8>(p, s);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t launch_quest_select(const QuestSelectParams& p, int dtype, int G, cudaStream_t s) {
    if (p.num_seqs == 0) return cudaSuccess;
    cudaError_t e;
    if (dtype == kBF16)
        e = p.head_dim == 128 ? bounds_g<kBF16, 128>(p, G, s) : bounds_g<kBF16, 64>(p, G, s);
    else
        e = p.head_dim == 128 ? bounds_g<kF16, 128>(p, G, s) : bounds_g<kF16, 64>(p, G, s);
    if (e != cudaSuccess) return e;
    const size_t smem = static_cast<size_t>(p.max_blocks_per_seq) * 8;  // key + block id per logical block
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(quest_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    quest_topk_kernel<<<dim3(p.num_kv_heads, p.num_seqs), kTopkThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
