// QUEST query-aware block selection (Tencent Cloud "LLMs serving
// challenges", section "Query-sparsity attention / QUEST"): per block the
// channel-wise minimum and maximum of its keys; for a query, the upper bound
//     U = sum_c max(q_c * min_c, q_c * max_c)
// of q.k over the block's keys; attention then reads only the K blocks with
// the largest bounds.
//
// Metadata layout: kmeta [num_blocks][Hkv][2][D] in the queries' 16-bit type
// (row 0 = min, row 1 = max over the block's filled slots).  For a 16-bit
// cache that is the cache's type, and min and max of 16-bit values are exact
// 16-bit values.  For an E4M3 cache the metadata holds the decoded codes
// without the per-tensor scale (every E4M3 value is exact in binary16 and in
// bfloat16): the bounds are then the true bounds divided by k_scale > 0,
// which ranks the blocks identically.
#include <cfloat>

#include "kernels.h"
#include "pkv_device.cuh"
#include "pkv_tc.cuh"
#include "tensor_map.cuh"

namespace pkv {

namespace {

template <int T>
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
    Vec16<T>::to_float(u, f);
}

// 8 consecutive cache elements -> floats (E4M3: the codes' values, unscaled).
template <int C>
__device__ __forceinline__ void load8(const void* src, float* f) {
    if constexpr (C == kE4M3) {
        const uint2 u = *reinterpret_cast<const uint2*>(src);
        const uint32_t w[2] = {u.x, u.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t h2 = e4m3x2_to_f16x2(static_cast<uint16_t>((w[i] >> (16 * j)) & 0xffffu));
                const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&h2));
                f[4 * i + 2 * j] = t.x;
                f[4 * i + 2 * j + 1] = t.y;
            }
        }
    } else {
        unpack8<C>(*reinterpret_cast<const uint4*>(src), f);
    }
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
// chunk) over the block's filled slots.  T: metadata type, C: cache type.
template <int T, int C>
__global__ void __launch_bounds__(256) quest_minmax_kernel(QuestMetaParams p) {
    constexpr int EB = C == kE4M3 ? 1 : 2;  // bytes per cache element
    const int chunks = p.head_dim / 8;
    const int64_t per_seq = static_cast<int64_t>(p.max_blocks_per_seq) * p.num_kv_heads * chunks;
    const int64_t total = per_seq * p.num_seqs;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // i = ((seq * max_blocks + j) * Hkv + kvh) * chunks + c
        int64_t q1, q2, q3;
        int c, kvh, j;
        divmod_u(i, chunks, q1, c);
        divmod_u(q1, p.num_kv_heads, q2, kvh);
        divmod_u(q2, p.max_blocks_per_seq, q3, j);
        const int seq = static_cast<int>(q3);
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
        const unsigned char* base =
            static_cast<const unsigned char*>(p.k_cache) +
            (((static_cast<int64_t>(blk) * p.num_kv_heads + kvh) * p.block_size) * p.head_dim + c * 8) * EB;
        for (int t = 0; t < filled; ++t) {
            float f[8];
            load8<C>(base + static_cast<int64_t>(t) * p.head_dim * EB, f);
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
// per call (as one decode step gives).  T: query / key / metadata type; an
// E4M3 cache (C) first stores each key as the append does, e4m3(x / k_scale)
// (binary32 division, round to nearest even, saturating), and the metadata
// takes the stored code's value.
template <int T, int C>
__global__ void __launch_bounds__(256) quest_append_minmax_kernel(QuestAppendParams p) {
    const float ks = C == kE4M3 ? *p.k_scale : 1.0f;
    const int chunks = p.head_dim / 8;
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * chunks;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t th, t, blk;  // th = token * Hkv + kv head
        int c, kvh, off;
        divmod_u(i, chunks, th, c);
        divmod_u(th, p.num_kv_heads, t, kvh);
        const int64_t slot = p.slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= static_cast<int64_t>(p.num_blocks) * p.block_size) {
            atomicOr(p.err, kErrBadSlot);
            continue;
        }
        divmod_u(slot, p.block_size, blk, off);
        const bool first = off == 0;
        float k[8];
        unpack8<T>(*reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k_new) + th * p.head_dim + c * 8), k);
        if constexpr (C == kE4M3) {
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const uint16_t lo = __nv_cvt_float_to_fp8(__fdiv_rn(k[e], ks), __NV_SATFINITE, __NV_E4M3);
                const uint16_t hi = __nv_cvt_float_to_fp8(__fdiv_rn(k[e + 1], ks), __NV_SATFINITE, __NV_E4M3);
                const uint32_t h2 = e4m3x2_to_f16x2(static_cast<uint16_t>(lo | (hi << 8)));
                const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&h2));
                k[e] = t.x;
                k[e + 1] = t.y;
            }
        }
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

// ---- selection, step 1: bounds on the tensor cores --------------------------
// For channel c the larger of q*min and q*max is q+ * max + q- * min (q+, q-
// the positive and negative parts of q), so a bound is a dot product of the
// block's metadata row [min | max] with [q- | q+].  For a group of HG kv
// heads (HG a power of two dividing Hkv, HG*G <= 32) and BPI = 128/HG blocks,
// all bounds come from one product
//     U[128 x N] = A[128 x 2D] * B[N x 2D]^T,
// A's row r = metadata row of (block r % BPI, kv head r / BPI) as stored,
// B's row n = [q- | q+] of query head n of the group (rows HG*G .. N-1 zero,
// N = HG*G rounded up to 16), accumulated in float32 by tcgen05.mma kind::f16
// with A in tensor memory and B in shared memory (each product of two 16-bit
// values is exact in float32).  Row r uses only its kv head's G columns; the
// bound is their max.
//
// An item is one (sequence, kv-head group, chunk of BPI blocks).  Persistent
// CTAs (one per SM) walk contiguous ranges of items:
//  warp 0     bulk-copies each block's HG metadata rows (one HG*4*D-byte copy:
//             the Hkv rows of a physical block are contiguous) into a ring of
//             staging stages, blocks 16 bytes apart beyond their rows; block
//             ids are fetched one item ahead.
//  warps 1-4  the warp owning tensor-memory lanes 32w'..32w'+31 loads rows
//             32w'.. of the item from staging (row-major reads; consecutive
//             rows are different blocks, so a quarter warp hits distinct
//             banks) and stores them into one of two A buffers in tensor
//             memory (tcgen05.st, 32 columns per instruction); rewrites B when
//             the (sequence, group) changes; frees the stage.
//  warp 5     allocates 512 tensor-memory columns (A: 2 x 128, D: 2 x 32) and
//             issues the 2D/16 MMAs of an item.
//  warps 6-9  thread i reads row i of the D buffer, takes the max over its kv
//             head's G columns and stores the bound; rows past the context or
//             with a bad block id get -inf.
// Bounds go to the workspace [B][Hkv][max_blocks].  Every barrier wait is
// bounded; a timeout stops the CTA's roles, which drain their copies and
// MMAs before the tensor memory is freed.
constexpr int kQRows = 128;
constexpr int kQTranscribeWarps = 4;
constexpr int kQMmaWarp = 1 + kQTranscribeWarps;
constexpr int kQThreads = 32 * (kQMmaWarp + 1 + 4);
constexpr int kQMaxN = 32;
constexpr int kQTmemCols = 512;
constexpr int kQTmemD = 256;  // first D column; A buffers at 0 and 128
constexpr int kQFetchAhead = 3;  // items whose lengths and block ids are in flight

template <int D>
struct QBoundsCfg {
    static constexpr int KCH = 2 * D / 8;               // 16-byte chunks per metadata row
    static constexpr int ROW = 4 * D;                   // bytes per metadata row
    static constexpr int SBO = KCH * 128;               // bytes between 8-row groups of B
    static constexpr int STG = kQRows * ROW + kQRows * 16;  // one staging stage (blocks padded by 16 bytes)
    static constexpr int B_BYTES = kQMaxN * ROW;
    static constexpr int NSTG_FIT = (224 * 1024 - B_BYTES) / STG;
    static constexpr int NSTG = NSTG_FIT > 4 ? 4 : NSTG_FIT;
    static constexpr int SMEM = NSTG * STG + B_BYTES + 128;  // + room to align the base
    static_assert(NSTG >= 2, "at least two staging stages");
    static_assert(KCH * 4 <= 128, "a row fits one 128-column A buffer");
};

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool q_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

// q+ and q- of eight 16-bit values, by their sign bits (exact).
__device__ __forceinline__ void split_signs(const uint4& u, uint4& pos, uint4& neg) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t pw[4], nw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t m = ((w[i] >> 15) & 0x00010001u) * 0xffffu;  // all ones in each negative half
        nw[i] = w[i] & m;
        pw[i] = w[i] & ~m;
    }
    pos = make_uint4(pw[0], pw[1], pw[2], pw[3]);
    neg = make_uint4(nw[0], nw[1], nw[2], nw[3]);
}

template <int T, int D, int G>
__global__ void __launch_bounds__(kQThreads, 1) quest_bounds_kernel(QuestSelectParams p, int64_t num_items) {
    using Cfg = QBoundsCfg<D>;
    constexpr int NSTG = Cfg::NSTG;
    constexpr int KS = 2 * D / 16;  // MMA k-steps of 16 elements (8 tensor-memory columns each)
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[NSTG], empty[NSTG], a_full[2], a_free[2], d_full[2], d_free[2], final_bar;
    __shared__ unsigned valid_mask[NSTG][kQRows / 32];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag_s;
    volatile int* abort_flag = &abort_flag_s;
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem) + 127) & ~uintptr_t(127));
    unsigned char* staging = sm;
    unsigned char* Btile = sm + NSTG * Cfg::STG;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HG = p.group_heads;                 // kv heads per item
    const int BPI = kQRows / HG;                  // blocks per item
    const int SB = HG * Cfg::ROW + 16;            // staging bytes per block
    const int HGG = HG * G;                       // query heads per item
    const int N = (HGG + 15) / 16 * 16;           // MMA N
    const int groups = p.num_kv_heads / HG;
    const int chunks = (p.max_blocks_per_seq + BPI - 1) / BPI;
    // items number fewer than 2^31 (checked on the host): 32-bit item arithmetic
    const int begin = static_cast<int>(num_items * blockIdx.x / gridDim.x);
    const int count = static_cast<int>(num_items * (blockIdx.x + 1) / gridDim.x - begin);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTG; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kQTranscribeWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&a_full[i], kQTranscribeWarps);
            mbar_init(&a_free[i], 1);
            mbar_init(&d_full[i], 1);
            mbar_init(&d_free[i], 4);
        }
        mbar_init(&final_bar, 1);
        abort_flag_s = 0;
        mbar_init_fence();
    }
    if (warp == kQMmaWarp) {
        tc::tmem_alloc(&tmem_base_s, kQTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_s;
    // item -> (sequence, kv-head group, first block)
    auto coords = [&](int i, int& seq, int& kvg, int& j0) {
        const unsigned it = static_cast<unsigned>(begin + i);
        const unsigned r = it / static_cast<unsigned>(chunks);
        j0 = static_cast<int>(it - r * chunks) * BPI;
        seq = static_cast<int>(r / static_cast<unsigned>(groups));
        kvg = static_cast<int>(r) - seq * groups;
    };
    auto nblocks_of = [&](int L) {
        return L >= 1 && L <= p.max_blocks_per_seq * p.block_size ? (L + p.block_size - 1) / p.block_size : 0;
    };

    if (warp == 0) {
        // ------------------------------------------------------------- producer
        // lane l copies blocks l, l+32, ... of the item.  Lengths and block ids
        // are loaded kQFetchAhead items ahead, in rotating registers (table
        // entries read for every j < max_blocks, checked against the length
        // when used).
        const uint64_t policy = l2_policy_evict_first();
        const unsigned char* kmeta = static_cast<const unsigned char*>(p.kmeta);
        const uint32_t copy_bytes = HG * Cfg::ROW;
        constexpr int BPL = kQRows / 32;  // most blocks per lane (HG = 1)
        int pf_len[kQFetchAhead], pf_blk[kQFetchAhead][BPL];
        auto fetch = [&](int i, int& len, int* blks) {
            len = 0;
            if (i >= count) return;
            int seq, kvg, j0;
            coords(i, seq, kvg, j0);
            len = p.context_lens[seq];
#pragma unroll
            for (int u = 0; u < BPL; ++u) {
                const int jl = u * 32 + lane, j = j0 + jl;
                blks[u] = jl < BPI && j < p.max_blocks_per_seq
                              ? p.block_tables[static_cast<int64_t>(seq) * p.max_blocks_per_seq + j]
                              : -1;
            }
        };
#pragma unroll
        for (int k = 0; k < kQFetchAhead; ++k) fetch(k, pf_len[k], pf_blk[k]);
        // one item: wait for its stage, check its block ids, refill the fetch
        // slot, issue its copies; false on an abort
        auto produce = [&](int i, int& len, int* pblk) {
            const int s = i % NSTG;
            if (i >= NSTG &&
                !__all_sync(0xffffffffu, q_wait(&empty[s], ((i / NSTG) - 1) & 1, abort_flag, p.err)))
                return false;
            int seq, kvg, j0;
            coords(i, seq, kvg, j0);
            const int nblk = nblocks_of(len);
            int blk[BPL];
            unsigned ncopies = 0;
#pragma unroll
            for (int u = 0; u < BPL; ++u) {
                const int jl = u * 32 + lane, j = j0 + jl;
                blk[u] = -1;
                if (jl < BPI && j < nblk) {
                    blk[u] = pblk[u];
                    if (blk[u] < 0 || blk[u] >= p.num_blocks) {
                        atomicOr(p.err, kErrBadBlock);
                        blk[u] = -1;
                    }
                }
                ncopies += __popc(__ballot_sync(0xffffffffu, blk[u] >= 0));
            }
            // valid rows: row r is valid when its block r % BPI is
            for (int w = 0; w < kQRows / 32; ++w) {
                const int jl = (w * 32 + lane) % BPI;
                int b = __shfl_sync(0xffffffffu, blk[0], jl & 31);
#pragma unroll
                for (int u = 1; u < BPL; ++u) {
                    const int bu = __shfl_sync(0xffffffffu, blk[u], jl & 31);
                    if ((jl >> 5) == u) b = bu;
                }
                const unsigned m = __ballot_sync(0xffffffffu, b >= 0);
                if (lane == 0) valid_mask[s][w] = m;
            }
            fetch(i + kQFetchAhead, len, pblk);
            if (lane == 0) mbar_arrive_expect_tx(&full[s], ncopies * copy_bytes);
            __syncwarp();
#pragma unroll
            for (int u = 0; u < BPL; ++u)
                if (blk[u] >= 0)
                    bulk_copy_g2s(staging + s * Cfg::STG + (u * 32 + lane) * SB,
                                  kmeta + (static_cast<int64_t>(blk[u]) * p.num_kv_heads + kvg * HG) * Cfg::ROW,
                                  copy_bytes, &full[s], policy);
            return true;
        };
        int i = 0;
        bool ok = true;
        for (int base = 0; base < count && ok; base += kQFetchAhead) {
#pragma unroll
            for (int k = 0; k < kQFetchAhead; ++k) {  // fetch slot k holds item base + k
                if (base + k >= count || !(ok = produce(base + k, pf_len[k], pf_blk[k]))) break;
                i = base + k + 1;
            }
        }
        // let every copy this warp issued land before the CTA can exit
        for (int k = i - 1; k >= 0 && k >= i - NSTG; --k)
            if (!mbar_wait(&full[k % NSTG], (k / NSTG) & 1) && lane == 0) atomicOr(p.err, kErrTimeout);
    } else if (warp <= kQTranscribeWarps) {
        // ----------------------------------------------------------- transcribe
        const int quad = warp & 3;            // tensor-memory lanes 32*quad .. 32*quad+31
        const int r = quad * 32 + lane;       // row of the item
        const int t = threadIdx.x - 32;       // 0..127, for the B rows
        const int h = r / BPI, jl = r % BPI;  // kv head within the group, block within the item
        for (int i = 0; i < count; ++i) {
            const int s = i % NSTG, ab = i & 1;
            int seq, kvg, j0;
            coords(i, seq, kvg, j0);
            bool same = false;
            if (i >= 1) {
                int ps, pg, pj;
                coords(i - 1, ps, pg, pj);
                same = ps == seq && pg == kvg;
            }
            if (!same) {
                // B = [q- | q+] of the group's query heads (rows HGG..N-1 zero),
                // written before this item's metadata arrives; the previous
                // item's MMAs read B, so they must have completed
                if (i >= 1 &&
                    !__all_sync(0xffffffffu, q_wait(&a_free[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag, p.err)))
                    break;
                const uint16_t* qrow = static_cast<const uint16_t*>(p.q) +
                                       (static_cast<int64_t>(seq) * p.num_q_heads + kvg * HGG) * D;
                for (int idx = t; idx < N * Cfg::KCH; idx += 32 * kQTranscribeWarps) {
                    const int n = idx / Cfg::KCH, c = idx % Cfg::KCH;
                    uint4 val = make_uint4(0, 0, 0, 0);
                    if (n < HGG) {
                        const bool positive = c >= Cfg::KCH / 2;
                        const int cc = positive ? c - Cfg::KCH / 2 : c;
                        uint4 pos, neg;
                        split_signs(*reinterpret_cast<const uint4*>(qrow + n * D + cc * 8), pos, neg);
                        val = positive ? pos : neg;
                    }
                    *reinterpret_cast<uint4*>(Btile + (n / 8) * Cfg::SBO + c * 128 + (n % 8) * 16) = val;
                }
                tc::fence_proxy_async_smem();
            }
            if (!__all_sync(0xffffffffu, q_wait(&full[s], (i / NSTG) & 1, abort_flag, p.err))) break;
            if (i >= 2 && !__all_sync(0xffffffffu, q_wait(&a_free[ab], ((i >> 1) - 1) & 1, abort_flag, p.err)))
                break;
            const bool valid = (valid_mask[s][r >> 5] >> (r & 31)) & 1u;
            const unsigned char* src = staging + s * Cfg::STG + jl * SB + h * Cfg::ROW;
            const uint32_t a_col = tmem + (static_cast<uint32_t>(quad * 32) << 16) + ab * 128;
#pragma unroll
            for (int g = 0; g < Cfg::KCH / 8; ++g) {  // 128 bytes = 32 columns per store
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = valid ? *reinterpret_cast<const uint4*>(src + (g * 8 + c) * 16) : make_uint4(0, 0, 0, 0);
                    w[4 * c] = u.x;
                    w[4 * c + 1] = u.y;
                    w[4 * c + 2] = u.z;
                    w[4 * c + 3] = u.w;
                }
                tc::tmem_st32(a_col + g * 32, w);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&a_full[ab]);
                mbar_arrive(&empty[s]);
            }
        }
    } else if (warp == kQMmaWarp) {
        // ------------------------------------------------------------------ MMA
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16(kQRows, N, T == kBF16, false, false);
            const uint32_t b0 = smem_addr(Btile);
            for (int i = 0; i < count; ++i) {
                const int ab = i & 1;
                if (!q_wait(&a_full[ab], (i >> 1) & 1, abort_flag, p.err)) break;
                if (i >= 2 && !q_wait(&d_free[ab], ((i >> 1) - 1) & 1, abort_flag, p.err)) break;
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
                    tc::mma_f16_ts(tmem + kQTmemD + ab * kQMaxN, tmem + ab * 128 + ks * 8,
                                   tc::desc_noswizzle(b0 + ks * 256, 128, Cfg::SBO), idesc, ks > 0 ? 1u : 0u);
                tc::commit(&d_full[ab]);
                tc::commit(&a_free[ab]);
            }
            // every MMA this thread issued completes before the tensor memory is freed
            tc::commit(&final_bar);
            if (!mbar_wait(&final_bar, 0)) atomicOr(p.err, kErrTimeout);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- epilogue
        // the row's length and block id load kQFetchAhead items ahead
        const int quad = warp & 3;  // tensor-memory lanes 32*quad .. 32*quad+31
        const int R = quad * 32 + lane;
        const int h = R / BPI, jl = R % BPI;
        int pf_len[kQFetchAhead], pf_blk[kQFetchAhead];
        auto fetch = [&](int i, int& len, int& blk) {
            len = 0;
            blk = -1;
            if (i >= count) return;
            int seq, kvg, j0;
            coords(i, seq, kvg, j0);
            len = p.context_lens[seq];
            if (j0 + jl < p.max_blocks_per_seq)
                blk = p.block_tables[static_cast<int64_t>(seq) * p.max_blocks_per_seq + j0 + jl];
        };
#pragma unroll
        for (int k = 0; k < kQFetchAhead; ++k) fetch(k, pf_len[k], pf_blk[k]);
        auto finish = [&](int i, int& len, int& pblk) {
            const int b = i & 1;
            int seq, kvg, j0;
            coords(i, seq, kvg, j0);
            const int j = j0 + jl;
            const bool valid = j < nblocks_of(len) && pblk >= 0 && pblk < p.num_blocks;
            fetch(i + kQFetchAhead, len, pblk);
            if (!__all_sync(0xffffffffu, q_wait(&d_full[b], (i >> 1) & 1, abort_flag, p.err))) return false;
            tc::fence_after_sync();
            float best = -INFINITY;
            for (int c0 = 0; c0 < N; c0 += 16) {  // columns h*G .. h*G+G-1 are this row's heads
                float v[16];
                tc::TmemLd<16>::load(tmem + (static_cast<uint32_t>(quad * 32) << 16) + kQTmemD + b * kQMaxN + c0,
                                     v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (c0 + k >= h * G && c0 + k < h * G + G) best = fmaxf(best, v[k]);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_free[b]);
            if (j < p.max_blocks_per_seq)
                p.bounds[(static_cast<int64_t>(seq) * p.num_kv_heads + kvg * HG + h) * p.max_blocks_per_seq + j] =
                    valid ? best : -INFINITY;
            return true;
        };
        bool ok = true;
        for (int base = 0; base < count && ok; base += kQFetchAhead) {
#pragma unroll
            for (int k = 0; k < kQFetchAhead; ++k)  // fetch slot k holds item base + k
                if (base + k >= count || !(ok = finish(base + k, pf_len[k], pf_blk[k]))) break;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kQMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kQTmemCols);
    }
}

// ---- selection, step 1, kv heads in groups of 8: A straight from TMA ---------
// When Hkv is a multiple of 8 the metadata of 8 consecutive kv heads of a
// block is 8 consecutive 4D-byte rows.  Viewed as a 3-D tensor (64 elements
// of a 128-byte atom; rows, 4D bytes apart; the 2D/64 atoms of a row, 128
// bytes apart), one TMA box of 64 x 8 x 2D/64 with 128-byte swizzle lands a
// block's 8 rows as 2D/64 consecutive 1 KB swizzle atoms of a K-major MMA
// operand, so the A operand needs no transcription: an item (sequence, group
// of 8 kv heads, chunk of 16 blocks) is 16 boxes, and A row 8*jl + h is the
// metadata row of (block jl of the chunk, kv head h of the group); 8-row
// groups (blocks) are 2D/64 KB apart.  B = [q- | q+] of the group's 8G query
// heads (zero-padded to N) as in the kernel above, D = A B^T in tensor memory.
// Roles (224 threads):
//  warps 0, 6 producers of the even and the odd items: block ids and lengths
//             fetched three items ahead, TMA boxes into a ring of stages
//  warp 1     tensor memory; lane 0 issues the 2D/16 MMAs of an item and frees
//             its stage when they complete
//  warps 2-5  write B for each new (sequence, group), N * 2D / 1024 16-byte
//             chunks a thread (2 to 16) with every load issued first (the
//             epilogue of the previous item has seen its MMAs, the last to
//             read the old B, complete); thread i reads D row i, keeps the max
//             over its kv head's G columns and stores the bound (-inf past the
//             context or for a bad block id)
// Every wait is bounded; a timeout stops the CTA's roles.  After the final
// barrier one thread waits for the copies last armed on each stage, and the
// MMA warp has waited for its MMAs, before the tensor memory is freed.
constexpr int kQ8Blocks = 16;  // blocks per item: 16 x 8 rows = M
constexpr int kQ8Threads = 32 * 7;

template <int D, int G>
struct QBounds8Cfg {
    static constexpr int NATOM = 2 * D / 64;             // 128-byte atoms of a metadata row
    static constexpr int BLK = NATOM * 1024;             // staging bytes of one block's 8 rows
    static constexpr int STG = kQ8Blocks * BLK;          // one stage (64 KB at D = 128)
    static constexpr int N = 8 * G < 16 ? 16 : 8 * G;    // MMA N: the group's query heads, padded
    static constexpr int KCH = 2 * D / 8;                // 16-byte chunks of a B row
    static constexpr int BSBO = KCH * 128;               // bytes between 8-row groups of B
    static constexpr int B_BYTES = N * 4 * D;
    static constexpr int NSTG_FIT = (227 * 1024 - B_BYTES - 1024 - 256) / STG;
    static constexpr int NSTG = NSTG_FIT > 6 ? 6 : NSTG_FIT;
    static constexpr int SMEM = NSTG * STG + B_BYTES + 1024;  // + room to align the base to 1 KB
    static constexpr int TMEM_COLS = 2 * N <= 32 ? 32 : (2 * N <= 64 ? 64 : 128);  // two D buffers
    static_assert(NSTG >= 2, "at least two staging stages");
    static_assert(N * KCH % 128 == 0, "the 128 epilogue threads share B's chunks evenly");
};

template <int T, int D, int G>
__global__ void __launch_bounds__(kQ8Threads, 1)
    quest_bounds8_kernel(const __grid_constant__ CUtensorMap mmap, QuestSelectParams p, int64_t num_items) {
    using Cfg = QBounds8Cfg<D, G>;
    constexpr int NSTG = Cfg::NSTG;
    constexpr int N = Cfg::N;
    constexpr int KS = 2 * D / 16;  // MMA k-steps of 16 elements
    extern __shared__ __align__(128) unsigned char smem8[];  // aligned to 1 KB below
    __shared__ uint64_t full[NSTG], empty[NSTG], d_full[2], d_free[2], b_full, final_bar;
    __shared__ int armed[NSTG];  // the last item whose copies were armed on each stage
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag_s;
    volatile int* abort_flag = &abort_flag_s;
    unsigned char* sm =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem8) + 1023) & ~uintptr_t(1023));
    unsigned char* staging = sm;
    unsigned char* Btile = sm + NSTG * Cfg::STG;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int groups = p.num_kv_heads / 8;
    const int chunks = (p.max_blocks_per_seq + kQ8Blocks - 1) / kQ8Blocks;
    // items number fewer than 2^31 (checked on the host): 32-bit item arithmetic
    const int begin = static_cast<int>(num_items * blockIdx.x / gridDim.x);
    const int count = static_cast<int>(num_items * (blockIdx.x + 1) / gridDim.x - begin);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTG; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
            armed[i] = -1;
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_free[i], 4);
        }
        mbar_init(&b_full, 4);  // the four epilogue warps
        mbar_init(&final_bar, 1);
        abort_flag_s = 0;
        mbar_init_fence();
        tc::prefetch_tensormap(&mmap);
    }
    if (warp == 1) {
        tc::tmem_alloc(&tmem_base_s, Cfg::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_s;
    // item -> (sequence, kv-head group, first block)
    auto coords = [&](int i, int& seq, int& kvg, int& j0) {
        const unsigned it = static_cast<unsigned>(begin + i);
        const unsigned r = it / static_cast<unsigned>(chunks);
        j0 = static_cast<int>(it - r * chunks) * kQ8Blocks;
        seq = static_cast<int>(r / static_cast<unsigned>(groups));
        kvg = static_cast<int>(r) - seq * groups;
    };
    // items i and i-1 read different B (a new (sequence, group)); true for i = 0
    auto new_b = [&](int i) {
        if (i == 0) return true;
        int s0, g0, j0, s1, g1, j1;
        coords(i - 1, s0, g0, j0);
        coords(i, s1, g1, j1);
        return s0 != s1 || g0 != g1;
    };
    auto nblocks_of = [&](int L) {
        return L >= 1 && L <= p.max_blocks_per_seq * p.block_size ? (L + p.block_size - 1) / p.block_size : 0;
    };

    if (warp == 0 || warp == 6) {
        // ------------------------------------------------------------ producers
        // warp 0 the even items, warp 6 the odd ones (the lanes of one copy
        // instruction issue one after another, so two warps issue twice as
        // fast); lane jl holds block jl of the item and loads its box
        const int pw = warp == 0 ? 0 : 1;
        const uint64_t policy = l2_policy_evict_first();
        int pf_len[kQFetchAhead], pf_blk[kQFetchAhead];
        auto fetch = [&](int i, int& len, int& blk) {
            len = 0;
            blk = -1;
            if (i >= count) return;
            int seq, kvg, j0;
            coords(i, seq, kvg, j0);
            len = p.context_lens[seq];
            if (lane < kQ8Blocks && j0 + lane < p.max_blocks_per_seq)
                blk = p.block_tables[static_cast<int64_t>(seq) * p.max_blocks_per_seq + j0 + lane];
        };
#pragma unroll
        for (int k = 0; k < kQFetchAhead; ++k) fetch(pw + 2 * k, pf_len[k], pf_blk[k]);
        auto produce = [&](int i, int& len, int& pblk) {
            const int s = i % NSTG;
            if (i >= NSTG &&
                !__all_sync(0xffffffffu, q_wait(&empty[s], ((i / NSTG) - 1) & 1, abort_flag, p.err)))
                return false;
            int seq, kvg, j0;
            coords(i, seq, kvg, j0);
            int blk = -1;
            if (lane < kQ8Blocks && j0 + lane < nblocks_of(len)) {
                blk = pblk;
                if (blk < 0 || blk >= p.num_blocks) {
                    atomicOr(p.err, kErrBadBlock);
                    blk = -1;
                }
            }
            const unsigned valid = __ballot_sync(0xffffffffu, blk >= 0);
            fetch(i + 2 * kQFetchAhead, len, pblk);
            if (lane == 0) {
                armed[s] = i;  // stage s is re-armed only after item i's copies landed
                mbar_arrive_expect_tx(&full[s], __popc(valid) * Cfg::BLK);
            }
            __syncwarp();
            if (blk >= 0)
                tc::tma_load_3d(staging + s * Cfg::STG + lane * Cfg::BLK, &mmap, 0, blk * p.num_kv_heads + kvg * 8, 0,
                                &full[s], policy);
            return true;
        };
        bool ok = true;
        for (int base = pw; base < count && ok; base += 2 * kQFetchAhead) {
#pragma unroll
            for (int k = 0; k < kQFetchAhead; ++k) {  // fetch slot k holds item base + 2k
                const int i = base + 2 * k;
                if (i >= count || !(ok = produce(i, pf_len[k], pf_blk[k]))) break;
            }
        }
        // (the copies still in flight are drained after the final barrier)
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16(kQRows, N, T == kBF16, false, false);
            const uint32_t b0 = smem_addr(Btile);
            int v = -1;  // B versions seen
            for (int i = 0; i < count; ++i) {
                const int s = i % NSTG, b = i & 1;
                if (new_b(i)) {
                    ++v;
                    if (!q_wait(&b_full, v & 1, abort_flag, p.err)) break;
                }
                if (!q_wait(&full[s], (i / NSTG) & 1, abort_flag, p.err)) break;
                if (i >= 2 && !q_wait(&d_free[b], ((i >> 1) - 1) & 1, abort_flag, p.err)) break;
                tc::fence_after_sync();
                const uint32_t a0 = smem_addr(staging + s * Cfg::STG);
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
                    tc::mma_f16(tmem + b * N, tc::desc_sw128(a0 + (ks >> 2) * 1024 + (ks & 3) * 32, 16, Cfg::BLK),
                                tc::desc_noswizzle(b0 + ks * 256, 128, Cfg::BSBO), idesc, ks > 0 ? 1u : 0u);
                tc::commit(&empty[s]);
                tc::commit(&d_full[b]);
            }
            // every MMA this thread issued completes before the tensor memory is freed
            tc::commit(&final_bar);
            if (!mbar_wait(&final_bar, 0)) atomicOr(p.err, kErrTimeout);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- epilogue
        const int quad = warp & 3;  // tensor-memory lanes 32*quad .. 32*quad+31
        const int R = quad * 32 + lane;
        const int jl = R >> 3, h = R & 7;  // block of the item, kv head of the group
        int pf_len[kQFetchAhead], pf_blk[kQFetchAhead];
        auto fetch = [&](int i, int& len, int& blk) {
            len = 0;
            blk = -1;
            if (i >= count) return;
            int seq, kvg, j0;
            coords(i, seq, kvg, j0);
            len = p.context_lens[seq];
            if (j0 + jl < p.max_blocks_per_seq)
                blk = p.block_tables[static_cast<int64_t>(seq) * p.max_blocks_per_seq + j0 + jl];
        };
#pragma unroll
        for (int k = 0; k < kQFetchAhead; ++k) fetch(k, pf_len[k], pf_blk[k]);
        auto finish = [&](int i, int& len, int& pblk) {
            const int b = i & 1;
            int seq, kvg, j0;
            coords(i, seq, kvg, j0);
            const int j = j0 + jl;
            const bool valid = j < nblocks_of(len) && pblk >= 0 && pblk < p.num_blocks;
            fetch(i + kQFetchAhead, len, pblk);
            if (!__all_sync(0xffffffffu, q_wait(&d_full[b], (i >> 1) & 1, abort_flag, p.err))) return false;
            tc::fence_after_sync();
            float best = -INFINITY;
#pragma unroll
            for (int c0 = 0; c0 < N; c0 += 16) {  // columns h*G .. h*G+G-1 are this row's heads
                float v[16];
                tc::TmemLd<16>::load(tmem + (static_cast<uint32_t>(quad * 32) << 16) + b * N + c0, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (c0 + k >= h * G && c0 + k < h * G + G) best = fmaxf(best, v[k]);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_free[b]);
            if (j < p.max_blocks_per_seq)
                p.bounds[(static_cast<int64_t>(seq) * p.num_kv_heads + kvg * 8 + h) * p.max_blocks_per_seq + j] =
                    valid ? best : -INFINITY;
            return true;
        };
        // B = [q- | q+] of the (sequence, group) of item i, rows 8G..N-1 zero
        const int t = threadIdx.x - 64;  // 0..127
        auto write_b = [&](int i) {
            int seq, kvg, j0;
            coords(i, seq, kvg, j0);
            const uint16_t* qrow =
                static_cast<const uint16_t*>(p.q) + (static_cast<int64_t>(seq) * p.num_q_heads + kvg * 8 * G) * D;
            constexpr int PER = N * Cfg::KCH / 128;  // chunks per thread
            uint4 raw[PER];
#pragma unroll
            for (int r = 0; r < PER; ++r) {
                const int idx = r * 128 + t;
                const int n = idx / Cfg::KCH, c = idx % Cfg::KCH;
                const int cc = c >= Cfg::KCH / 2 ? c - Cfg::KCH / 2 : c;
                raw[r] = n < 8 * G ? *reinterpret_cast<const uint4*>(qrow + n * D + cc * 8) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int r = 0; r < PER; ++r) {
                const int idx = r * 128 + t;
                const int n = idx / Cfg::KCH, c = idx % Cfg::KCH;
                uint4 pos, neg;
                split_signs(raw[r], pos, neg);
                *reinterpret_cast<uint4*>(Btile + (n / 8) * Cfg::BSBO + c * 128 + (n % 8) * 16) =
                    c >= Cfg::KCH / 2 ? pos : neg;
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&b_full);
        };
        bool ok = true;
        for (int base = 0; base < count && ok; base += kQFetchAhead) {
#pragma unroll
            for (int k = 0; k < kQFetchAhead; ++k) {  // fetch slot k holds item base + k
                const int i = base + k;
                if (i >= count) break;
                // a new B: the previous item's epilogue saw the last MMAs on the old one complete
                if (new_b(i)) write_b(i);
                if (!(ok = finish(i, pf_len[k], pf_blk[k]))) break;
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) {
        // every copy armed on a stage has landed before the CTA exits: a stage's
        // last arming is its latest phase (no role arms anything past the barrier)
        for (int st = 0; st < NSTG; ++st)
            if (armed[st] >= 0 && !mbar_wait(&full[st], (armed[st] / NSTG) & 1)) atomicOr(p.err, kErrTimeout);
    }
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

// Order-preserving map of a float bound to an unsigned key (larger bound,
// larger key).
__device__ __forceinline__ uint32_t bound_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Selection, step 2: one CTA of 1024 threads per (kv head, sequence) finds the
// budget_blocks largest bounds of its row by radix selection: four passes of
// 8-bit digit histograms in shared memory give the key of the K-th largest
// bound.  Blocks above that key are kept, and blocks equal to it are kept in
// ascending logical order until K are chosen.  One block-wide scan over
// contiguous per-thread ranges places the chosen blocks in logical order.
constexpr int kTopkThreads = 1024;

__global__ void __launch_bounds__(kTopkThreads) quest_topk_kernel(QuestSelectParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int hist[256];
    __shared__ uint32_t warp_scan[kTopkThreads / 32];
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
        if (tid < 256) hist[tid] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        for (int b0 = 0; b0 < nblk; b0 += kTopkThreads) {  // uniform trip count
            const int j = b0 + tid;
            const uint32_t k = j < nblk ? keys[j] : 0u;
            const bool in = j < nblk && (k & mask) == prefix;
            const int digit = in ? static_cast<int>((k >> shift) & 255u) : 256;
            if (shift == 24) {
                // the top byte: a row's bounds share sign and most of the exponent,
                // so equal digits are aggregated per warp
                const unsigned same = __match_any_sync(0xffffffffu, digit);
                if (in && lane == __ffs(same) - 1) atomicAdd(&hist[digit], __popc(same));
            } else if (in) {
                atomicAdd(&hist[digit], 1);  // spread digits, or few keys in the prefix
            }
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
    for (int j = lo; j < hi; ++j) {
        const uint32_t k = keys[j];
        const bool kept = k > kth || (k == kth && eq < ties);
        if (kept) out_row[gt + min(eq, ties)] = blocks[j];
        // exactly budget_blocks blocks are kept, all full but the row's last
        // block: its owner writes the selected token count
        if (j == nblk - 1)
            *out_len = p.budget_blocks * p.block_size - (kept ? p.block_size - (L - j * p.block_size) : 0);
        if (k > kth) ++gt;
        else if (k == kth) ++eq;
    }
}

cudaError_t launch_quest_minmax(const QuestMetaParams& p, int meta, int cache, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(p.num_seqs) * p.max_blocks_per_seq * p.num_kv_heads * (p.head_dim / 8);
    if (total == 0) return cudaSuccess;
    const int blocks = static_cast<int>(total / 256 + 1 < 152 * 32 ? total / 256 + 1 : 152 * 32);
    if (cache == kE4M3) {
        if (meta == kBF16)
            quest_minmax_kernel<kBF16, kE4M3><<<blocks, 256, 0, s>>>(p);
        else
            quest_minmax_kernel<kF16, kE4M3><<<blocks, 256, 0, s>>>(p);
    } else if (meta == kBF16) {
        quest_minmax_kernel<kBF16, kBF16><<<blocks, 256, 0, s>>>(p);
    } else {
        quest_minmax_kernel<kF16, kF16><<<blocks, 256, 0, s>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_quest_append_minmax(const QuestAppendParams& p, int act, int cache, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * (p.head_dim / 8);
    if (total == 0) return cudaSuccess;
    const int blocks = static_cast<int>(total / 256 + 1 < 152 * 16 ? total / 256 + 1 : 152 * 16);
    if (cache == kE4M3) {
        if (act == kBF16)
            quest_append_minmax_kernel<kBF16, kE4M3><<<blocks, 256, 0, s>>>(p);
        else
            quest_append_minmax_kernel<kF16, kE4M3><<<blocks, 256, 0, s>>>(p);
    } else if (act == kBF16) {
        quest_append_minmax_kernel<kBF16, kBF16><<<blocks, 256, 0, s>>>(p);
    } else {
        quest_append_minmax_kernel<kF16, kF16><<<blocks, 256, 0, s>>>(p);
    }
    return cudaGetLastError();
}

namespace {
template <int T, int D, int G>
cudaError_t bounds_one(const QuestSelectParams& p, cudaStream_t s) {
    const int bpi = kQRows / p.group_heads;
    const int64_t items = static_cast<int64_t>(p.num_seqs) * (p.num_kv_heads / p.group_heads) *
                          ((p.max_blocks_per_seq + bpi - 1) / bpi);
    if (items > 0x7fffffff) return cudaErrorInvalidValue;
    constexpr int smem = QBoundsCfg<D>::SMEM;
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
    const int grid = static_cast<int>(items < sms ? items : sms);
    quest_bounds_kernel<T, D, G><<<grid, kQThreads, smem, s>>>(p, items);
    return cudaGetLastError();
}
// Hkv a multiple of 8: the metadata as a 3-D tensor (64 elements; rows,
// 4D bytes apart; 2D/64 atoms, 128 bytes apart) read in 64 x 8 x 2D/64
// boxes, 128-byte swizzled.  False if the driver does not encode it.
template <int D>
bool make_meta_map(CUtensorMap* m, const QuestSelectParams& p, int T) {
    auto fn = encode_fn();
    if (!fn) return false;
    constexpr int NATOM = 2 * D / 64;
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(p.num_blocks) * p.num_kv_heads, NATOM};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(4 * D), 128};
    cuuint32_t box[3] = {64, 8, NATOM};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    return fn(m, T == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<void*>(p.kmeta), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
template <int T, int D, int G>
cudaError_t bounds8_one(const QuestSelectParams& p, const CUtensorMap& m, cudaStream_t s) {
    using Cfg = QBounds8Cfg<D, G>;
    const int64_t items = static_cast<int64_t>(p.num_seqs) * (p.num_kv_heads / 8) *
                          ((p.max_blocks_per_seq + kQ8Blocks - 1) / kQ8Blocks);
    if (items > 0x7fffffff) return cudaErrorInvalidValue;
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || !configured[dev]) {
        e = cudaFuncSetAttribute(quest_bounds8_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) configured[dev] = true;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(items < sms ? items : sms);
    quest_bounds8_kernel<T, D, G><<<grid, kQ8Threads, Cfg::SMEM, s>>>(m, p, items);
    return cudaGetLastError();
}
template <int T, int D>
cudaError_t bounds8_g(const QuestSelectParams& p, const CUtensorMap& m, int G, cudaStream_t s) {
    switch (G) {
        case 1: return bounds8_one<T, D, 1>(p, m, s);
        case 2: return bounds8_one<T, D, 2>(p, m, s);
        case 4: return bounds8_one<T, D, 4>(p, m, s);
        case 8: return bounds8_one<T, D, 8>(p, m, s);
        default: return cudaErrorInvalidValue;
    }
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

cudaError_t launch_quest_select(const QuestSelectParams& p_in, int dtype, int G, cudaStream_t s) {
    if (p_in.num_seqs == 0) return cudaSuccess;
    // kv heads per bound item: the largest power of two dividing Hkv with at
    // most 32 query heads (the MMA's N) and at most 128 rows
    QuestSelectParams p = p_in;
    cudaError_t e;
    CUtensorMap m;
    const bool box8 = p.num_kv_heads % 8 == 0 && G <= 8 &&
                      (p.head_dim == 128 ? make_meta_map<128>(&m, p, dtype) : make_meta_map<64>(&m, p, dtype));
    if (box8) {
        // groups of 8 kv heads: A straight from TMA boxes
        p.group_heads = 8;
        if (dtype == kBF16)
            e = p.head_dim == 128 ? bounds8_g<kBF16, 128>(p, m, G, s) : bounds8_g<kBF16, 64>(p, m, G, s);
        else
            e = p.head_dim == 128 ? bounds8_g<kF16, 128>(p, m, G, s) : bounds8_g<kF16, 64>(p, m, G, s);
    } else {
        int hg = 1;
        while (p.num_kv_heads % (2 * hg) == 0 && 2 * hg * G <= kQMaxN && 2 * hg <= kQRows) hg *= 2;
        p.group_heads = hg;
        if (dtype == kBF16)
            e = p.head_dim == 128 ? bounds_g<kBF16, 128>(p, G, s) : bounds_g<kBF16, 64>(p, G, s);
        else
            e = p.head_dim == 128 ? bounds_g<kF16, 128>(p, G, s) : bounds_g<kF16, 64>(p, G, s);
    }
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
