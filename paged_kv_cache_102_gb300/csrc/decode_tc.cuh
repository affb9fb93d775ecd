// Paged decode attention for grouped-query heads on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory), sm_103a.
//
// Same result as the CUDA-core kernel (decode.cuh): for sequence b, kv head
// kvh and its G query heads, softmax(scale * q K^T) V over the context,
// gathered block by block through the block table (Ultralytics glossary
// "PagedAttention", section "How paging works"; query heads sharing a KV
// head: section "Related techniques").  When G query heads read the same
// K/V, the step is a real dense product: S = K Q^T is [tokens x G] and
// O = V^T P is [D x G], so it runs on the tensor cores and the K/V bytes are
// read once for all G heads.
//
// Work item: (sequence, kv head, partition of up to 512 tokens).  The kernel
// is persistent: each CTA walks items blockIdx.x, blockIdx.x + gridDim.x, ...
// Roles (192 threads):
//  warp 0   producer: table entries -> 2-D TMA loads (128-byte swizzle) of
//           each (block, kv head) tile, two 64-column halves of head_dim,
//           into a ring of 128-token stages; K tiles of an item, then its V
//           tiles; Q rows of the item's G heads.
//  warp 1   MMA: allocates tensor memory; S[t][h] = sum_d K[t][d] Q[h][d]
//           with M = 128 tokens, N = 16 (G heads, padded), K = 128 (D), one
//           16-column slot per tile; then O[d][h] = sum_t V[t][d] P[t][h]
//           with M = 128 (D), N = 16, K = tokens.
//  warps 2-5 softmax + epilogue: thread i owns tensor-memory lane i (token i
//           of each tile for S, dimension i of O).  They take the
//           partition-wide max and sum per head (no online rescaling: the
//           whole partition's scores sit in tensor memory), write P in bf16
//           (or f16) in the MMA's shared-memory layout, and finally write the
//           output (one partition) or the split-K partial (m, l, O/l).
// All barrier waits are bounded (kWaitLimitNs); on a timeout the CTA stops
// issuing work, drains its in-flight copies and MMAs, frees tensor memory and
// reports kErrTimeout.
#pragma once

#include "kernels.h"
#include "pkv_tc.cuh"

namespace pkv {

constexpr int kTcThreads = 192;
constexpr int kTcTile = 128;        // tokens per tile (MMA M of S = K Q^T)
constexpr int kTcMaxTiles = 4;      // tiles per item: partitions of at most 512 tokens
constexpr int kTcD = 128;           // head_dim served by this kernel
constexpr int kTcN = 16;            // MMA N: query heads padded to 16
constexpr int kTcHalf = kTcTile * 128;       // one 64-column half of a tile: 128 rows x 128 bytes
constexpr int kTcStage = 2 * kTcHalf;        // 32 KB
constexpr int kTcQBytes = 2 * kTcN * 128;    // 4 KB
constexpr int kTcPTile = 2 * kTcN * 128;     // P of one tile: 2 token halves x 16 rows x 128 bytes
constexpr int kTcTmemCols = 128;             // S: 4 x 16 columns, O: 16 columns
constexpr int kTcOCol = kTcMaxTiles * kTcN;  // 64

template <int NS>
struct TcSmem {
    static constexpr int RING = 0;
    static constexpr int Q = NS * kTcStage;
    static constexpr int P = Q + kTcQBytes;
    static constexpr int BARS = P + kTcMaxTiles * kTcPTile;
    // full[NS], empty[NS], q_full, q_empty, s_full, p_full, o_full, tmem_free, final
    static constexpr int NBARS = 2 * NS + 7;
    static constexpr int RED = BARS + NBARS * 8;
    static constexpr int RED_FLOATS = 2 * 4 * 8;  // red_max[4][8], red_sum[4][8]
    static constexpr int MISC = RED + RED_FLOATS * 4;  // tmem base, abort flag
    static constexpr int BYTES = MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024
};

struct TcItem {
    int seq, kvh, part, tok_begin, n_tok, n_tiles;
};

__device__ __forceinline__ bool tc_item(int idx, const DecodeParams& p, int BS, TcItem& it) {
    it.part = idx % p.max_parts;
    const int rest = idx / p.max_parts;
    it.kvh = rest % p.num_kv_heads;
    it.seq = rest / p.num_kv_heads;
    const int L = p.context_lens[it.seq];
    if (L < 1 || L > p.max_blocks_per_seq * BS) return false;
    it.tok_begin = it.part * p.partition_size;
    if (it.tok_begin >= L) return false;
    it.n_tok = min(p.partition_size, L - it.tok_begin);
    it.n_tiles = (it.n_tok + kTcTile - 1) / kTcTile;
    return true;
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

// Named barrier over `count` threads that also ORs a predicate across them.
__device__ __forceinline__ int named_bar_or(int id, int count, int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.b32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred), "r"(id), "r"(count)
        : "memory");
    return r;
}

template <int ACT, int BS, int G, int NS>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const __grid_constant__ CUtensorMap qmap, const DecodeParams p) {
    using S = TcSmem<NS>;
    constexpr int BPT = kTcTile / BS;  // blocks per tile
    constexpr uint32_t IDESC_S = tc::idesc_f16(128, kTcN, ACT == kBF16, false, false);
    constexpr uint32_t IDESC_O = tc::idesc_f16(128, kTcN, ACT == kBF16, true, false);
    static_assert(G == 2 || G == 4 || G == 8, "query heads per kv head");
    static_assert(kTcMaxTiles * kTcTile / BS <= 32, "one warp holds the table entries of an item");

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* ring = sm + S::RING;
    unsigned char* qbuf = sm + S::Q;
    unsigned char* pbuf = sm + S::P;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::BARS);
    uint64_t* full = bars;
    uint64_t* empty = bars + NS;
    uint64_t* q_full = bars + 2 * NS;
    uint64_t* q_empty = q_full + 1;
    uint64_t* s_full = q_full + 2;
    uint64_t* p_full = q_full + 3;
    uint64_t* o_full = q_full + 4;
    uint64_t* tmem_free = q_full + 5;
    uint64_t* final_bar = q_full + 6;
    float* red_max = reinterpret_cast<float*>(sm + S::RED);
    float* red_sum = red_max + 32;
    uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(sm + S::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + S::MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total_items = p.num_seqs * p.num_kv_heads * p.max_parts;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 7; ++i) mbar_init(&q_full[i], 1);
        *abort_flag = 0;
        mbar_init_fence();
        tc::prefetch_tensormap(&kmap);
        tc::prefetch_tensormap(&vmap);
        tc::prefetch_tensormap(&qmap);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_base_smem, kTcTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_base_smem;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        const uint64_t policy = l2_policy_evict_first();
        uint32_t use = 0;  // stage uses issued so far
        int qn = 0;        // items whose Q was loaded
        for (int idx = blockIdx.x; idx < total_items; idx += gridDim.x) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            TcItem it;
            if (!tc_item(idx, p, BS, it)) {
                if (lane == 0 && it.part == 0 && it.kvh == 0) {
                    const int L = p.context_lens[it.seq];
                    if (L < 1 || L > p.max_blocks_per_seq * BS) atomicOr(p.err, kErrBadLen);
                }
                continue;
            }
            const int n_blk = (it.n_tok + BS - 1) / BS;
            int phys = -1;
            if (lane < n_blk) {
                phys = p.block_tables[static_cast<size_t>(it.seq) * p.max_blocks_per_seq + it.tok_begin / BS + lane];
                if (phys < 0 || phys >= p.num_blocks) {
                    atomicOr(p.err, kErrBadBlock);
                    phys = -1;
                }
            }
            bool ok = true;
            if (lane == 0) {
                if (qn > 0) ok = tc_wait(q_empty, (qn - 1) & 1, abort_flag, p.err);
                if (ok) {
                    mbar_arrive_expect_tx(q_full, 2 * G * 128);
                    const int row = it.seq * p.num_q_heads + it.kvh * G;
                    tc::tma_load_2d(qbuf, &qmap, 0, row, q_full, policy);
                    tc::tma_load_2d(qbuf + kTcN * 128, &qmap, 64, row, q_full, policy);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ++qn;
            for (int pass = 0; pass < 2 && ok; ++pass) {
                const CUtensorMap* map = pass == 0 ? &kmap : &vmap;
                for (int t = 0; t < it.n_tiles && ok; ++t) {
                    int pb[BPT];
#pragma unroll
                    for (int j = 0; j < BPT; ++j) pb[j] = __shfl_sync(0xffffffffu, phys, (t * BPT + j) & 31);
                    if (lane == 0) {
                        const int s = use % NS;
                        if (use >= NS) ok = tc_wait(&empty[s], ((use / NS) - 1) & 1, abort_flag, p.err);
                        if (ok) {
                            uint32_t bytes = 0;
#pragma unroll
                            for (int j = 0; j < BPT; ++j)
                                if (t * BPT + j < n_blk && pb[j] >= 0) bytes += BS * 256;
                            mbar_arrive_expect_tx(&full[s], bytes);
                            unsigned char* st = ring + s * kTcStage;
#pragma unroll
                            for (int j = 0; j < BPT; ++j) {
                                if (t * BPT + j < n_blk && pb[j] >= 0) {
                                    const int y = (pb[j] * p.num_kv_heads + it.kvh) * BS;
                                    tc::tma_load_2d(st + j * BS * 128, map, 0, y, &full[s], policy);
                                    tc::tma_load_2d(st + kTcHalf + j * BS * 128, map, 64, y, &full[s], policy);
                                }
                            }
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (ok) ++use;  // only stages actually armed are drained below
                }
            }
            if (!ok) break;
        }
        // Leave only when every copy into this CTA's shared memory has landed.
        if (lane == 0) {
            const uint32_t first = use > static_cast<uint32_t>(NS) ? use - NS : 0;
            for (uint32_t u = first; u < use; ++u)
                if (!mbar_wait(&full[u % NS], (u / NS) & 1)) atomicOr(p.err, kErrTimeout);
            if (qn > 0 && !mbar_wait(q_full, (qn - 1) & 1)) atomicOr(p.err, kErrTimeout);
        }
    } else if (warp == 1) {
        // --------------------------------------------------------------------- MMA
        uint32_t use = 0;
        int n = 0;  // valid items processed
        for (int idx = blockIdx.x; idx < total_items; idx += gridDim.x) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            TcItem it;
            if (!tc_item(idx, p, BS, it)) continue;
            bool ok = true;
            if (lane == 0) {
                ok = tc_wait(q_full, n & 1, abort_flag, p.err);
                if (ok && n > 0) ok = tc_wait(tmem_free, (n - 1) & 1, abort_flag, p.err);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc::fence_after_sync();
            // S = K Q^T, one 16-column slot per tile
            for (int t = 0; t < it.n_tiles && ok; ++t) {
                const int s = use % NS;
                if (lane == 0) ok = tc_wait(&full[s], (use / NS) & 1, abort_flag, p.err);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t kb = smem_addr(ring + s * kTcStage);
                    const uint32_t qb = smem_addr(qbuf);
#pragma unroll
                    for (int k = 0; k < kTcD / 16; ++k) {
                        const uint32_t off = (k >> 2) * kTcHalf + (k & 3) * 32;
                        const uint32_t qoff = (k >> 2) * (kTcN * 128) + (k & 3) * 32;
                        tc::mma_f16(tmem + t * kTcN, tc::desc_sw128(kb + off, 16, 1024),
                                    tc::desc_sw128(qb + qoff, 16, 1024), IDESC_S, k > 0);
                    }
                    tc::commit(&empty[s]);
                }
                __syncwarp();
                ++use;
            }
            if (!ok) break;
            if (lane == 0) {
                tc::commit(q_empty);
                tc::commit(s_full);
                ok = tc_wait(p_full, n & 1, abort_flag, p.err);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc::fence_after_sync();
            // O = V^T P over the item's tiles
            for (int t = 0; t < it.n_tiles && ok; ++t) {
                const int s = use % NS;
                ok = __all_sync(0xffffffffu, tc_wait(&full[s], (use / NS) & 1, abort_flag, p.err));
                if (!ok) break;
                unsigned char* vb = ring + s * kTcStage;
                const int valid = min(kTcTile, it.n_tok - t * kTcTile);
                const int ksteps = (valid + 15) / 16;
                // rows past the context inside the last 16-token step: zero them so
                // that unwritten pool slots cannot leak NaN through P = 0
                const int zero_rows = ksteps * 16 - valid;
                if (zero_rows > 0) {
                    for (int i = lane; i < zero_rows * 16; i += 32) {
                        const int r = valid + (i >> 4);
                        const int c = i & 15;  // 16-byte chunk of the 256-byte row (two halves)
                        unsigned char* dst = vb + (c >> 3) * kTcHalf + r * 128 + (c & 7) * 16;
                        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                }
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t vaddr = smem_addr(vb);
                    const uint32_t pb = smem_addr(pbuf + t * kTcPTile);
                    for (int j = 0; j < ksteps; ++j) {
                        const uint32_t poff = (j >> 2) * (kTcN * 128) + (j & 3) * 32;
                        tc::mma_f16(tmem + kTcOCol, tc::desc_sw128(vaddr + j * 2048, kTcHalf, 1024),
                                    tc::desc_sw128(pb + poff, 16, 1024), IDESC_O, (t > 0 || j > 0) ? 1u : 0u);
                    }
                    tc::commit(&empty[s]);
                }
                __syncwarp();
                ++use;
            }
            if (!ok) break;
            if (lane == 0) tc::commit(o_full);
            __syncwarp();
            ++n;
        }
        // every MMA this thread issued has completed before tensor memory is freed
        if (lane == 0) {
            tc::commit(final_bar);
            if (!mbar_wait(final_bar, 0)) atomicOr(p.err, kErrTimeout);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ softmax + epilogue
        const int q4 = warp & 3;         // tensor-memory lane quarter of this warp
        const int row = q4 * 32 + lane;  // token of each tile (S) / dimension d (O)
        const int tid = threadIdx.x - 64;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
        int n = 0;
        for (int idx = blockIdx.x; idx < total_items; idx += gridDim.x) {
            TcItem it;
            if (!tc_item(idx, p, BS, it)) continue;
            // Every wait below is followed by a barrier that all 128 threads
            // reach; a failure is OR-reduced there so that the four warps
            // leave together and no named barrier is left waiting.
            bool ok = __all_sync(0xffffffffu, tc_wait(s_full, n & 1, abort_flag, p.err));
            float sc[kTcMaxTiles][G] = {};
            if (ok) {
                tc::fence_after_sync();
#pragma unroll
                for (int t = 0; t < kTcMaxTiles; ++t)
                    if (t < it.n_tiles) tc::TmemLd<G>::load(lane_addr + t * kTcN, sc[t]);
                tc::tmem_wait_ld();
                float mx[G];
#pragma unroll
                for (int g = 0; g < G; ++g) mx[g] = -INFINITY;
#pragma unroll
                for (int t = 0; t < kTcMaxTiles; ++t) {
                    const bool valid = t < it.n_tiles && t * kTcTile + row < it.n_tok;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        sc[t][g] = valid ? sc[t][g] * p.scale_log2 : -INFINITY;
                        mx[g] = fmaxf(mx[g], sc[t][g]);
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1)
                        mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], off));
                }
                if (lane == 0) {
#pragma unroll
                    for (int g = 0; g < G; ++g) red_max[q4 * 8 + g] = mx[g];
                }
            }
            if (named_bar_or(1, 128, !ok)) break;
            float M[G], sum[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                M[g] = fmaxf(fmaxf(red_max[g], red_max[8 + g]), fmaxf(red_max[16 + g], red_max[24 + g]));
                sum[g] = 0.f;
            }
#pragma unroll
            for (int t = 0; t < kTcMaxTiles; ++t) {
                if (t < it.n_tiles) {
                    unsigned char* pt = pbuf + t * kTcPTile + (row >> 6) * (kTcN * 128);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float pv = sc[t][g] == -INFINITY ? 0.f : exp2f(sc[t][g] - M[g]);
                        sum[g] += pv;
                        const int chunk = ((row & 63) >> 3) ^ (g & 7);
                        *reinterpret_cast<uint16_t*>(pt + g * 128 + chunk * 16 + (row & 7) * 2) = float_to_act<ACT>(pv);
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) sum[g] += __shfl_xor_sync(0xffffffffu, sum[g], off);
            }
            if (lane == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) red_sum[q4 * 8 + g] = sum[g];
            }
            tc::fence_proxy_async_smem();
            asm volatile("bar.sync 2, 128;" ::: "memory");
            float Lsum[G];
#pragma unroll
            for (int g = 0; g < G; ++g) Lsum[g] = red_sum[g] + red_sum[8 + g] + red_sum[16 + g] + red_sum[24 + g];
            if (tid == 0) mbar_arrive(p_full);

            ok = __all_sync(0xffffffffu, tc_wait(o_full, n & 1, abort_flag, p.err));
            float o[G];
            if (ok) {
                tc::fence_after_sync();
                tc::TmemLd<G>::load(lane_addr + kTcOCol, o);
                tc::tmem_wait_ld();
                tc::fence_before_sync();
            }
            if (named_bar_or(1, 128, !ok)) break;
            if (tid == 0) mbar_arrive(tmem_free);

            const int d = row;
            const bool single = p.max_parts == 1 || p.context_lens[it.seq] <= p.partition_size;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float val = o[g] / Lsum[g];
                const size_t hrow = static_cast<size_t>(it.seq) * p.num_q_heads + it.kvh * G + g;
                if (single) {
                    static_cast<uint16_t*>(p.out)[hrow * kTcD + d] = float_to_act<ACT>(val);
                } else {
                    const size_t slot = hrow * p.max_parts + it.part;
                    p.ws_o[slot * kTcD + d] = val;
                    if (d == 0) {
                        p.ws_ml[slot * 2] = M[g];
                        p.ws_ml[slot * 2 + 1] = Lsum[g];
                    }
                }
            }
            ++n;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, kTcTmemCols);
}

}  // namespace pkv
