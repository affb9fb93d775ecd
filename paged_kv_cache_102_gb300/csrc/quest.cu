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

// Selection, step 1: the bound of every (sequence, kv head, logical block),
// one thread per block over all SMs (the bound of a kv head is the largest
// over its G query heads).  Consecutive threads share (sequence, kv head), so
// their query loads are warp-uniform; each reads its block's min and max rows
// with 16-byte loads.  Bounds go to the workspace [B][Hkv][max_blocks].
template <int T, int D, int G>
__global__ void __launch_bounds__(256) quest_bounds_kernel(QuestSelectParams p) {
    const int64_t per_row = p.max_blocks_per_seq;
    const int64_t total = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads * per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int j = static_cast<int>(i % per_row);
        const int64_t r = i / per_row;
        const int kvh = static_cast<int>(r % p.num_kv_heads);
        const int seq = static_cast<int>(r / p.num_kv_heads);
        const int L = p.context_lens[seq];
        if (L < 1 || L > p.max_blocks_per_seq * p.block_size || j * p.block_size >= L) continue;
        const int blk = p.block_tables[static_cast<int64_t>(seq) * p.max_blocks_per_seq + j];
        float best = -INFINITY;
        if (blk < 0 || blk >= p.num_blocks) {
            atomicOr(p.err, kErrBadBlock);
        } else {
            const uint16_t* meta =
                static_cast<const uint16_t*>(p.kmeta) + ((static_cast<int64_t>(blk) * p.num_kv_heads + kvh) * 2) * D;
            const uint16_t* qrow =
                static_cast<const uint16_t*>(p.q) + (static_cast<int64_t>(seq) * p.num_q_heads + kvh * G) * D;
            float u[G];
#pragma unroll
            for (int g = 0; g < G; ++g) u[g] = 0.f;
#pragma unroll 4
            for (int c = 0; c < D; c += 8) {
                float mn[8], mx[8];
                unpack8<T>(*reinterpret_cast<const uint4*>(meta + c), mn);
                unpack8<T>(*reinterpret_cast<const uint4*>(meta + D + c), mx);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float qv[8];
                    unpack8<T>(*reinterpret_cast<const uint4*>(qrow + g * D + c), qv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) u[g] += fmaxf(qv[e] * mn[e], qv[e] * mx[e]);
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) best = fmaxf(best, u[g]);
        }
        p.bounds[i] = best;
    }
}

// Selection, step 2: one CTA per (kv head, sequence) sorts the row's bounds
// (descending bound, ascending logical index on equal bounds) with a bitonic
// network in shared memory, keeps the first budget_blocks and writes them in
// logical order.
template <int NT>
__global__ void __launch_bounds__(NT) quest_topk_kernel(QuestSelectParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int kvh = blockIdx.x;
    const int seq = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = p.context_lens[seq];
    const int32_t* table = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq;
    int32_t* out_row = p.sel_tables + (static_cast<int64_t>(seq) * p.num_kv_heads + kvh) * p.budget_blocks;
    int32_t* out_len = p.sel_lens + static_cast<int64_t>(seq) * p.num_kv_heads + kvh;
    if (L < 1 || L > p.max_blocks_per_seq * p.block_size) {
        if (threadIdx.x == 0) {
            if (kvh == 0) atomicOr(p.err, kErrBadLen);
            *out_len = 0;
        }
        return;
    }
    const int nblk = (L + p.block_size - 1) / p.block_size;
    if (nblk <= p.budget_blocks) {
        for (int j = threadIdx.x; j < p.budget_blocks; j += blockDim.x) out_row[j] = j < nblk ? table[j] : 0;
        if (threadIdx.x == 0) *out_len = L;
        return;
    }
    int n2 = 32;  // power of two >= nblk
    while (n2 < nblk) n2 <<= 1;
    float* U = reinterpret_cast<float*>(smem);
    int* idx = reinterpret_cast<int*>(U + n2);
    unsigned char* chosen = reinterpret_cast<unsigned char*>(idx + n2);
    const float* row = p.bounds + (static_cast<int64_t>(seq) * p.num_kv_heads + kvh) * p.max_blocks_per_seq;
    for (int j = threadIdx.x; j < n2; j += NT) {
        U[j] = j < nblk ? row[j] : -INFINITY;
        idx[j] = j < nblk ? j : 0x7fffffff;
        if (j < nblk) chosen[j] = 0;
    }
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1) {
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            for (int i = threadIdx.x; i < n2; i += NT) {
                const int partner = i ^ jj;
                if (partner > i) {
                    const bool desc = (i & k) == 0;
                    const float ua = U[i], ub = U[partner];
                    const int ia = idx[i], ib = idx[partner];
                    const bool a_first = ua > ub || (ua == ub && ia < ib);
                    if (a_first != desc) {
                        U[i] = ub;
                        U[partner] = ua;
                        idx[i] = ib;
                        idx[partner] = ia;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int r = threadIdx.x; r < p.budget_blocks; r += NT)
        if (idx[r] >= 0 && idx[r] < nblk) chosen[idx[r]] = 1;  // (NaN bounds could misorder the padding)
    __syncthreads();
    if (warp == 0) {
        int base = 0, tokens = 0;
        for (int j0 = 0; j0 < nblk; j0 += 32) {
            const int j = j0 + lane;
            const bool c = j < nblk && chosen[j];
            const unsigned m = __ballot_sync(0xffffffffu, c);
            if (c) {
                out_row[base + __popc(m & ((1u << lane) - 1))] = table[j];
                tokens += j == nblk - 1 ? L - j * p.block_size : p.block_size;
            }
            base += __popc(m);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) tokens += __shfl_xor_sync(0xffffffffu, tokens, off);
        for (int i = base + lane; i < p.budget_blocks; i += 32) out_row[i] = 0;
        if (lane == 0) *out_len = tokens;
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
    const int64_t total = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads * p.max_blocks_per_seq;
    const int blocks = static_cast<int>(total / 256 + 1 < 152 * 64 ? total / 256 + 1 : 152 * 64);
    quest_bounds_kernel<T, D, G><<<blocks, 256, 0, s>>>(p);
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
template <int NT>
cudaError_t topk(const QuestSelectParams& p, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(p.sort_size) * 9;  // bound, index, chosen flag
    auto kern = quest_topk_kernel<NT>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    kern<<<dim3(p.num_kv_heads, p.num_seqs), NT, smem, s>>>(p);
    return cudaGetLastError();
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
    // threads: half the sort size (one compare-exchange each per stage), 32..1024
    if (p.sort_size <= 64) return topk<32>(p, s);
    if (p.sort_size <= 256) return topk<128>(p, s);
    if (p.sort_size <= 1024) return topk<512>(p, s);
    return topk<1024>(p, s);
}

}  // namespace pkv
