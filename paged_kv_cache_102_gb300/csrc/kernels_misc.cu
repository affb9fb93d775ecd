// Slot-mapped KV append, copy-on-write block copy and the split-K merge.
#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

// ---------------------------------------------------------------------------
// Append (Ultralytics glossary "PagedAttention", section "How paging works":
// the key of position pos goes to block table[pos // bs], offset pos % bs).
// One thread per 8-element chunk of one (token, kv head) row, grid-stride.
// Same type: one 16-byte load and store per chunk for K and for V (bit copy).
// E4M3 cache: x / scale in binary32 (correctly rounded division), converted
// with round-to-nearest-even and saturation to +-448.
// ---------------------------------------------------------------------------
template <int ACT, int CACHE>
__global__ void __launch_bounds__(256) paged_kv_append_kernel(AppendParams p) {
    const int chunks_per_row = p.head_dim / 8;
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * chunks_per_row;
    const int64_t num_slots = static_cast<int64_t>(p.num_blocks) * p.block_size;
    float ks = 1.f, vs = 1.f;
    if (CACHE == kE4M3) {
        ks = *p.k_scale;
        vs = *p.v_scale;
    }
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t th, t, blk;  // th = token * Hkv + head
        int c, h, off;
        divmod_u(i, chunks_per_row, th, c);
        divmod_u(th, p.num_kv_heads, t, h);
        const int64_t slot = p.slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            atomicOr(p.err, kErrBadSlot);
            continue;
        }
        divmod_u(slot, p.block_size, blk, off);
        const int64_t dst = ((blk * p.num_kv_heads + h) * p.block_size + off) * p.head_dim + c * 8;
        const int64_t src = th * p.head_dim + c * 8;
        const uint4 kin = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k) + src);
        const uint4 vin = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.v) + src);
        if (CACHE == ACT) {
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.k_cache) + dst) = kin;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.v_cache) + dst) = vin;
        } else {
            const uint16_t* ke = reinterpret_cast<const uint16_t*>(&kin);
            const uint16_t* ve = reinterpret_cast<const uint16_t*>(&vin);
            uint8_t kq[8], vq[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                kq[j] = __nv_cvt_float_to_fp8(__fdiv_rn(act_to_float<ACT>(ke[j]), ks), __NV_SATFINITE, __NV_E4M3);
                vq[j] = __nv_cvt_float_to_fp8(__fdiv_rn(act_to_float<ACT>(ve[j]), vs), __NV_SATFINITE, __NV_E4M3);
            }
            *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.k_cache) + dst) = *reinterpret_cast<const uint2*>(kq);
            *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.v_cache) + dst) = *reinterpret_cast<const uint2*>(vq);
        }
    }
}

cudaError_t launch_append(const AppendParams& p, int act, int cache, cudaStream_t stream) {
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * (p.head_dim / 8);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t want = (total + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 152 * 16 ? want : 152 * 16);
    if (act == kF16 && cache == kF16)
        paged_kv_append_kernel<kF16, kF16><<<blocks, threads, 0, stream>>>(p);
    else if (act == kBF16 && cache == kBF16)
        paged_kv_append_kernel<kBF16, kBF16><<<blocks, threads, 0, stream>>>(p);
    else if (act == kF16 && cache == kE4M3)
        paged_kv_append_kernel<kF16, kE4M3><<<blocks, threads, 0, stream>>>(p);
    else if (act == kBF16 && cache == kE4M3)
        paged_kv_append_kernel<kBF16, kE4M3><<<blocks, threads, 0, stream>>>(p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Copy-on-write block copy (iThome "how to store the KV cache", section
// "Copy-on-Write": the new block receives a copy of the old block's
// contents).  grid.x = pair, grid.y = 16 KB chunk of the block; 16-byte
// vectors, K and V.
// ---------------------------------------------------------------------------
constexpr int kCopyChunkBytes = 16384;

__global__ void __launch_bounds__(256) paged_block_copy_kernel(CopyParams p) {
    const int pair = blockIdx.x;
    const int src = p.pairs[2 * pair];
    const int dst = p.pairs[2 * pair + 1];
    if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) atomicOr(p.err, kErrBadPair);
        return;
    }
    const size_t begin = static_cast<size_t>(blockIdx.y) * kCopyChunkBytes;
    const size_t end = min(begin + kCopyChunkBytes, p.block_bytes);
    const size_t so = static_cast<size_t>(src) * p.block_bytes;
    const size_t d0 = static_cast<size_t>(dst) * p.block_bytes;
    const unsigned char* ks = static_cast<const unsigned char*>(p.k_cache) + so;
    const unsigned char* vs = static_cast<const unsigned char*>(p.v_cache) + so;
    unsigned char* kd = static_cast<unsigned char*>(p.k_cache) + d0;
    unsigned char* vd = static_cast<unsigned char*>(p.v_cache) + d0;
    for (size_t o = begin + threadIdx.x * 16; o < end; o += blockDim.x * 16) {
        const uint4 a = *reinterpret_cast<const uint4*>(ks + o);
        const uint4 b = *reinterpret_cast<const uint4*>(vs + o);
        *reinterpret_cast<uint4*>(kd + o) = a;
        *reinterpret_cast<uint4*>(vd + o) = b;
    }
}

cudaError_t launch_block_copy(const CopyParams& p, int num_pairs, cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    const unsigned chunks = static_cast<unsigned>((p.block_bytes + kCopyChunkBytes - 1) / kCopyChunkBytes);
    paged_block_copy_kernel<<<dim3(num_pairs, chunks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Block swap (PagedAttention notes, section "Preemption": swapping moves the
// KV cache of a sequence that is not running to CPU DRAM and brings it back
// later).  One launch gathers (out) or scatters (in) whole physical blocks,
// K and V, between the pools and a staging buffer [n][K block, V block]
// that may live in pinned host memory: the kernel reads or writes it
// directly, so scattered small blocks cost no per-copy overhead.
// grid.x = block i of the list, grid.y = 16 KB chunk of the block.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) paged_block_swap_kernel(SwapParams p) {
    const int i = blockIdx.x;
    const int b = p.block_ids[i];
    if (b < 0 || b >= p.num_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) atomicOr(p.err, kErrBadPair);
        return;
    }
    const size_t begin = static_cast<size_t>(blockIdx.y) * kCopyChunkBytes;
    const size_t end = min(begin + kCopyChunkBytes, p.block_bytes);
    unsigned char* kd = static_cast<unsigned char*>(p.k_cache) + static_cast<size_t>(b) * p.block_bytes;
    unsigned char* vd = static_cast<unsigned char*>(p.v_cache) + static_cast<size_t>(b) * p.block_bytes;
    unsigned char* ks = static_cast<unsigned char*>(p.staging) + static_cast<size_t>(i) * 2 * p.block_bytes;
    unsigned char* vs = ks + p.block_bytes;
    for (size_t o = begin + threadIdx.x * 16; o < end; o += blockDim.x * 16) {
        if (p.to_staging) {
            const uint4 a = *reinterpret_cast<const uint4*>(kd + o);
            const uint4 c = *reinterpret_cast<const uint4*>(vd + o);
            *reinterpret_cast<uint4*>(ks + o) = a;
            *reinterpret_cast<uint4*>(vs + o) = c;
        } else {
            const uint4 a = *reinterpret_cast<const uint4*>(ks + o);
            const uint4 c = *reinterpret_cast<const uint4*>(vs + o);
            *reinterpret_cast<uint4*>(kd + o) = a;
            *reinterpret_cast<uint4*>(vd + o) = c;
        }
    }
}

cudaError_t launch_block_swap(const SwapParams& p, int n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const unsigned chunks = static_cast<unsigned>((p.block_bytes + kCopyChunkBytes - 1) / kCopyChunkBytes);
    paged_block_swap_kernel<<<dim3(n, chunks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Split-K merge.  Each partition p of a sequence left (m_p, l_p, o_p) with
// o_p already divided by l_p and m_p in log2 units; the full softmax is
//   out = sum_p w_p o_p / sum_p w_p,  w_p = l_p * 2^(m_p - max_p m_p).
// W warps per (sequence, query head) row (1 when there are enough rows to fill
// the GPU, else 2, 4 or 8 from the largest partition count), 8 warps per CTA.  Every warp of a row reads the
// partitions' (m, l) pairs with its lanes in parallel and reduces their max
// with shuffles; warp j then sums partitions j, j+W, ... over its lane's D/32
// output channels with independent vector loads, and the row's warps combine
// their sums through shared memory.  Rows that fit one partition were written
// directly by the partition kernel.  The kernel is launched as a programmatic
// dependent of the partition kernel: griddepcontrol.wait returns once that
// grid has completed and its writes are visible.
// ---------------------------------------------------------------------------
constexpr int kMergeWarps = 8;

template <int ACT, int D, int W>
__global__ void __launch_bounds__(32 * kMergeWarps) paged_decode_merge_kernel(MergeParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int V = D / 32;  // channels per lane
    constexpr int ROWS = kMergeWarps / W;
    __shared__ float s_acc[W > 1 ? kMergeWarps : 1][D];
    __shared__ float s_den[kMergeWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = warp % W;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * ROWS + warp / W;
    bool active = row < static_cast<int64_t>(p.num_seqs) * p.num_q_heads;
    int n_parts = 0;
    if (active) {
        int64_t seq64;
        int h;
        divmod_u(row, p.num_q_heads, seq64, h);
        const int seq = static_cast<int>(seq64);
        const int L =
            p.context_lens[static_cast<int64_t>(seq) * p.lens_seq_stride + (h / p.group) * p.lens_kvh_stride];
        // a bad length was flagged by the partition kernel; one partition was written directly
        active = L >= 1 && L <= p.max_context;
        n_parts = active ? (L + p.partition_size - 1) / p.partition_size : 0;
        active = n_parts > 1;
    }
    float acc[V] = {};
    float den = 0.f;
    if (active && W == 1 && n_parts <= 32) {
        // One round trip for up to 16 partitions: part `lane`'s (max, sum) and
        // the first 16 partial vectors are all loaded before any is used.
        constexpr int C = 16;
        const float* ml = p.ws_ml + row * p.max_parts * 2;
        const float* o = p.ws_o + row * p.max_parts * D + lane * V;
        const float2 a =
            lane < n_parts ? *reinterpret_cast<const float2*>(ml + 2 * lane) : make_float2(-INFINITY, 0.f);
        float x[C][V];
#pragma unroll
        for (int k = 0; k < C; ++k) {
            if (k < n_parts) {
                if constexpr (V == 4) {
                    const float4 t = *reinterpret_cast<const float4*>(o + static_cast<int64_t>(k) * D);
                    x[k][0] = t.x;
                    x[k][1] = t.y;
                    x[k][2] = t.z;
                    x[k][3] = t.w;
                } else {
                    const float2 t = *reinterpret_cast<const float2*>(o + static_cast<int64_t>(k) * D);
                    x[k][0] = t.x;
                    x[k][1] = t.y;
                }
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) x[k][v] = 0.f;
            }
        }
        float M = a.x;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float w = lane < n_parts ? a.y * exp2f(a.x - M) : 0.f;
        den = w;
#pragma unroll
        for (int k = 0; k < C; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, k);
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] = fmaf(wk, x[k][v], acc[v]);
        }
        for (int k = C; k < n_parts; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, k);
            const float* src = o + static_cast<int64_t>(k) * D;
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] = fmaf(wk, src[v], acc[v]);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    } else if (active) {
        const float* ml = p.ws_ml + row * p.max_parts * 2;
        const float* o = p.ws_o + row * p.max_parts * D + lane * V;
        float M = -INFINITY;
        for (int i = lane; i < n_parts; i += 32) M = fmaxf(M, ml[2 * i]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        for (int base = 0; base < n_parts; base += 32) {
            const int i = base + lane;
            const float w = i < n_parts ? ml[2 * i + 1] * exp2f(ml[2 * i] - M) : 0.f;
            if (lane % W == sub) den += w;  // base is a multiple of W
            const int cnt = min(32, n_parts - base);
#pragma unroll 4
            for (int k = sub; k < cnt; k += W) {
                const float wk = __shfl_sync(0xffffffffu, w, k);
                const float* src = o + static_cast<int64_t>(base + k) * D;
                if constexpr (V == 4) {
                    const float4 x = *reinterpret_cast<const float4*>(src);
                    acc[0] = fmaf(wk, x.x, acc[0]);
                    acc[1] = fmaf(wk, x.y, acc[1]);
                    acc[2] = fmaf(wk, x.z, acc[2]);
                    acc[3] = fmaf(wk, x.w, acc[3]);
                } else {
                    const float2 x = *reinterpret_cast<const float2*>(src);
                    acc[0] = fmaf(wk, x.x, acc[0]);
                    acc[1] = fmaf(wk, x.y, acc[1]);
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    }
    if constexpr (W > 1) {
#pragma unroll
        for (int v = 0; v < V; ++v) s_acc[warp][lane * V + v] = acc[v];
        if (lane == 0) s_den[warp] = den;
        __syncthreads();
        if (!active || sub != 0) return;
#pragma unroll
        for (int j = 1; j < W; ++j) {
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] += s_acc[warp + j][lane * V + v];
            den += s_den[warp + j];
        }
    }
    if (!active) return;
    uint16_t* dst = static_cast<uint16_t*>(p.out) + row * D + lane * V;
#pragma unroll
    for (int v = 0; v < V; ++v) dst[v] = float_to_act<ACT>(acc[v] / den);
}

template <int ACT, int D, int W>
cudaError_t merge_one(const MergeParams& p, cudaStream_t stream) {
    constexpr int ROWS = kMergeWarps / W;
    const int64_t rows = static_cast<int64_t>(p.num_seqs) * p.num_q_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + ROWS - 1) / ROWS));
    cfg.blockDim = dim3(32 * kMergeWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, paged_decode_merge_kernel<ACT, D, W>, p);
}

template <int ACT, int D>
cudaError_t merge_w(const MergeParams& p, cudaStream_t stream) {
    // enough rows to fill the GPU with one warp each: no cross-warp combine
    if (static_cast<int64_t>(p.num_seqs) * p.num_q_heads >= 4096) return merge_one<ACT, D, 1>(p, stream);
    if (p.max_parts >= 32) return merge_one<ACT, D, 8>(p, stream);
    if (p.max_parts >= 8) return merge_one<ACT, D, 4>(p, stream);
    if (p.max_parts >= 4) return merge_one<ACT, D, 2>(p, stream);
    return merge_one<ACT, D, 1>(p, stream);
}

// Bounded-wait check: nothing arrives on the barrier, so the wait must give
// up after limit_ns and report kErrTimeout.
__global__ void selftest_wait_kernel(uint64_t limit_ns, int* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_for(&bar, 0, limit_ns)) atomicOr(err, kErrTimeout);
}

cudaError_t launch_selftest_wait(uint64_t limit_ns, int* err, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
    return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams& p, int act, cudaStream_t stream) {
    if (p.num_seqs == 0) return cudaSuccess;
    if (p.head_dim == 128) return act == kF16 ? merge_w<kF16, 128>(p, stream) : merge_w<kBF16, 128>(p, stream);
    return act == kF16 ? merge_w<kF16, 64>(p, stream) : merge_w<kBF16, 64>(p, stream);
}

}  // namespace pkv
