// Instantiates the partition kernel for one (activation, cache) type pair
// over head_dim {64, 128}, block_size {16, 32}, group {1, 2, 4, 8}.
// Include after defining PKV_ACT, PKV_CACHE and PKV_LAUNCH_NAME.
#include "decode.cuh"

namespace pkv {

namespace {

template <int D, int BS, int G>
cudaError_t launch_one(const DecodeParams& p, cudaStream_t s) {
    using C = DecodeCfg<PKV_CACHE, D, BS, G>;
    auto kern = paged_decode_partition_kernel<PKV_ACT, PKV_CACHE, D, BS, G>;
    static bool configured[kMaxDevices] = {};  // shared-memory attribute set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    dim3 grid(p.max_parts, p.num_kv_heads, p.num_seqs);
    kern<<<grid, kDecodeThreads, C::SMEM_BYTES, s>>>(p);
    return cudaGetLastError();
}

template <int D, int BS>
cudaError_t by_group(const DecodeParams& p, int G, cudaStream_t s) {
    switch (G) {
        case 1: return launch_one<D, BS, 1>(p, s);
        case 2: return launch_one<D, BS, 2>(p, s);
        case 4: return launch_one<D, BS, 4>(p, s);
        case 8: return launch_one<D, BS, 8>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t PKV_LAUNCH_NAME(const DecodeParams& p, int D, int BS, int G, cudaStream_t s) {
    if (D == 64 && BS == 16) return by_group<64, 16>(p, G, s);
    if (D == 64 && BS == 32) return by_group<64, 32>(p, G, s);
    if (D == 128 && BS == 16) return by_group<128, 16>(p, G, s);
    if (D == 128 && BS == 32) return by_group<128, 32>(p, G, s);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
