// Tensor-core grouped-query decode for E4M3 caches: kernel instantiations and
// their launch.  A translation unit of their own, so that the 16-bit
// instantiations (decode_tc.cu) do not move these in the module.
#include "decode_tc_host.cuh"

namespace pkv {

namespace {

// E4M3 cache: 16 KB stages; ten at one CTA per SM (variant 0), else five (or
// four, when the per-row tables leave no room) at two CTAs per SM.
template <int ACT>
cudaError_t launch_fp8(const DecodeParams& p, const CUtensorMap& km, const CUtensorMap& vm, int BS, int G,
                       int variant, bool five, cudaStream_t s) {
    if (variant == 0) return by_shape<ACT, kE4M3, 10>(p, km, vm, km, BS, G, 1, s);
    if (five) return by_shape<ACT, kE4M3, 5>(p, km, vm, km, BS, G, 2, s);
    return by_shape<ACT, kE4M3, 4>(p, km, vm, km, BS, G, 2, s);
}

}  // namespace

cudaError_t launch_decode_tc_e4m3(const DecodeParams& p, int act, int BS, int G, int variant, cudaStream_t s) {
    const int rows = p.table_kvh_stride != 0 ? p.num_seqs * p.num_kv_heads : p.num_seqs;
    const uint64_t cache_rows = static_cast<uint64_t>(p.num_blocks) * p.num_kv_heads * BS;
    CUtensorMap km, vm;
    if (!make_map8(&km, p.k_cache, cache_rows, BS) || !make_map8(&vm, p.v_cache, cache_rows, BS))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(p.work_counter, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
    const bool five = 2 * (TcSmem<5, kTcStage8>::alloc(rows) + 1024) <= kTcSmemPerSm;
    return act == kBF16 ? launch_fp8<kBF16>(p, km, vm, BS, G, variant, five, s)
                        : launch_fp8<kF16>(p, km, vm, BS, G, variant, five, s);
}

}  // namespace pkv
