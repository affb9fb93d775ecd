// Tensor-core grouped-query decode at head_dim 64 (16-bit caches, tables
// shared by a sequence's kv heads): kernel instantiations and their launch.
// Each item covers two kv heads, laid side by side as one 128-wide head.
#include "decode_tc_host.cuh"

namespace pkv {

cudaError_t launch_decode_tc_d64(const DecodeParams& p, int act, int BS, int G, int variant, cudaStream_t s) {
    if (p.table_kvh_stride != 0 || p.num_kv_heads % 2 != 0) return cudaErrorInvalidValue;
    const uint64_t cache_rows = static_cast<uint64_t>(p.num_blocks) * p.num_kv_heads * BS;
    CUtensorMap km, vm, qm;
    if (!make_map(&km, p.k_cache, act, cache_rows, BS, 64) || !make_map(&vm, p.v_cache, act, cache_rows, BS, 64) ||
        !make_map(&qm, p.q, act, static_cast<uint64_t>(p.num_seqs) * p.num_q_heads, G, 64))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(p.work_counter, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
    // variant 0: five 32 KB stages, one CTA per SM; variant 1: two stages, two
    // CTAs per SM (the 4 KB Q and 16 KB P buffers leave no room for three)
    static_assert(2 * (TcSmem<2, kTcStage, true>::alloc(kTcMaxSeqs) + 1024) <= kTcSmemPerSm, "two CTAs per SM");
    if (act == kBF16) {
        if (variant == 0) return by_shape<kBF16, kBF16, 5, true>(p, km, vm, qm, BS, G, 1, s);
        return by_shape<kBF16, kBF16, 2, true>(p, km, vm, qm, BS, G, 2, s);
    }
    if (variant == 0) return by_shape<kF16, kF16, 5, true>(p, km, vm, qm, BS, G, 1, s);
    return by_shape<kF16, kF16, 2, true>(p, km, vm, qm, BS, G, 2, s);
}

}  // namespace pkv
