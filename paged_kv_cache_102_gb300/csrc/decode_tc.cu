// Tensor-core grouped-query decode for 16-bit caches at head_dim 128: kernel
// instantiations and their launch (E4M3 caches: decode_tc_e4m3.cu; head_dim
// 64: decode_tc_d64.cu).
#include "decode_tc_host.cuh"

namespace pkv {

int decode_tc_max_rows() { return kTcMaxSeqs; }

bool decode_tc_supported(int head_dim, int block_size, int group, int act, int cache, int partition_size,
                         int num_kv_heads, bool per_kvh_tables) {
    // head_dim 64: pairs of kv heads (2v, 2v+1) that share the sequence's table, 16-bit caches
    const bool dims = head_dim == kTcD ||
                      (head_dim == 64 && cache == act && num_kv_heads % 2 == 0 && !per_kvh_tables);
    return dims && (block_size == 16 || block_size == 32) && (group == 2 || group == 4 || group == 8) &&
           (act == kF16 || act == kBF16) && (cache == act || cache == kE4M3) &&
           partition_size <= kTcMaxTiles * kTcTile && encode_fn() != nullptr;
}

cudaError_t launch_decode_tc(const DecodeParams& p, int act, int cache, int head_dim, int BS, int G, int variant,
                             cudaStream_t s) {
    if (head_dim == 64) return launch_decode_tc_d64(p, act, BS, G, variant, s);
    if (head_dim != kTcD) return cudaErrorInvalidValue;
    if (cache == kE4M3) return launch_decode_tc_e4m3(p, act, BS, G, variant, s);
    const int rows = p.table_kvh_stride != 0 ? p.num_seqs * p.num_kv_heads : p.num_seqs;
    const uint64_t cache_rows = static_cast<uint64_t>(p.num_blocks) * p.num_kv_heads * BS;
    CUtensorMap km, vm, qm;
    if (!make_map(&km, p.k_cache, act, cache_rows, BS) || !make_map(&vm, p.v_cache, act, cache_rows, BS) ||
        !make_map(&qm, p.q, act, static_cast<uint64_t>(p.num_seqs) * p.num_q_heads, G))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(p.work_counter, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
    // variant 0: five 32 KB stages, one CTA per SM; variant 1: two CTAs per SM
    // with three stages when the per-row tables leave room for them, else two
    const bool three = 2 * (TcSmem<3>::alloc(rows) + 1024) <= kTcSmemPerSm;
    if (act == kBF16) {
        if (variant == 0) return by_shape<kBF16, kBF16, 5>(p, km, vm, qm, BS, G, 1, s);
        return three ? by_shape<kBF16, kBF16, 3>(p, km, vm, qm, BS, G, 2, s)
                     : by_shape<kBF16, kBF16, 2>(p, km, vm, qm, BS, G, 2, s);
    }
    if (variant == 0) return by_shape<kF16, kF16, 5>(p, km, vm, qm, BS, G, 1, s);
    return three ? by_shape<kF16, kF16, 3>(p, km, vm, qm, BS, G, 2, s)
                 : by_shape<kF16, kF16, 2>(p, km, vm, qm, BS, G, 2, s);
}

}  // namespace pkv
