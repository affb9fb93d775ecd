// Kernel parameter blocks and launchers (host-visible, no device code).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

constexpr int kMaxDevices = 64;

struct AppendParams {
    const void* k;
    const void* v;
    const int64_t* slot_mapping;
    void* k_cache;
    void* v_cache;
    const float* k_scale;
    const float* v_scale;
    int* err;
    int num_tokens;
    int num_kv_heads;
    int head_dim;
    int block_size;
    int num_blocks;
};

struct CopyParams {
    void* k_cache;
    void* v_cache;
    const int32_t* pairs;
    int* err;
    size_t block_bytes;
    int num_blocks;
};

struct SwapParams {
    void* k_cache;
    void* v_cache;
    const int32_t* block_ids;
    void* staging;  // [n][2][block_bytes]: K then V of each listed block
    int* err;
    size_t block_bytes;
    int num_blocks;
    int to_staging;  // 1: pools -> staging (swap out), 0: staging -> pools (swap in)
};

struct DecodeParams {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    void* out;
    float* ws_ml;  // [num_seqs][num_q_heads][max_parts][2]: (max in log2 units, sum)
    float* ws_o;   // [num_seqs][num_q_heads][max_parts][head_dim]: normalised partial outputs
    int* work_counter;  // workspace header: next item to claim (tensor-core path), zero at launch
    // fused append (optional): new K/V row of each sequence ([num_seqs][Hkv][D], act dtype) and its
    // slot; the row is the sequence's last context token
    const void* k_new;
    const void* v_new;
    const int64_t* new_slots;
    // table row of (seq, kvh) = block_tables + seq*table_seq_stride + kvh*table_kvh_stride;
    // its length = context_lens[seq*lens_seq_stride + kvh*lens_kvh_stride]
    // (per-sequence tables: max_blocks_per_seq, 0, 1, 0)
    int64_t table_seq_stride;
    int64_t table_kvh_stride;
    int lens_seq_stride;
    int lens_kvh_stride;
    const float* k_scale;
    const float* v_scale;
    int* err;
    int max_blocks_per_seq;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int num_blocks;
    int partition_size;  // tokens per partition, a multiple of 32 and of the block size
    int max_parts;
    float scale_log2;  // scale * log2(e)
};

struct MergeParams {
    const int32_t* context_lens;
    int num_seqs;
    int lens_seq_stride;
    int lens_kvh_stride;
    int group;  // query heads per kv head
    const float* ws_ml;
    const float* ws_o;
    void* out;
    int num_q_heads;
    int head_dim;
    int partition_size;
    int max_parts;
    int max_context;
};

struct QuestMetaParams {
    const void* k_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    void* kmeta;
    int* err;
    int num_seqs;
    int max_blocks_per_seq;
    int num_kv_heads;
    int block_size;
    int head_dim;
    int num_blocks;
};

struct QuestAppendParams {
    const void* k_new;
    const int64_t* slot_mapping;
    const float* k_scale;  // E4M3 cache only
    void* kmeta;
    int* err;
    int num_tokens;
    int num_kv_heads;
    int block_size;
    int head_dim;
    int num_blocks;
};

struct QuestSelectParams {
    const void* q;
    const void* kmeta;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t* sel_tables;
    int32_t* sel_lens;
    float* bounds;  // workspace [num_seqs][num_kv_heads][max_blocks_per_seq]
    int* err;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int block_size;
    int head_dim;
    int num_blocks;
    int max_blocks_per_seq;
    int budget_blocks;
    int group_heads;  // kv heads per bound item (set by launch_quest_select)
};

cudaError_t launch_quest_minmax(const QuestMetaParams& p, int meta, int cache, cudaStream_t s);
cudaError_t launch_quest_append_minmax(const QuestAppendParams& p, int act, int cache, cudaStream_t s);
cudaError_t launch_quest_select(const QuestSelectParams& p, int dtype, int G, cudaStream_t s);

cudaError_t launch_append(const AppendParams& p, int act, int cache, cudaStream_t stream);
cudaError_t launch_block_copy(const CopyParams& p, int num_pairs, cudaStream_t stream);
cudaError_t launch_block_swap(const SwapParams& p, int n, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, int act, cudaStream_t stream);
cudaError_t launch_selftest_wait(uint64_t limit_ns, int* err, cudaStream_t stream);

// Partition kernel for one (act, cache) pair; returns cudaErrorInvalidValue
// for a (head_dim, block_size, group) it was not built for.
cudaError_t launch_decode_f16_f16(const DecodeParams& p, int D, int BS, int G, cudaStream_t s);
cudaError_t launch_decode_bf16_bf16(const DecodeParams& p, int D, int BS, int G, cudaStream_t s);
cudaError_t launch_decode_f16_e4m3(const DecodeParams& p, int D, int BS, int G, cudaStream_t s);
cudaError_t launch_decode_bf16_e4m3(const DecodeParams& p, int D, int BS, int G, cudaStream_t s);

// Tensor-core grouped-query path (head_dim 128 with a 16-bit or E4M3 cache,
// or head_dim 64 with a 16-bit cache, an even kv-head count and shared
// tables; group 2/4/8; partitions of at most 512 tokens).  variant 0: one CTA
// per SM; variant 1: two CTAs per SM.
bool decode_tc_supported(int head_dim, int block_size, int group, int act, int cache, int partition_size,
                         int num_kv_heads, bool per_kvh_tables);
int decode_tc_max_rows();  // table rows (sequences, or (sequence, kv head) pairs) of one launch
cudaError_t launch_decode_tc(const DecodeParams& p, int act, int cache, int head_dim, int BS, int G, int variant,
                             cudaStream_t s);
cudaError_t launch_decode_tc_e4m3(const DecodeParams& p, int act, int BS, int G, int variant, cudaStream_t s);
cudaError_t launch_decode_tc_d64(const DecodeParams& p, int act, int BS, int G, int variant, cudaStream_t s);

}  // namespace pkv
