// C-ABI entry points of libpagedkv.so: argument checks, partition-size
// choice, workspace carving and kernel dispatch.  Declarations and the
// contract of each call are in include/pagedkv.h.
#include <atomic>
#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>

#include "../../include/pagedkv.h"
#include "kernels.h"
#include "pkv_error.h"

// Per-device error word written by the kernels (OR of pkv_device_error_bits).
static __device__ int g_pkv_device_error;

namespace pkv {

namespace {
thread_local std::string t_last_error;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device address of g_pkv_device_error on the current device.
int* device_error_word() {
    static std::mutex mu;
    static int* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_device_error) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<int*>(p);
    }
    return addr[dev];
}

int cuda_fail(const char* where, cudaError_t e) {
    return fail(PKV_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kStageTokens = 32;  // tokens per shared-memory stage of the decode kernel
constexpr int kAutoPartition = 1024;
constexpr int kAutoPartitionGrouped = 512;
// Grouped shapes with a few hundred (sequence, kv head, partition) items get
// 256-token partitions, so that the persistent grid's CTAs each get several
// to balance.  Below 256 items every CTA has at most about one, and smaller
// partitions only add merge work (QUEST's sparse decode of 8 x 8 rows: 41.0 ->
// 37.1 us at 4096 selected tokens a row, 29.4 -> 28.7 at 2048, 20.6 -> 22.6 at
// 1024 if it were applied there).
constexpr long long kAutoGroupedItemsLow = 256, kAutoGroupedItemsHigh = 1024;
constexpr size_t kWorkspaceHeader = 256;  // work counter of the tensor-core path

std::atomic<int> g_kernel_path{PKV_PATH_AUTO};

}  // namespace

void set_error(const std::string& msg) { t_last_error = msg; }

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_last_error(void) { return t_last_error.c_str(); }

int pkv_version(void) { return 100; }

int pkv_selftest_wait_timeout(int limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 2000000)
        return fail(PKV_ERR_INVALID, "pkv_selftest_wait_timeout: limit_us must be in 1 .. 2,000,000");
    int* err = device_error_word();
    if (!err) return fail(PKV_ERR_CUDA, "pkv_selftest_wait_timeout: cannot resolve the device error word");
    const cudaError_t e =
        launch_selftest_wait(static_cast<uint64_t>(limit_us) * 1000u, err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail("pkv_selftest_wait_timeout: launch", e);
}

int pkv_set_kernel_path(int path) {
    if (path < PKV_PATH_AUTO || path > PKV_PATH_TENSOR_2CTA) return -1;
    return g_kernel_path.exchange(path);
}

int pkv_device_error(int* bits, int reset, void* stream) {
    if (!bits) return fail(PKV_ERR_INVALID, "pkv_device_error: bits is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail("pkv_device_error: stream synchronize", e);
    int* word = device_error_word();
    if (!word) return fail(PKV_ERR_CUDA, "pkv_device_error: cannot resolve the device error word");
    e = cudaMemcpy(bits, word, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail("pkv_device_error: read", e);
    if (reset) {
        e = cudaMemset(word, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_fail("pkv_device_error: reset", e);
    }
    return PKV_OK;
}

int pkv_resolve_partition_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int max_blocks_per_seq, int block_size, int partition_size) {
    if (max_blocks_per_seq < 1 || block_size < 1 || num_kv_heads < 1 || num_q_heads < 1) return -1;
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    const long long single = (max_ctx + kStageTokens - 1) / kStageTokens * kStageTokens;
    long long P;
    if (partition_size == PKV_PARTITION_SINGLE) {
        P = single;
    } else if (partition_size == PKV_PARTITION_AUTO) {
        // the tensor-core grouped-query kernel holds 512 tokens of scores in tensor
        // memory; the CUDA-core kernel amortises its per-partition work over 1024
        const int G = num_q_heads / num_kv_heads;
        const bool grouped = G >= 4 && (head_dim == 128 || (head_dim == 64 && num_kv_heads % 2 == 0));
        P = grouped ? kAutoPartitionGrouped : kAutoPartition;
        if (grouped) {
            // items: (sequence, kv head, partition), or (sequence, pair of kv heads, partition) at head_dim 64
            const int item_heads = head_dim == 64 ? num_kv_heads / 2 : num_kv_heads;
            auto items = [&](long long p) { return static_cast<long long>(num_seqs) * item_heads * ((max_ctx + p - 1) / p); };
            if (items(P) >= kAutoGroupedItemsLow && items(P) < kAutoGroupedItemsHigh && (P / 2) % block_size == 0)
                P /= 2;
        }
    } else if (partition_size > 0) {
        if (partition_size % kStageTokens != 0 || partition_size % block_size != 0) return -1;
        P = partition_size;
    } else {
        return -1;
    }
    if (P >= single) P = single;
    if (P > 0x7fffffff) return -1;
    return static_cast<int>(P);
}

size_t pkv_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int max_blocks_per_seq, int block_size, int partition_size) {
    const int P = pkv_resolve_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                             block_size, partition_size);
    if (P <= 0 || num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    const long long parts = (max_ctx + P - 1) / P;
    if (parts <= 1) return kWorkspaceHeader;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * static_cast<size_t>(parts);
    return kWorkspaceHeader + align_up(rows * 2 * sizeof(float), 256) +
           rows * static_cast<size_t>(head_dim) * sizeof(float);
}

int paged_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens, void* k_cache,
                    void* v_cache, int num_blocks, int num_kv_heads, int block_size, int head_dim, int act_dtype,
                    int cache_dtype, const float* k_scale, const float* v_scale, void* stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0 || head_dim <= 0 ||
        head_dim % 8 != 0)
        return fail(PKV_ERR_INVALID, "paged_kv_append: sizes must be positive and head_dim a multiple of 8");
    if (act_dtype != PKV_F16 && act_dtype != PKV_BF16)
        return fail(PKV_ERR_INVALID, "paged_kv_append: act_dtype must be PKV_F16 or PKV_BF16");
    if (cache_dtype != act_dtype && cache_dtype != PKV_E4M3)
        return fail(PKV_ERR_INVALID, "paged_kv_append: cache_dtype must equal act_dtype or be PKV_E4M3");
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache)
        return fail(PKV_ERR_INVALID, "paged_kv_append: null pointer");
    if (cache_dtype == PKV_E4M3 && (!k_scale || !v_scale))
        return fail(PKV_ERR_INVALID, "paged_kv_append: an E4M3 cache needs k_scale and v_scale");
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return fail(PKV_ERR_INVALID, "paged_kv_append: buffers must be 16-byte aligned (slot_mapping 8)");
    int* err = device_error_word();
    if (!err) return fail(PKV_ERR_CUDA, "paged_kv_append: cannot resolve the device error word");
    AppendParams p{k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, err,
                   num_tokens, num_kv_heads, head_dim, block_size, num_blocks};
    cudaError_t e = launch_append(p, act_dtype, cache_dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("paged_kv_append: launch", e);
    return PKV_OK;
}

int paged_block_copy(void* k_cache, void* v_cache, const int32_t* src_dst_pairs, int num_pairs, int num_blocks,
                     size_t block_bytes, void* stream) {
    if (num_pairs < 0 || num_blocks <= 0 || block_bytes == 0 || block_bytes % 16 != 0)
        return fail(PKV_ERR_INVALID, "paged_block_copy: num_pairs >= 0, num_blocks > 0, block_bytes a positive multiple of 16");
    if (num_pairs == 0) return PKV_OK;
    if (num_pairs > 65535 * 64) return fail(PKV_ERR_INVALID, "paged_block_copy: too many pairs in one call");
    if (!k_cache || !v_cache || !src_dst_pairs) return fail(PKV_ERR_INVALID, "paged_block_copy: null pointer");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_dst_pairs, 4))
        return fail(PKV_ERR_INVALID, "paged_block_copy: caches must be 16-byte aligned");
    int* err = device_error_word();
    if (!err) return fail(PKV_ERR_CUDA, "paged_block_copy: cannot resolve the device error word");
    CopyParams p{k_cache, v_cache, src_dst_pairs, err, block_bytes, num_blocks};
    cudaError_t e = launch_block_copy(p, num_pairs, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("paged_block_copy: launch", e);
    return PKV_OK;
}

int paged_block_swap(void* k_cache, void* v_cache, const int32_t* block_ids, int num_ids, int num_blocks,
                     size_t block_bytes, void* staging, int direction, void* stream) {
    if (num_ids < 0 || num_blocks <= 0 || block_bytes == 0 || block_bytes % 16 != 0 ||
        (direction != PKV_SWAP_OUT && direction != PKV_SWAP_IN))
        return fail(PKV_ERR_INVALID, "paged_block_swap: bad sizes or direction");
    if (num_ids == 0) return PKV_OK;
    if (num_ids > 0x7fffffff / 2) return fail(PKV_ERR_INVALID, "paged_block_swap: too many blocks");
    if (!k_cache || !v_cache || !block_ids || !staging) return fail(PKV_ERR_INVALID, "paged_block_swap: null pointer");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(staging, 16) || !aligned(block_ids, 4))
        return fail(PKV_ERR_INVALID, "paged_block_swap: buffers must be 16-byte aligned");
    cudaPointerAttributes attr{};
    cudaError_t e = cudaPointerGetAttributes(&attr, staging);
    if (e != cudaSuccess) return cuda_fail("paged_block_swap: staging pointer", e);
    if (attr.type == cudaMemoryTypeUnregistered)
        return fail(PKV_ERR_INVALID, "paged_block_swap: staging must be device memory or pinned/registered host memory");
    int* err = device_error_word();
    if (!err) return fail(PKV_ERR_CUDA, "paged_block_swap: cannot resolve the device error word");
    void* dev_staging = attr.type == cudaMemoryTypeHost && attr.devicePointer ? attr.devicePointer : staging;
    SwapParams p{k_cache, v_cache, block_ids, dev_staging, err, block_bytes, num_blocks,
                 direction == PKV_SWAP_OUT ? 1 : 0};
    e = launch_block_swap(p, num_ids, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("paged_block_swap: launch", e);
    return PKV_OK;
}

}  // extern "C"

static int decode_impl(const char* fn, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                       int num_q_heads, int num_kv_heads, int block_size, int head_dim, int num_blocks, float scale,
                       void* out, int act_dtype, int cache_dtype, const float* k_scale, const float* v_scale,
                       int partition_size, void* workspace, size_t workspace_bytes, void* stream, const void* k_new,
                       const void* v_new, const int64_t* new_slots, bool per_kvh_tables = false) {
    const std::string F(fn);
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0)
        return fail(PKV_ERR_INVALID, F + ": " + "sizes must be positive");
    if (num_q_heads % num_kv_heads != 0)
        return fail(PKV_ERR_SHAPE, F + ": " + "num_q_heads must be a multiple of num_kv_heads");
    const int G = num_q_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PKV_ERR_INVALID, F + ": " + "query heads per kv head must be 1, 2, 4 or 8");
    if (head_dim != 64 && head_dim != 128)
        return fail(PKV_ERR_INVALID, F + ": " + "head_dim must be 64 or 128");
    if (block_size != 16 && block_size != 32)
        return fail(PKV_ERR_INVALID, F + ": " + "block_size must be 16 or 32");
    if (act_dtype != PKV_F16 && act_dtype != PKV_BF16)
        return fail(PKV_ERR_INVALID, F + ": " + "act_dtype must be PKV_F16 or PKV_BF16");
    if (cache_dtype != act_dtype && cache_dtype != PKV_E4M3)
        return fail(PKV_ERR_INVALID, F + ": " + "cache_dtype must equal act_dtype or be PKV_E4M3");
    if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID, F + ": " + "scale must be finite");
    if (num_seqs == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return fail(PKV_ERR_INVALID, F + ": " + "null pointer");
    if (cache_dtype == PKV_E4M3 && (!k_scale || !v_scale))
        return fail(PKV_ERR_INVALID, F + ": " + "an E4M3 cache needs k_scale and v_scale");
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(workspace, 16))
        return fail(PKV_ERR_INVALID, F + ": " + "q, caches, out, workspace must be 16-byte aligned");
    const int P = pkv_resolve_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                             block_size, partition_size);
    if (P <= 0)
        return fail(PKV_ERR_INVALID, F + ": " + "partition_size must be 0, -1 or a positive multiple of 32 and of block_size");
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    if (max_ctx > 0x7fffffffLL) return fail(PKV_ERR_INVALID, F + ": " + "table too long");
    const int max_parts = static_cast<int>((max_ctx + P - 1) / P);
    if (max_parts > 65535 || num_kv_heads > 65535 || num_seqs > 65535)
        return fail(PKV_ERR_INVALID, F + ": " + "grid too large (partitions, kv heads or sequences > 65535)");
    const size_t need = pkv_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                           block_size, partition_size);
    if (!workspace || workspace_bytes < need)
        return fail(PKV_ERR_INVALID, F + ": " + "workspace of " + std::to_string(need) +
                                         " bytes required (pkv_workspace_size)");
    int* err = device_error_word();
    if (!err) return fail(PKV_ERR_CUDA, F + ": " + "cannot resolve the device error word");

    DecodeParams p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = out;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * static_cast<size_t>(max_parts);
    char* ws = static_cast<char*>(workspace);
    p.work_counter = reinterpret_cast<int*>(ws);
    p.ws_ml = max_parts > 1 ? reinterpret_cast<float*>(ws + kWorkspaceHeader) : nullptr;
    p.ws_o = max_parts > 1 ? reinterpret_cast<float*>(ws + kWorkspaceHeader + align_up(rows * 2 * sizeof(float), 256))
                           : nullptr;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.err = err;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.partition_size = P;
    p.max_parts = max_parts;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.k_new = k_new;
    p.v_new = v_new;
    p.new_slots = new_slots;
    if (per_kvh_tables) {  // tables [B][Hkv][max_blocks], lengths [B][Hkv]
        p.table_seq_stride = static_cast<int64_t>(num_kv_heads) * max_blocks_per_seq;
        p.table_kvh_stride = max_blocks_per_seq;
        p.lens_seq_stride = num_kv_heads;
        p.lens_kvh_stride = 1;
    } else {
        p.table_seq_stride = max_blocks_per_seq;
        p.table_kvh_stride = 0;
        p.lens_seq_stride = 1;
        p.lens_kvh_stride = 0;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    const int path = g_kernel_path.load();
    // the tensor-core kernel keeps per-row tables in shared memory: larger
    // batches run as several launches over consecutive sequences
    const int rows_per_seq = per_kvh_tables ? num_kv_heads : 1;
    const bool tc_ok = rows_per_seq <= decode_tc_max_rows() &&
                       decode_tc_supported(head_dim, block_size, G, act_dtype, cache_dtype, P, num_kv_heads,
                                           per_kvh_tables);
    if ((path == PKV_PATH_TENSOR || path == PKV_PATH_TENSOR_2CTA) && !tc_ok)
        return fail(PKV_ERR_INVALID, F + ": " + "the tensor-core path needs head_dim 128 (16-bit or E4M3 "
                                     "cache) or 64 (16-bit cache, even kv heads, shared tables), 2/4/8 query "
                                     "heads per kv head and partitions of at most 512 tokens");
    const bool use_tc = path == PKV_PATH_TENSOR || path == PKV_PATH_TENSOR_2CTA ||
                        (path == PKV_PATH_AUTO && tc_ok && G >= 4);
    if (use_tc) {
        const int chunk = decode_tc_max_rows() / rows_per_seq;
        const size_t act_bytes = 2;
        e = cudaSuccess;
        for (int s0 = 0; s0 < num_seqs && e == cudaSuccess; s0 += chunk) {
            DecodeParams c = p;
            c.num_seqs = std::min(chunk, num_seqs - s0);
            c.q = static_cast<const char*>(q) + static_cast<size_t>(s0) * num_q_heads * head_dim * act_bytes;
            c.out = static_cast<char*>(out) + static_cast<size_t>(s0) * num_q_heads * head_dim * act_bytes;
            c.block_tables = block_tables + s0 * p.table_seq_stride;
            c.context_lens = context_lens + static_cast<int64_t>(s0) * p.lens_seq_stride;
            if (new_slots) {
                c.k_new = static_cast<const char*>(k_new) + static_cast<size_t>(s0) * num_kv_heads * head_dim * act_bytes;
                c.v_new = static_cast<const char*>(v_new) + static_cast<size_t>(s0) * num_kv_heads * head_dim * act_bytes;
                c.new_slots = new_slots + s0;
            }
            if (max_parts > 1) {
                const size_t hrow0 = static_cast<size_t>(s0) * num_q_heads * max_parts;
                c.ws_ml = p.ws_ml + hrow0 * 2;
                c.ws_o = p.ws_o + hrow0 * head_dim;
            }
            e = launch_decode_tc(c, act_dtype, cache_dtype, head_dim, block_size, G, path == PKV_PATH_TENSOR ? 0 : 1,
                                 s);
        }
    } else if (act_dtype == PKV_F16)
        e = cache_dtype == PKV_E4M3 ? launch_decode_f16_e4m3(p, head_dim, block_size, G, s)
                                    : launch_decode_f16_f16(p, head_dim, block_size, G, s);
    else
        e = cache_dtype == PKV_E4M3 ? launch_decode_bf16_e4m3(p, head_dim, block_size, G, s)
                                    : launch_decode_bf16_bf16(p, head_dim, block_size, G, s);
    if (e != cudaSuccess) return cuda_fail((F + ": partition kernel launch").c_str(), e);
    if (max_parts > 1) {
        MergeParams m{};
        m.context_lens = context_lens;
        m.num_seqs = num_seqs;
        m.lens_seq_stride = p.lens_seq_stride;
        m.lens_kvh_stride = p.lens_kvh_stride;
        m.group = G;
        m.ws_ml = p.ws_ml;
        m.ws_o = p.ws_o;
        m.out = out;
        m.num_q_heads = num_q_heads;
        m.head_dim = head_dim;
        m.partition_size = P;
        m.max_parts = max_parts;
        m.max_context = static_cast<int>(max_ctx);
        e = launch_merge(m, act_dtype, s);
        if (e != cudaSuccess) return cuda_fail((F + ": merge kernel launch").c_str(), e);
    }
    return PKV_OK;
}

extern "C" {

int paged_attention_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int block_size, int head_dim, int num_blocks, float scale, void* out,
                           int act_dtype, int cache_dtype, const float* k_scale, const float* v_scale,
                           int partition_size, void* workspace, size_t workspace_bytes, void* stream) {
    return decode_impl("paged_attention_decode", q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       num_seqs, num_q_heads, num_kv_heads, block_size, head_dim, num_blocks, scale, out, act_dtype,
                       cache_dtype, k_scale, v_scale, partition_size, workspace, workspace_bytes, stream, nullptr,
                       nullptr, nullptr);
}

int paged_attention_decode_append(const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                  void* k_cache, void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                                  int block_size, int head_dim, int num_blocks, float scale, void* out, int act_dtype,
                                  int cache_dtype, const float* k_scale, const float* v_scale, int partition_size,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping))
        return fail(PKV_ERR_INVALID, "paged_attention_decode_append: null pointer");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8))
        return fail(PKV_ERR_INVALID, "paged_attention_decode_append: k_new, v_new must be 16-byte aligned");
    return decode_impl("paged_attention_decode_append", q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, num_q_heads, num_kv_heads, block_size, head_dim, num_blocks, scale, out,
                       act_dtype, cache_dtype, k_scale, v_scale, partition_size, workspace, workspace_bytes, stream,
                       k_new, v_new, slot_mapping);
}


int paged_attention_decode_sparse(const void* q, const void* k_cache, const void* v_cache, const int32_t* sel_tables,
                                  int max_sel_blocks, const int32_t* sel_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int block_size, int head_dim, int num_blocks, float scale,
                                  void* out, int act_dtype, int cache_dtype, const float* k_scale,
                                  const float* v_scale, int partition_size, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    return decode_impl("paged_attention_decode_sparse", q, k_cache, v_cache, sel_tables, max_sel_blocks, sel_lens,
                       num_seqs, num_q_heads, num_kv_heads, block_size, head_dim, num_blocks, scale, out, act_dtype,
                       cache_dtype, k_scale, v_scale, partition_size, workspace, workspace_bytes, stream, nullptr,
                       nullptr, nullptr, true);
}

int quest_block_minmax(const void* k_cache, const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int num_seqs, int num_kv_heads, int block_size, int head_dim,
                       int num_blocks, int cache_dtype, int meta_dtype, void* kmeta, void* stream) {
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0 ||
        head_dim <= 0 || head_dim % 8 != 0)
        return fail(PKV_ERR_INVALID, "quest_block_minmax: sizes must be positive, head_dim a multiple of 8");
    if (meta_dtype != PKV_F16 && meta_dtype != PKV_BF16)
        return fail(PKV_ERR_INVALID, "quest_block_minmax: meta_dtype must be PKV_F16 or PKV_BF16");
    if (cache_dtype != meta_dtype && cache_dtype != PKV_E4M3)
        return fail(PKV_ERR_INVALID, "quest_block_minmax: the cache must be of meta_dtype or PKV_E4M3");
    if (num_seqs == 0) return PKV_OK;
    if (!k_cache || !block_tables || !context_lens || !kmeta) return fail(PKV_ERR_INVALID, "quest_block_minmax: null pointer");
    if (!aligned(k_cache, 16) || !aligned(kmeta, 16)) return fail(PKV_ERR_INVALID, "quest_block_minmax: misaligned");
    int* err = device_error_word();
    if (!err) return fail(PKV_ERR_CUDA, "quest_block_minmax: cannot resolve the device error word");
    QuestMetaParams p{k_cache, block_tables, context_lens, kmeta, err, num_seqs, max_blocks_per_seq, num_kv_heads,
                      block_size, head_dim, num_blocks};
    cudaError_t e = launch_quest_minmax(p, meta_dtype, cache_dtype, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail("quest_block_minmax: launch", e);
}

int quest_append_minmax(const void* k_new, const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                        int block_size, int head_dim, int num_blocks, int act_dtype, int cache_dtype,
                        const float* k_scale, void* kmeta, void* stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0 || head_dim <= 0 || head_dim % 8 != 0)
        return fail(PKV_ERR_INVALID, "quest_append_minmax: sizes must be positive, head_dim a multiple of 8");
    if (act_dtype != PKV_F16 && act_dtype != PKV_BF16)
        return fail(PKV_ERR_INVALID, "quest_append_minmax: act_dtype must be PKV_F16 or PKV_BF16");
    if (cache_dtype != act_dtype && cache_dtype != PKV_E4M3)
        return fail(PKV_ERR_INVALID, "quest_append_minmax: the cache must be of act_dtype or PKV_E4M3");
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !slot_mapping || !kmeta) return fail(PKV_ERR_INVALID, "quest_append_minmax: null pointer");
    if (cache_dtype == PKV_E4M3 && !k_scale)
        return fail(PKV_ERR_INVALID, "quest_append_minmax: an E4M3 cache needs k_scale");
    if (!aligned(k_new, 16) || !aligned(kmeta, 16) || !aligned(slot_mapping, 8))
        return fail(PKV_ERR_INVALID, "quest_append_minmax: misaligned");
    int* err = device_error_word();
    if (!err) return fail(PKV_ERR_CUDA, "quest_append_minmax: cannot resolve the device error word");
    QuestAppendParams p{k_new, slot_mapping, cache_dtype == PKV_E4M3 ? k_scale : nullptr, kmeta, err, num_tokens,
                        num_kv_heads, block_size, head_dim, num_blocks};
    cudaError_t e = launch_quest_append_minmax(p, act_dtype, cache_dtype, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail("quest_append_minmax: launch", e);
}

size_t quest_workspace_size(int num_seqs, int num_kv_heads, int max_blocks_per_seq) {
    if (num_seqs <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0) return 0;
    return static_cast<size_t>(num_seqs) * num_kv_heads * max_blocks_per_seq * sizeof(float);
}

int quest_select(const void* q, const void* kmeta, const int32_t* block_tables, int max_blocks_per_seq,
                 const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int block_size,
                 int head_dim, int num_blocks, int act_dtype, int budget_blocks, int32_t* sel_tables, int32_t* sel_lens,
                 void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0 || budget_blocks <= 0)
        return fail(PKV_ERR_INVALID, "quest_select: sizes must be positive, num_q_heads a multiple of num_kv_heads");
    const int G = num_q_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return fail(PKV_ERR_INVALID, "quest_select: group must be 1, 2, 4 or 8");
    if (head_dim != 64 && head_dim != 128) return fail(PKV_ERR_INVALID, "quest_select: head_dim must be 64 or 128");
    if (act_dtype != PKV_F16 && act_dtype != PKV_BF16)
        return fail(PKV_ERR_INVALID, "quest_select: act_dtype must be PKV_F16 or PKV_BF16");
    if (max_blocks_per_seq > 16384) return fail(PKV_ERR_INVALID, "quest_select: at most 16384 blocks per sequence");
    if (num_seqs == 0) return PKV_OK;
    if (num_seqs > 65535 || num_kv_heads > 65535) return fail(PKV_ERR_INVALID, "quest_select: grid too large");
    if (!q || !kmeta || !block_tables || !context_lens || !sel_tables || !sel_lens)
        return fail(PKV_ERR_INVALID, "quest_select: null pointer");
    if (!aligned(q, 16) || !aligned(kmeta, 16)) return fail(PKV_ERR_INVALID, "quest_select: q and kmeta must be 16-byte aligned");
    const size_t need = quest_workspace_size(num_seqs, num_kv_heads, max_blocks_per_seq);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16))
        return fail(PKV_ERR_INVALID, "quest_select: workspace of " + std::to_string(need) +
                                         " bytes (16-byte aligned) required (quest_workspace_size)");
    int* err = device_error_word();
    if (!err) return fail(PKV_ERR_CUDA, "quest_select: cannot resolve the device error word");
    QuestSelectParams p{q, kmeta, block_tables, context_lens, sel_tables, sel_lens, static_cast<float*>(workspace),
                        err, num_seqs, num_q_heads, num_kv_heads, block_size, head_dim, num_blocks,
                        max_blocks_per_seq, budget_blocks, /*group_heads: chosen at launch*/ 0};
    cudaError_t e = launch_quest_select(p, act_dtype, G, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail("quest_select: launch", e);
}

}  // extern "C"
