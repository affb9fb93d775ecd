// paged_attention_decode_noalloc: the decode entry point for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc, or anything else that allocates, where
// they run decode: an engine that reserves all free device memory up front for
// its own pool, so that a further cudaMalloc fails or competes with it; a host
// framework that forbids allocation on its decode path because cudaMalloc can
// block and synchronise the device; a plain C caller with no device allocator
// of its own.  Those callers cannot provide the split-K workspace that
// paged_attention_decode asks for.  This entry point takes its workspace from a
// file-scope device array of fixed size instead.  The caller still passes
// every input and output buffer.
//
// The array lives in the library's device image: every GPU that loads the
// library holds PKV_NOALLOC_MAX_WORKSPACE_BYTES of it until the process exits.
#include <mutex>
#include <string>

#include "../../include/pagedkv.h"
#include "kernels.h"
#include "pkv_error.h"

// Split-K scratch shared by every call of the no-allocation entry point.
static __device__ __align__(256) unsigned char g_pkv_noalloc_scratch[PKV_NOALLOC_MAX_WORKSPACE_BYTES];

namespace {

// Device address of g_pkv_noalloc_scratch on the current device, looked up once
// per device.  In host code the array's name only stands in for the symbol; its
// device address must come from the runtime.
int scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[pkv::kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, std::string("paged_attention_decode_noalloc: cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= pkv::kMaxDevices) return pkv::fail(PKV_ERR_CUDA, "paged_attention_decode_noalloc: device index out of range");
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_pkv_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return pkv::fail(PKV_ERR_CUDA, std::string("paged_attention_decode_noalloc: cudaGetSymbolAddress: ") +
                                               cudaGetErrorString(e));
        addr[dev] = p;
    }
    *out = addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int paged_attention_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* block_tables, int max_blocks_per_seq,
                                              const int32_t* context_lens, int num_seqs, int num_q_heads,
                                              int num_kv_heads, int block_size, int head_dim, int num_blocks,
                                              float scale, void* out, int act_dtype, int cache_dtype,
                                              const float* k_scale, const float* v_scale, int partition_size,
                                              void* stream) {
    const size_t need = pkv_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                           block_size, partition_size);
    if (need > PKV_NOALLOC_MAX_WORKSPACE_BYTES)
        return pkv::fail(PKV_ERR_INVALID,
                         "paged_attention_decode_noalloc: this request needs " + std::to_string(need) +
                             " bytes of split-K workspace, more than the fixed " +
                             std::to_string(static_cast<size_t>(PKV_NOALLOC_MAX_WORKSPACE_BYTES)) +
                             "-byte scratch; use fewer sequences, a shorter table or a larger partition_size, "
                             "or call paged_attention_decode with your own workspace");
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != PKV_OK) return rc;
    // The decode call zeroes the work counter itself and the partition kernel
    // writes every partial the merge kernel reads, so the scratch needs no
    // clearing between calls.
    return paged_attention_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                  num_q_heads, num_kv_heads, block_size, head_dim, num_blocks, scale, out, act_dtype,
                                  cache_dtype, k_scale, v_scale, partition_size, scratch,
                                  static_cast<size_t>(PKV_NOALLOC_MAX_WORKSPACE_BYTES), stream);
}
