// Host side of the tensor-core grouped-query decode kernel shared by its
// translation units (16-bit caches at head_dim 128 in decode_tc.cu, E4M3
// caches in decode_tc_e4m3.cu, head_dim-64 pairs in decode_tc_d64.cu): TMA
// tensor maps over the caches and the queries, persistent grid sizing, the
// launch template.
#pragma once

#include <cstring>

#include "decode_tc.cuh"
#include "tensor_map.cuh"

namespace pkv {

namespace {  // each translation unit keeps its own copy of the SM count cache

// A [rows][cols] 16-bit matrix (cols 128, or 64 for head_dim-64 pairs) read
// in boxes of 64 columns x box_rows rows, 128-byte swizzled in shared memory
// (the layout the MMA descriptors expect).
bool make_map(CUtensorMap* m, const void* base, int act, uint64_t rows, uint32_t box_rows, int cols = kTcD) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t elem_strides[2] = {1, 1};
    CUresult r = fn(m, act == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// E4M3 cache: a [rows][128] byte matrix read in boxes of 128 bytes x
// box_rows rows, 128-byte swizzled.
bool make_map8(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kTcD), rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kTcD)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcD), box_rows};
    cuuint32_t elem_strides[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count() {
    static int counts[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (!counts[dev]) cudaDeviceGetAttribute(&counts[dev], cudaDevAttrMultiProcessorCount, dev);
    return counts[dev];
}

template <int ACT, int CACHE, int BS, int G, int NS, bool PAIR>
cudaError_t launch(const DecodeParams& p, const CUtensorMap& km, const CUtensorMap& vm, const CUtensorMap& qm,
                   int ctas_per_sm, cudaStream_t s) {
    auto kern = paged_decode_tc_kernel<ACT, CACHE, BS, G, NS, PAIR>;
    using Smem = TcSmem<NS, CACHE == kE4M3 ? kTcStage8 : kTcStage, PAIR>;
    constexpr int threads = kTcThreads;
    const int rows = p.table_kvh_stride != 0 ? p.num_seqs * p.num_kv_heads : p.num_seqs;
    const int smem = Smem::alloc(rows);
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::alloc(kTcMaxSeqs));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const long long items = static_cast<long long>(p.num_seqs) * (PAIR ? p.num_kv_heads / 2 : p.num_kv_heads) *
                            p.max_parts;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = static_cast<int>(items < static_cast<long long>(sms) * ctas_per_sm ? items : sms * ctas_per_sm);
    if (grid <= 0) return cudaSuccess;
    kern<<<grid, threads, smem, s>>>(km, vm, qm, p);
    return cudaGetLastError();
}

template <int ACT, int CACHE, int NS, bool PAIR = false>
cudaError_t by_shape(const DecodeParams& p, const CUtensorMap& km, const CUtensorMap& vm, const CUtensorMap& qm,
                     int BS, int G, int ctas_per_sm, cudaStream_t s) {
    if (BS == 16) {
        if (G == 2) return launch<ACT, CACHE, 16, 2, NS, PAIR>(p, km, vm, qm, ctas_per_sm, s);
        if (G == 4) return launch<ACT, CACHE, 16, 4, NS, PAIR>(p, km, vm, qm, ctas_per_sm, s);
        if (G == 8) return launch<ACT, CACHE, 16, 8, NS, PAIR>(p, km, vm, qm, ctas_per_sm, s);
    } else if (BS == 32) {
        if (G == 2) return launch<ACT, CACHE, 32, 2, NS, PAIR>(p, km, vm, qm, ctas_per_sm, s);
        if (G == 4) return launch<ACT, CACHE, 32, 4, NS, PAIR>(p, km, vm, qm, ctas_per_sm, s);
        if (G == 8) return launch<ACT, CACHE, 32, 8, NS, PAIR>(p, km, vm, qm, ctas_per_sm, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

}  // namespace pkv
