// Device helpers shared by the sm_103a kernels: element conversion, mbarrier
// and bulk-copy (TMA) wrappers written as inline PTX, bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

enum : int { kF16 = 0, kBF16 = 1, kE4M3 = 2 };

// Bits of the per-device error word (mirrors pkv_device_error_bits).
enum : int { kErrBadBlock = 1, kErrBadLen = 2, kErrBadSlot = 4, kErrBadPair = 8, kErrTimeout = 16 };

// Longest time a kernel waits on one on-chip barrier before it reports
// kErrTimeout and stops (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes initialised barriers visible to the other threads and to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait until the phase with the given parity has completed; false once
// limit_ns of %globaltimer have passed.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// The wait every kernel uses: false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// ---- bulk async copy (TMA, non-tensor form) -------------------------------
// L2 policy for data read exactly once per launch.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Copy `bytes` (multiple of 16, both addresses 16-byte aligned) from global to
// this CTA's shared memory; completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 2^x with the hardware's base-2 exponential (PTX ex2.approx.ftz.f32: relative
// error below 2^-22 by the PTX ISA, subnormal results flushed to zero, 2^-inf =
// +0).  The softmax weights it computes are rounded to 16 (or 8) bits or summed
// in float32 afterwards, so its error is far below the output's rounding.
// q = x / d, r = x % d for x >= 0, d > 0: one 32-bit unsigned division when x
// fits 32 bits (every index of the workloads this library serves), the
// 64-bit routine otherwise.
__device__ __forceinline__ void divmod_u(int64_t x, int d, int64_t& q, int& r) {
    if ((static_cast<uint64_t>(x) >> 32) == 0) {
        const uint32_t x32 = static_cast<uint32_t>(x), q32 = x32 / static_cast<uint32_t>(d);
        q = q32;
        r = static_cast<int>(x32 - q32 * static_cast<uint32_t>(d));
    } else {
        q = x / d;
        r = static_cast<int>(x - q * d);
    }
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Maximum of x over the 32 lanes of the warp, in one warp-wide reduction
// (redux.sync.max.f32; every lane of the warp must call it).
__device__ __forceinline__ float warp_max(float x) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
    return r;
}

// ---- element conversion ---------------------------------------------------
// 16 bytes of cache elements -> floats (8 for 16-bit types, 16 for E4M3).
template <int T>
struct Vec16;

template <>
struct Vec16<kBF16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void to_float(const uint4& u, float* f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

template <>
struct Vec16<kF16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void to_float(const uint4& u, float* f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            float2 t = __half22float2(h);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
};

template <>
struct Vec16<kE4M3> {
    static constexpr int N = 16;
    __device__ __forceinline__ static void to_float(const uint4& u, float* f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * j)) & 0xffffu);
                __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
                __half2 h = *reinterpret_cast<__half2*>(&hr);
                float2 t = __half22float2(h);
                f[4 * i + 2 * j] = t.x;
                f[4 * i + 2 * j + 1] = t.y;
            }
        }
    }
};

// E4M3 pair -> binary16 pair (exact: every E4M3 value is a binary16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
    uint32_t d;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
    return d;
}

// Mixed-precision fused multiply-adds with binary16 sources and binary32
// accumulators (the product of two binary16 values is exact in binary32):
// d0 += a.lo * b.lo, d1 += a.hi * b.hi.
__device__ __forceinline__ void fma_f16x2_f32(uint32_t a, uint32_t b, float& d0, float& d1) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "mov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "r"(a), "r"(b));
}

// d0 += s * b.lo, d1 += s * b.hi (s, b binary16; d0, d1 binary32).
__device__ __forceinline__ void fma_f16s_f32(uint16_t s, uint32_t b, float& d0, float& d1) {
    asm("{\n\t.reg .b16 bl, bh;\n\t"
        "mov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.f16 %0, %2, bl, %0;\n\t"
        "fma.rn.f32.f16 %1, %2, bh, %1;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "h"(s), "r"(b));
}

// Activation (16-bit) scalar conversion.
template <int T>
__device__ __forceinline__ float act_to_float(uint16_t bits);
template <>
__device__ __forceinline__ float act_to_float<kBF16>(uint16_t bits) {
    return __uint_as_float(static_cast<uint32_t>(bits) << 16);
}
template <>
__device__ __forceinline__ float act_to_float<kF16>(uint16_t bits) {
    return __half2float(__ushort_as_half(bits));
}

template <int T>
__device__ __forceinline__ uint16_t float_to_act(float x);
template <>
__device__ __forceinline__ uint16_t float_to_act<kBF16>(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <>
__device__ __forceinline__ uint16_t float_to_act<kF16>(float x) {
    return __half_as_ushort(__float2half_rn(x));
}

// Fused append: one warp writes row (seq, kvh) of the new K and V into slot
// `slot` of the caches (16-bit copy, or E4M3 codes of x / scale), then fences
// the generic-proxy writes against later TMA (async-proxy) reads of the same
// block issued by this warp.  A slot outside the pool is skipped and flagged
// (kErrBadSlot); a negative slot means no new token.
template <int ACT, int CACHE>
__device__ __forceinline__ void append_row_warp(const void* k_new, const void* v_new, int64_t slot, int seq, int kvh,
                                                int num_kv_heads, int block_size, int head_dim, int num_blocks,
                                                void* k_cache, void* v_cache, const float* k_scale,
                                                const float* v_scale, int* err, int lane) {
    if (slot < 0) return;
    if (slot >= static_cast<int64_t>(num_blocks) * block_size) {
        if (lane == 0) atomicOr(err, kErrBadSlot);
        return;
    }
    int64_t blk;
    int off;
    divmod_u(slot, block_size, blk, off);
    const int64_t dst = ((blk * num_kv_heads + kvh) * block_size + off) * head_dim;
    const int64_t src = (static_cast<int64_t>(seq) * num_kv_heads + kvh) * head_dim;
    for (int c = lane; c < head_dim / 8; c += 32) {
        const uint4 kin = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(k_new) + src + c * 8);
        const uint4 vin = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(v_new) + src + c * 8);
        if (CACHE == ACT) {
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(k_cache) + dst + c * 8) = kin;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(v_cache) + dst + c * 8) = vin;
        } else {
            const float ks = *k_scale, vs = *v_scale;
            const uint16_t* ke = reinterpret_cast<const uint16_t*>(&kin);
            const uint16_t* ve = reinterpret_cast<const uint16_t*>(&vin);
            uint8_t kq[8], vq[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                kq[j] = __nv_cvt_float_to_fp8(__fdiv_rn(act_to_float<ACT>(ke[j]), ks), __NV_SATFINITE, __NV_E4M3);
                vq[j] = __nv_cvt_float_to_fp8(__fdiv_rn(act_to_float<ACT>(ve[j]), vs), __NV_SATFINITE, __NV_E4M3);
            }
            *reinterpret_cast<uint2*>(static_cast<uint8_t*>(k_cache) + dst + c * 8) = *reinterpret_cast<const uint2*>(kq);
            *reinterpret_cast<uint2*>(static_cast<uint8_t*>(v_cache) + dst + c * 8) = *reinterpret_cast<const uint2*>(vq);
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
}

}  // namespace pkv
