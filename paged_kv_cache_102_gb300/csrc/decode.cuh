// Paged decode attention for sm_103a: CUDA-core path (any query-head group).
//
// What is computed: for sequence b, query head h and kv head kvh = h / G,
//   s_j = scale * <q[b][h], K[j]>,  p = softmax(s),  out[b][h] = sum_j p_j V[j]
// over the L = context_lens[b] tokens, where token j sits in physical block
// block_tables[b][j / BS] at offset j % BS (Ultralytics glossary
// "PagedAttention", section "How paging works": the attention kernel reads
// keys and values block by block through the block table; OptiVerse "Paged
// KV cache", section "Block table and non-contiguous allocation").
//
// Work decomposition.  One CTA per (partition, kv head, sequence).  A
// partition is `partition_size` consecutive tokens of one sequence; it is
// streamed through shared memory in stages of 32 tokens.  Warp 4 is the
// producer: its lanes fetch 32 block-table entries at a time and lane 0
// issues one 1-D bulk TMA copy per (block, kv head) tile -- BS*D contiguous
// cache elements, 4 KB for BS=16, D=128, bf16 -- for K and for V, completing
// on the stage's `full` mbarrier.  Warps 0-3 consume: each owns 8 tokens of
// every stage and keeps its own fp32 online-softmax state (running max m,
// running sum l, accumulator acc) for the G query heads of the kv head.
// Lanes are laid out so that one warp-wide 16-byte shared load covers whole
// token rows: LPR = D*elem/16 lanes per row, TPP = 32/LPR rows per load.
// Dot products reduce over the LPR lanes of a row with xor-shuffles; the
// stage max reduces over rows with xor-shuffles.  After the last stage the
// four warps' states are merged in shared memory (log-sum-exp weights) and
// either written as the output (one partition) or as a partial
// (m, l, o = acc/l) for the split-K merge kernel.
#pragma once

#include <type_traits>

#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

constexpr int kStageTokens = 32;
constexpr float kRescaleLog2 = 8.0f;  // largest log2 growth of the running max left unrescaled
constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;

template <int CACHE, int D, int BS, int G>
struct DecodeCfg {
    static constexpr int E = CACHE == kE4M3 ? 1 : 2;  // bytes per cache element
    static constexpr int VEC = 16 / E;                // elements per 16-byte vector
    static constexpr int LPR = D / VEC;               // lanes per token row
    static constexpr int TPP = 32 / LPR;              // token rows per warp-wide load
    static constexpr int TW = kStageTokens / kConsumerWarps;  // tokens per warp per stage
    static constexpr int PASSES = TW / TPP;
    static constexpr int BPS = kStageTokens / BS;  // blocks per stage
    static constexpr int TILE_BYTES = BS * D * E;  // one (block, kv head) tile
    static constexpr int STAGE_BYTES = kStageTokens * D * E;  // K (or V) part of a stage
    static constexpr int STAGES_RAW = 65536 / (2 * STAGE_BYTES);
    static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
    static constexpr int RED_FLOATS = kConsumerWarps * G * (D + 2);
    static constexpr int SMEM_BYTES = 2 * STAGES * STAGE_BYTES + 2 * STAGES * 8 + RED_FLOATS * 4;
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row layout");
    static_assert(TW % TPP == 0, "tokens per warp must be a multiple of rows per load");
    static_assert(kStageTokens % BS == 0, "block size must divide the stage");
    static_assert(TILE_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");
};

template <int ACT, int CACHE, int D, int BS, int G>
__global__ void __launch_bounds__(kDecodeThreads, (G <= 2 ? 3 : 2))
    paged_decode_partition_kernel(const DecodeParams p) {
    using C = DecodeCfg<CACHE, D, BS, G>;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ int s_failed;
    unsigned char* kbuf = smem;
    unsigned char* vbuf = smem + C::STAGES * C::STAGE_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + 2 * C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    float* red = reinterpret_cast<float*>(empty + C::STAGES);
    float* red_m = red;                                     // [NW][G]
    float* red_l = red + kConsumerWarps * G;                // [NW][G]
    float* red_acc = red + 2 * kConsumerWarps * G;          // [NW][G][D]

    // the merge kernel may be scheduled once every CTA got here; it waits for
    // this grid to finish
    asm volatile("griddepcontrol.launch_dependents;");
    const int part = blockIdx.x;
    const int kvh = blockIdx.y;
    const int seq = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int L = p.context_lens[static_cast<int64_t>(seq) * p.lens_seq_stride + kvh * p.lens_kvh_stride];
    if (L < 1 || L > p.max_blocks_per_seq * BS) {
        if (part == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(p.err, kErrBadLen);
        return;
    }
    const int tok_begin = part * p.partition_size;
    if (tok_begin >= L) return;
    const int tok_end = min(L, tok_begin + p.partition_size);
    const int n_stage = (tok_end - tok_begin + kStageTokens - 1) / kStageTokens;
    const int blk_begin = tok_begin / BS;
    const int n_blk = (tok_end - tok_begin + BS - 1) / BS;

    if (threadIdx.x == 0) {
        s_failed = 0;
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        const int32_t* table =
            p.block_tables + seq * p.table_seq_stride + kvh * p.table_kvh_stride + blk_begin;
        const uint64_t policy = l2_policy_evict_first();
        if (p.new_slots != nullptr && tok_end == L) {
            // fused append: this CTA's partition holds the new (last) token; write it
            // before any TMA read of its block
            append_row_warp<ACT, CACHE>(p.k_new, p.v_new, p.new_slots[seq], seq, kvh, p.num_kv_heads, BS, D,
                                        p.num_blocks, const_cast<void*>(p.k_cache), const_cast<void*>(p.v_cache),
                                        p.k_scale, p.v_scale, p.err, lane);
        }
        const unsigned char* kc = static_cast<const unsigned char*>(p.k_cache);
        const unsigned char* vc = static_cast<const unsigned char*>(p.v_cache);
        bool ok = true;
        int issued = 0;
        for (int chunk = 0; chunk < n_blk && ok; chunk += 32) {
            const bool have = chunk + lane < n_blk;
            int phys = have ? table[chunk + lane] : 0;
            const bool bad = have && (phys < 0 || phys >= p.num_blocks);
            if (bad) {
                atomicOr(p.err, kErrBadBlock);
                phys = -1;
            }
            const int chunk_blocks = min(32, n_blk - chunk);
            for (int j = 0; j < chunk_blocks; j += C::BPS) {
                int pb[C::BPS];
#pragma unroll
                for (int bi = 0; bi < C::BPS; ++bi) pb[bi] = __shfl_sync(0xffffffffu, phys, (j + bi) & 31);
                const int st = (chunk + j) / C::BPS;
                if (lane == 0) {
                    const int s = st % C::STAGES;
                    if (st >= C::STAGES && !mbar_wait(&empty[s], ((st / C::STAGES) - 1) & 1)) {
                        atomicOr(p.err, kErrTimeout);
                        ok = false;
                    }
                    if (ok) {
                        uint32_t bytes = 0;
#pragma unroll
                        for (int bi = 0; bi < C::BPS; ++bi)
                            if (j + bi < chunk_blocks && pb[bi] >= 0) bytes += 2 * C::TILE_BYTES;
                        mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
                        for (int bi = 0; bi < C::BPS; ++bi) {
                            if (j + bi < chunk_blocks && pb[bi] >= 0) {
                                const size_t off =
                                    (static_cast<size_t>(pb[bi]) * p.num_kv_heads + kvh) * C::TILE_BYTES;
                                bulk_copy_g2s(kbuf + s * C::STAGE_BYTES + bi * C::TILE_BYTES, kc + off,
                                              C::TILE_BYTES, &full[s], policy);
                                bulk_copy_g2s(vbuf + s * C::STAGE_BYTES + bi * C::TILE_BYTES, vc + off,
                                              C::TILE_BYTES, &full[s], policy);
                            }
                        }
                        ++issued;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
        }
        // Do not leave while copies into this CTA's shared memory are in flight.
        if (lane == 0) {
            const int first = issued > C::STAGES ? issued - C::STAGES : 0;
            for (int st = first; st < issued; ++st) {
                if (!mbar_wait(&full[st % C::STAGES], (st / C::STAGES) & 1)) {
                    atomicOr(p.err, kErrTimeout);
                    break;
                }
            }
        }
        return;
    }

    // ------------------------------- consumers -------------------------------
    const int r = lane / C::LPR;  // token row within a warp-wide load
    const int c = lane % C::LPR;  // 16-byte chunk within the row
    const int h0 = kvh * G;

    const float kmul = CACHE == kE4M3 ? *p.k_scale : 1.0f;
    const float qscale = p.scale_log2 * kmul;
    const uint16_t* qsrc = static_cast<const uint16_t*>(p.q) + (static_cast<size_t>(seq) * p.num_q_heads + h0) * D;

    // An E4M3 cache takes the mixed-precision path: K and V pairs become
    // binary16 pairs (exact), q is held in binary16 (exact for a 16-bit value
    // of magnitude <= 65504, checked per warp), products accumulate in
    // binary32 with fma.rn.f32.f16, and the scale multiplies the reduced dot
    // product.  P·V takes the probability rounded to binary16.
    bool mixed = false;
    if constexpr (CACHE == kE4M3) {
        bool fits = true;
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int v = 0; v < C::VEC; v += 8) {
                const uint4 u = *reinterpret_cast<const uint4*>(qsrc + g * D + c * C::VEC + v);
                const uint16_t* e = reinterpret_cast<const uint16_t*>(&u);
#pragma unroll
                for (int i = 0; i < 8; ++i) fits = fits && fabsf(act_to_float<ACT>(e[i])) <= 65504.f;
            }
        }
        mixed = __all_sync(0xffffffffu, fits);
    }

    float m[G], l[G], acc[G][C::VEC];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int v = 0; v < C::VEC; ++v) acc[g][v] = 0.f;
    }

    auto consume = [&](auto mixed_tag) {
        constexpr bool MIX = decltype(mixed_tag)::value;
        constexpr int QN = MIX ? C::VEC / 2 : C::VEC;
        // float path: q * scale (log2 units, k_scale folded in); mixed path: binary16 pairs of q
        float qf[G][MIX ? 1 : C::VEC];
        uint32_t qh[G][MIX ? QN : 1];
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int v = 0; v < C::VEC; v += 8) {
                const uint4 u = *reinterpret_cast<const uint4*>(qsrc + g * D + c * C::VEC + v);
                const uint16_t* e = reinterpret_cast<const uint16_t*>(&u);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float x = act_to_float<ACT>(e[i]);
                    if constexpr (MIX) {
                        const uint32_t h = __half_as_ushort(__float2half_rn(x));
                        if (i % 2 == 0) qh[g][(v + i) / 2] = h;
                        else qh[g][(v + i) / 2] |= h << 16;
                    } else {
                        qf[g][v + i] = x * qscale;
                    }
                }
            }
        }

        for (int st = 0; st < n_stage; ++st) {
            const int s = st % C::STAGES;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (st / C::STAGES) & 1))) {
                if (lane == 0) {
                    atomicOr(p.err, kErrTimeout);
                    s_failed = 1;
                }
                break;
            }
            const unsigned char* kb = kbuf + s * C::STAGE_BYTES;
            const unsigned char* vb = vbuf + s * C::STAGE_BYTES;
            const int tok0 = tok_begin + st * kStageTokens;

            float sc[C::PASSES][G];
#pragma unroll
            for (int pp = 0; pp < C::PASSES; ++pp) {
                const int tt = warp * C::TW + pp * C::TPP + r;
                const bool valid = tok0 + tt < tok_end;
                const uint4 u = *reinterpret_cast<const uint4*>(kb + (tt * D * C::E) + c * 16);
                if constexpr (MIX) {
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                    uint32_t kh[QN];
#pragma unroll
                    for (int i = 0; i < QN; ++i)
                        kh[i] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i / 2] >> (16 * (i % 2))));
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float d0 = 0.f, d1 = 0.f;
#pragma unroll
                        for (int i = 0; i < QN; ++i) fma_f16x2_f32(qh[g][i], kh[i], d0, d1);
                        float d = d0 + d1;
#pragma unroll
                        for (int off = C::LPR / 2; off >= 1; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
                        sc[pp][g] = valid ? d * qscale : -INFINITY;
                    }
                } else {
                    float kf[C::VEC];
                    Vec16<CACHE>::to_float(u, kf);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float d = 0.f;
#pragma unroll
                        for (int v = 0; v < C::VEC; ++v) d = fmaf(qf[g][v], kf[v], d);
#pragma unroll
                        for (int off = C::LPR / 2; off >= 1; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
                        sc[pp][g] = valid ? d : -INFINITY;
                    }
                }
            }

            float pr[C::PASSES][G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float mx = sc[0][g];
#pragma unroll
                for (int pp = 1; pp < C::PASSES; ++pp) mx = fmaxf(mx, sc[pp][g]);
#pragma unroll
                for (int off = C::LPR; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                // Lazy rescaling: the reference max m moves only when the
                // stage max exceeds it by more than kRescaleLog2 (warp-uniform
                // test), so probabilities stay below 2^kRescaleLog2 and l and
                // acc, both relative to m, stay consistent.
                if (mx > m[g] + kRescaleLog2) {
                    const float alpha = m[g] == -INFINITY ? 0.f : fast_exp2(m[g] - mx);
                    m[g] = mx;
                    l[g] *= alpha;
#pragma unroll
                    for (int v = 0; v < C::VEC; ++v) acc[g][v] *= alpha;
                }
#pragma unroll
                for (int pp = 0; pp < C::PASSES; ++pp) {
                    pr[pp][g] = sc[pp][g] == -INFINITY ? 0.f : fast_exp2(sc[pp][g] - m[g]);
                    l[g] += pr[pp][g];
                }
            }

#pragma unroll
            for (int pp = 0; pp < C::PASSES; ++pp) {
                const int tt = warp * C::TW + pp * C::TPP + r;
                if (tok0 + tt < tok_end) {
                    const uint4 u = *reinterpret_cast<const uint4*>(vb + (tt * D * C::E) + c * 16);
                    if constexpr (MIX) {
                        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int i = 0; i < QN; ++i) {
                            const uint32_t vh = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i / 2] >> (16 * (i % 2))));
#pragma unroll
                            for (int g = 0; g < G; ++g)
                                fma_f16s_f32(__half_as_ushort(__float2half_rn(pr[pp][g])), vh, acc[g][2 * i],
                                             acc[g][2 * i + 1]);
                        }
                    } else {
                        float vf[C::VEC];
                        Vec16<CACHE>::to_float(u, vf);
#pragma unroll
                        for (int g = 0; g < G; ++g)
#pragma unroll
                            for (int v = 0; v < C::VEC; ++v) acc[g][v] = fmaf(pr[pp][g], vf[v], acc[g][v]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    };
    if constexpr (CACHE == kE4M3) {
        if (mixed) consume(std::true_type{});
        else consume(std::false_type{});
    } else {
        consume(std::false_type{});
    }

    // Merge the token rows of this warp: lanes of equal chunk c hold partial sums.
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int off = C::LPR; off < 32; off <<= 1) {
            l[g] += __shfl_xor_sync(0xffffffffu, l[g], off);
#pragma unroll
            for (int v = 0; v < C::VEC; ++v) acc[g][v] += __shfl_xor_sync(0xffffffffu, acc[g][v], off);
        }
    }
    if (r == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int v = 0; v < C::VEC; ++v) red_acc[(warp * G + g) * D + c * C::VEC + v] = acc[g][v];
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            red_m[warp * G + g] = m[g];
            red_l[warp * G + g] = l[g];
        }
    }
    // all consumer warps (not the producer) meet here
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    if (s_failed) return;

    const float vmul = CACHE == kE4M3 ? *p.v_scale : 1.0f;
    const int tid = threadIdx.x;
    const bool single = p.max_parts == 1 || L <= p.partition_size;  // per (seq, kvh) length
    for (int idx = tid; idx < G * D; idx += kConsumerWarps * 32) {
        const int g = idx / D;
        const int d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_m[w * G + g]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = red_m[w * G + g];
            const float wt = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
            num = fmaf(wt, red_acc[(w * G + g) * D + d], num);
            den = fmaf(wt, red_l[w * G + g], den);
        }
        const float o = num / den * vmul;
        const size_t row = static_cast<size_t>(seq) * p.num_q_heads + h0 + g;
        if (single) {
            static_cast<uint16_t*>(p.out)[row * D + d] = float_to_act<ACT>(o);
        } else {
            const size_t slot = row * p.max_parts + part;
            p.ws_o[slot * D + d] = o;
            if (d == 0) {
                p.ws_ml[slot * 2] = M;
                p.ws_ml[slot * 2 + 1] = den;
            }
        }
    }
}

}  // namespace pkv
