// Paged decode attention for grouped-query heads on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory), sm_103a.
//
// Same result as the CUDA-core kernel (decode.cuh): for sequence b, kv head
// kvh and its G query heads, softmax(scale * q K^T) V over the context,
// gathered block by block through the block table (Ultralytics glossary
// "PagedAttention", section "How paging works"; query heads sharing a KV
// head: section "Related techniques").  When G query heads read the same
// K/V, the step is a real dense product: S = K Q^T is [tokens x G] and
// O = V^T P is [D x G], so it runs on the tensor cores and the K/V bytes are
// read once for all G heads.
//
// Work item: (sequence, kv head, partition of up to 512 tokens).  Only
// non-empty items are numbered, in an order that keeps the tail short: every
// row's full partitions first, then each row's last, partly filled partition,
// longest first (8 length buckets; a stable counting sort in shared memory
// that every CTA computes alike).
// The kernel is persistent and balances ragged lengths dynamically: the
// scheduler warp of each CTA claims the next item number from a counter in the
// workspace (zeroed before the launch) and passes it, with the item's block-
// table entries, to the other roles through a 2-entry queue in shared memory
// (a deeper queue leaves more claimed work per CTA when the counter runs dry).
// Roles (256 threads):
//  warp 0    scheduler: claims, block-table entries, the fused append (fenced
//            for the copy engine before the item is published), and for an
//            E4M3 cache the exact power-of-2 scale of the item's queries.
//  warps 6-7 producers: 2-D TMA loads (128-byte swizzle) of each (block, kv
//            head) tile into a ring of 128-token stages, warp 6 the even
//            stage uses and Q, warp 7 the odd uses.  16-bit caches: a tile is
//            two 64-column halves of head_dim; E4M3: one 128-byte row per
//            token.  Order: K(0), then for each item n: K(n+1), V(n).
//  warp 1    MMA: S = K Q^T (M = 128 tokens, N = 16, K = 128) into a
//            16-column slot per tile; O = V^T P (M = 128 = D, N = 16, K =
//            tokens).  Order: S(0), then for each n: S(n+1), O(n).  16-bit:
//            kind::f16; E4M3: kind::f8f6f4 with q and P as E4M3 high + low
//            parts in rows 0-7 and 8-15 of the N = 16 operand.
//  warps 2-5 softmax + epilogue: thread i owns tensor-memory lane i (token i
//            of a tile for S, dimension i of O).  Partition-wide max and sum
//            per head (the whole partition's scores sit in tensor memory, so
//            there is no online rescaling), P written in the MMA's shared
//            memory layout, then the output (one partition) or the split-K
//            partial (m, l, O/l).  Order: softmax(0), then for each n:
//            softmax(n+1), epilogue(n).
// S and O (tensor memory) are double-buffered by item parity, so the MMA and
// softmax roles run one item ahead of the epilogue; Q is single, P single
// (16-bit) or double (E4M3).  With 16-bit operands N = 16 columns are
// computed for at most 8 heads: rows 8-15 of the Q and P operands alias the
// next 1 KB of shared memory, and the matching output columns are never read.
// head_dim 64 (PAIR): an item covers kv heads 2v and 2v+1 of a sequence (the
// two share its block table), laid side by side as one 128-wide head: tile
// half h holds kv head 2v+h, and the Q operand is block-diagonal (rows 0-7:
// the queries of 2v on dimensions 0-63, rows 8-15: those of 2v+1 on 64-127,
// zeros elsewhere), so S columns 0-7 and 8-15 are the two heads' scores.  P
// fills all 16 rows; O = V^T P is right on dimensions 0-63 in columns 0-7 and
// on 64-127 in columns 8-15, the only ones read.  The K/V bytes per item and
// the MMA shapes are those of head_dim 128.
// Every barrier wait is bounded (kWaitLimitNs); on a timeout the CTA stops
// issuing work, drains its in-flight copies and MMAs, frees tensor memory and
// reports kErrTimeout.
#pragma once

#include "kernels.h"
#include "pkv_tc.cuh"

namespace pkv {

constexpr int kTcThreads = 256;
constexpr int kTcTile = 128;                  // tokens per tile (MMA M of S = K Q^T)
constexpr int kTcMaxTiles = 4;                // partitions of at most 512 tokens
constexpr int kTcD = 128;                     // head_dim served by this kernel
constexpr int kTcN = 16;                      // MMA N: query heads padded to 16
constexpr int kTcHalf = kTcTile * 128;        // one 64-column half of a tile: 128 rows x 128 B
constexpr int kTcStage = 2 * kTcHalf;         // 32 KB
constexpr int kTcStage8 = kTcTile * kTcD;     // E4M3 cache: 128 tokens x 128 one-byte codes, 16 KB
constexpr int kTcQBuf = 3 * 1024;             // Q: two 8-row halves + 1 KB that rows 8-15 of half 1 alias
constexpr int kTcPBuf = (2 * kTcMaxTiles + 1) * 1024;  // P: tile x token-half 8-row regions + alias pad
constexpr int kTcSlotCols = kTcMaxTiles * kTcN + kTcN;  // S (4 x 16) + O (16) per buffer
constexpr int kTcTmemCols = 256;              // two buffers of 80 columns, rounded to a power of 2
constexpr int kTcMaxSeqs = 2048;              // sequences served (lengths and item prefix in shared memory)
constexpr int kTcSmemPerSm = 228 * 1024;      // shared memory of one SM, including the 1 KB each CTA reserves
constexpr int kTcQueue = 2;                   // claimed items in flight between the roles
constexpr int kTcLenBuckets = 8;              // length buckets of the partly filled partitions

template <int NS, int STG = kTcStage, bool PAIR = false>
struct TcSmem {
    static constexpr int RING = 0;
    static constexpr int Q = NS * STG;
    // E4M3 cache: two 4 KB Q buffers (high + middle parts, low part + 8 zero
    // rows) and two 8 KB P buffers (4 tiles x 16 rows x 128 one-byte codes).
    // Pairs of head_dim-64 kv heads: a 4 KB Q buffer (two 8-row regions of
    // queries around 2 KB of zeros) and a 16 KB P buffer (16 rows per region).
    static constexpr int QBUF = STG == kTcStage8 || PAIR ? 4096 : kTcQBuf;  // one Q buffer
    static constexpr int QBUFS = STG == kTcStage8 ? 2 : 1;                  // Q buffers
    static constexpr int P = Q + QBUFS * QBUF;
    static constexpr int PBUF = STG == kTcStage8 ? 8192 : PAIR ? 2 * kTcMaxTiles * 2048 : kTcPBuf;  // one P buffer
    static constexpr int PBUFS = STG == kTcStage8 ? 2 : 1;           // P buffers
    static constexpr int QUEUE = P + PBUFS * PBUF;  // item numbers, q shifts, block-table entries [32] per entry
    static constexpr int BARS = (QUEUE + 2 * kTcQueue * 4 + kTcQueue * 32 * 4 + 7) / 8 * 8;
    // full[NS], empty[NS], q_full[2], q_empty[2], s_full[2], p_full[2], o_full[2], o_free[2], final,
    // item_full[kTcQueue], item_empty[kTcQueue] (a single Q or P buffer uses entry 0 of its pair)
    static constexpr int NBARS = 2 * NS + 13 + 2 * kTcQueue;
    static constexpr int RED = BARS + NBARS * 8;
    static constexpr int RED_FLOATS = 64 + 64;  // red_max[4][8], red_sum[4][8], stats[2][2][2][8]
    static constexpr int MISC = RED + RED_FLOATS * 4;
    // per row: length (int), item prefix (int, rows + 2 entries), length order (uint16)
    static constexpr int ROWS = (MISC + 16 + 15) / 16 * 16;
    __host__ __device__ static constexpr int bytes(int rows) { return ROWS + rows * 4 + (rows + 2) * 4 + rows * 2; }
    __host__ __device__ static constexpr int alloc(int rows) { return bytes(rows) + 1024; }  // room to align the base
};

struct TcItem {
    int seq, kvh, row, part, tok_begin, n_tok, n_tiles;
    int qshift;  // E4M3 cache: q enters the MMA scaled by 2^-qshift
};

// Rows: a sequence (tables shared by its kv heads) or, with per-(sequence,
// kv head) tables, one (sequence, kv head) pair; row r has length
// context_lens[r] either way.
__device__ __forceinline__ bool tc_per_kvh(const DecodeParams& p) { return p.table_kvh_stride != 0; }
__device__ __forceinline__ int tc_rows(const DecodeParams& p) {
    return tc_per_kvh(p) ? p.num_seqs * p.num_kv_heads : p.num_seqs;
}

// Item number ci -> (sequence, kv head, partition).  Items [0, F), F =
// prefix[rows], are full partitions: prefix[r] counts those of the rows
// before r, a row of L tokens has floor(L / partition_size) of them per kv
// head it covers, kv head major.  Items [F, F + H * prefix[rows + 1]) are the
// partly filled last partitions of the rows listed in `order`, H per row
// (H = the item heads a row covers: its kv heads, or at head_dim 64 the pairs
// of kv heads, when it.kvh is the pair's index).
__device__ __forceinline__ void tc_decode_item(int ci, const DecodeParams& p, const int* lens, const int* prefix,
                                               const uint16_t* order, int H, TcItem& it) {
    const int rows = tc_rows(p);
    const int F = prefix[rows];
    int row, part, h;
    if (ci < F) {
        int lo = 0, hi = rows;  // the last r with prefix[r] <= ci
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= ci) lo = mid;
            else hi = mid;
        }
        row = lo;
        const int nfull = lens[row] / p.partition_size;
        const int r = ci - prefix[row];
        h = r / nfull;
        part = r - h * nfull;
    } else {
        const int j = ci - F;
        const int idx = j / H;
        row = order[idx];
        h = j - idx * H;
        part = lens[row] / p.partition_size;
    }
    const int L = lens[row];
    it.row = row;
    if (tc_per_kvh(p)) {
        it.seq = row / p.num_kv_heads;
        it.kvh = row - it.seq * p.num_kv_heads;
    } else {
        it.seq = row;
        it.kvh = h;
    }
    it.part = part;
    it.tok_begin = part * p.partition_size;
    it.n_tok = min(p.partition_size, L - it.tok_begin);
    it.n_tiles = (it.n_tok + kTcTile - 1) / kTcTile;
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

// Named barrier over `count` threads that also ORs a predicate across them.
__device__ __forceinline__ int named_bar_or(int id, int count, int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.b32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred), "r"(id), "r"(count)
        : "memory");
    return r;
}

// x0, x1 -> E4M3 codes hi (nearest) and lo (nearest to the exact remainder
// x - hi), x0 in the low byte of each.  hi + lo carries about 8 significant
// bits of x; the remainder is exact in binary32 (hi lies within a factor of 2
// of x).
__device__ __forceinline__ void split_e4m3x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
    __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
    const float2 hv = __half22float2(*reinterpret_cast<__half2*>(&hr));
    hi = h;
    lo = __nv_cvt_float2_to_fp8x2(make_float2(x0 - hv.x, x1 - hv.y), __NV_SATFINITE, __NV_E4M3);
}

// x0, x1 -> three E4M3 codes each, hi + mid + lo carrying about 12
// significant bits (enough for binary16 queries).
__device__ __forceinline__ void split3_e4m3x2(float x0, float x1, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
    const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
    __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
    const float2 hv = __half22float2(*reinterpret_cast<__half2*>(&hr));
    hi = h;
    split_e4m3x2(x0 - hv.x, x1 - hv.y, mid, lo);
}

template <int ACT, int CACHE, int BS, int G, int NS, bool PAIR = false>
__global__ void __launch_bounds__(kTcThreads, 2)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const __grid_constant__ CUtensorMap qmap, const DecodeParams p) {
    constexpr bool FP8 = CACHE == kE4M3;
    constexpr int STG = FP8 ? kTcStage8 : kTcStage;  // bytes of one ring stage
    // PAIR: head_dim 64, kv heads 2v and 2v+1 of a sequence in one item, as
    // dimensions 0-63 and 64-127 of a 128-wide head (tile halves, Q regions)
    constexpr int HD = PAIR ? 64 : kTcD;  // head_dim of the caches, queries and output
    static_assert(!PAIR || !FP8, "pairs of head_dim-64 kv heads: 16-bit caches");
    using S = TcSmem<NS, STG, PAIR>;
    constexpr int THREADS = kTcThreads;
    constexpr int BPT = kTcTile / BS;  // blocks per tile
    // E4M3 x E4M3 (kind::f8f6f4) has the same descriptor bits as binary16 x binary16
    constexpr uint32_t IDESC_S = tc::idesc_f16(128, kTcN, !FP8 && ACT == kBF16, false, false);
    // E4M3: P is the B operand in the MN-major layout without swizzle (a token's
    // 16 codes, 8 high and 8 low parts, are 16 contiguous bytes)
    constexpr uint32_t IDESC_O = tc::idesc_f16(128, kTcN, !FP8 && ACT == kBF16, true, FP8);
    static_assert(!FP8 || G <= 8, "E4M3 cache: rows 0-7 of Q and P hold the high parts, rows 8-15 the low parts");
    constexpr bool Q3 = FP8 && ACT == kF16;  // binary16 queries: three E4M3 parts
    static_assert(G == 2 || G == 4 || G == 8, "query heads per kv head");
    static_assert(kTcMaxTiles * kTcTile / BS <= 32, "one warp holds the table entries of an item");

    // the merge kernel may be scheduled now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;");
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* ring = sm + S::RING;
    unsigned char* qbuf = sm + S::Q;
    unsigned char* pbuf = sm + S::P;
    volatile int* item_q = reinterpret_cast<volatile int*>(sm + S::QUEUE);
    volatile int* item_shift = item_q + kTcQueue;
    volatile int* item_phys = item_shift + kTcQueue;  // [slot][32]: the item's physical blocks
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::BARS);
    uint64_t* full = bars;
    uint64_t* empty = bars + NS;
    uint64_t* q_full = bars + 2 * NS;
    uint64_t* q_empty = q_full + 2;
    uint64_t* s_full = q_full + 4;
    uint64_t* p_full = q_full + 6;
    uint64_t* o_full = q_full + 8;
    uint64_t* o_free = q_full + 10;
    uint64_t* final_bar = q_full + 12;
    uint64_t* item_full = q_full + 13;
    uint64_t* item_empty = item_full + kTcQueue;
    float* red_max = reinterpret_cast<float*>(sm + S::RED);
    float* red_sum = red_max + 32;
    float* stats = red_max + 64;  // [buffer][kv head of a pair][max, sum][8]
    uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(sm + S::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + S::MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int B = tc_rows(p);  // rows: <= kTcMaxSeqs (checked on the host)
    int* s_lens = reinterpret_cast<int*>(sm + S::ROWS);
    int* s_prefix = s_lens + B;
    uint16_t* s_order = reinterpret_cast<uint16_t*>(s_prefix + B + 2);
    // item heads per row (per-(sequence, kv head) tables: one; pairs need shared tables)
    const int heads_per_row = tc_per_kvh(p) ? 1 : PAIR ? p.num_kv_heads / 2 : p.num_kv_heads;

    // Lengths, the exclusive prefix of full-partition items per row and the
    // rows with a partly filled partition sorted by its length, longest first
    // (a row with a length outside 1..max_blocks*BS has no items).  Each
    // thread owns a contiguous chunk of rows; one block-wide scan gives the
    // full-item prefix and every bucket's offsets, so the order is the same in
    // every CTA.
    {
        constexpr int NBK = kTcLenBuckets;
        const int chunk = (B + THREADS - 1) / THREADS;
        const int s0 = min(B, threadIdx.x * chunk), s1 = min(B, s0 + chunk);
        auto bucket_of = [&](int L) { return (L % p.partition_size) * NBK / p.partition_size; };
        auto valid_len = [&](int L) { return L >= 1 && L <= p.max_blocks_per_seq * BS; };
        int cnt[NBK + 1] = {};  // [0]: full items, [1 + k]: rows in length bucket k
        for (int s = s0; s < s1; ++s) {
            const int L = p.context_lens[s];
            s_lens[s] = L;
            if (!valid_len(L)) continue;
            cnt[0] += heads_per_row * (L / p.partition_size);
            if (L % p.partition_size != 0) {
                const int k = bucket_of(L);
#pragma unroll
                for (int kk = 0; kk < NBK; ++kk) cnt[1 + kk] += kk == k;
            }
        }
        int incl[NBK + 1];
#pragma unroll
        for (int k = 0; k <= NBK; ++k) {
            incl[k] = cnt[k];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl[k], off);
                if (lane >= off) incl[k] += v;
            }
        }
        int* warp_tot = reinterpret_cast<int*>(red_max);  // [warps][NBK + 1]
        if (lane == 31) {
#pragma unroll
            for (int k = 0; k <= NBK; ++k) warp_tot[warp * (NBK + 1) + k] = incl[k];
        }
        __syncthreads();
        int run[NBK + 1], total[NBK + 1];
#pragma unroll
        for (int k = 0; k <= NBK; ++k) {
            int before = 0, all = 0;
            for (int w = 0; w < THREADS / 32; ++w) {
                const int t = warp_tot[w * (NBK + 1) + k];
                if (w < warp) before += t;
                all += t;
            }
            run[k] = before + incl[k] - cnt[k];
            total[k] = all;
        }
        // bucket k starts after the rows of the longer buckets k+1 .. NBK-1
#pragma unroll
        for (int k = 0; k < NBK; ++k) {
            int start = 0;
#pragma unroll
            for (int k2 = k + 1; k2 < NBK; ++k2) start += total[1 + k2];
            run[1 + k] += start;
        }
        for (int s = s0; s < s1; ++s) {
            s_prefix[s] = run[0];
            const int L = s_lens[s];
            if (!valid_len(L)) continue;
            run[0] += heads_per_row * (L / p.partition_size);
            if (L % p.partition_size != 0) {
                const int k = bucket_of(L);
#pragma unroll
                for (int kk = 0; kk < NBK; ++kk)
                    if (kk == k) s_order[run[1 + kk]++] = static_cast<uint16_t>(s);
            }
        }
        if (threadIdx.x == 0) {
            int partial = 0;
#pragma unroll
            for (int k = 0; k < NBK; ++k) partial += total[1 + k];
            s_prefix[B] = total[0];
            s_prefix[B + 1] = partial;
        }
    }
    if constexpr (PAIR) {
        // rows 8-15 of the dimension 0-63 Q operand and rows 0-7 of the 64-127
        // one: zero for the whole launch (the sync below orders them before any MMA)
        for (int i = threadIdx.x; i < 2048 / 16; i += THREADS)
            reinterpret_cast<uint4*>(qbuf + 1024)[i] = make_uint4(0u, 0u, 0u, 0u);
        tc::fence_proxy_async_smem();
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 13; ++i) mbar_init(&q_full[i], 1);
        for (int i = 0; i < kTcQueue; ++i) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], 4);  // the two tile producers, the MMA warp and the softmax warps
        }
        *abort_flag = 0;
        mbar_init_fence();
        tc::prefetch_tensormap(&kmap);
        tc::prefetch_tensormap(&vmap);
        if constexpr (!FP8) tc::prefetch_tensormap(&qmap);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_base_smem, kTcTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_base_smem;
    const int total = s_prefix[B] + heads_per_row * s_prefix[B + 1];

    const uint64_t policy = l2_policy_evict_first();
    // Two producer warps share the ring: one arms the even stage uses, the other
    // the odd ones (the lanes of one copy instruction are issued one after the
    // other, so a single warp cannot issue the small copies fast enough).  Both
    // follow the same tile order; `use` counts every tile, armed here or not.
    // Arm one ring stage with tile t of an item; `map` is the K or V tensor map.
    // Lane 0 waits for the stage and sets its byte count; lane 2j+h then loads
    // half h of block j of the tile, so one warp instruction issues the tile's
    // 2*BPT copies (PAIR: half h is block j of kv head 2v+h).  E4M3: a token's
    // 128 codes are one 128-byte row, so lane j loads block j whole.
    auto issue_tile = [&](uint32_t& use, uint32_t parity, const TcItem& it, int phys, int t,
                          const CUtensorMap* map) {
        if ((use & 1u) != parity) {
            ++use;
            return true;
        }
        constexpr int PER_BLOCK = FP8 ? 1 : 2;  // copies per block
        const int n_blk = (it.n_tok + BS - 1) / BS;
        const int j = (lane / PER_BLOCK) < BPT ? (lane / PER_BLOCK) : 0;
        const int half = FP8 ? 0 : (lane & 1);
        const int pbj = __shfl_sync(0xffffffffu, phys, (t * BPT + j) & 31);
        const bool mine = lane < PER_BLOCK * BPT && t * BPT + j < n_blk && pbj >= 0;
        const unsigned loads = __ballot_sync(0xffffffffu, mine);
        const int s = use % NS;
        bool good = true;
        if (lane == 0) {
            if (use >= NS) good = tc_wait(&empty[s], ((use / NS) - 1) & 1, abort_flag, p.err);
            if (good) mbar_arrive_expect_tx(&full[s], __popc(loads) * (BS * 128));
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) return false;
        if (mine) {
            const int y = (pbj * p.num_kv_heads + (PAIR ? 2 * it.kvh + half : it.kvh)) * BS;
            tc::tma_load_2d(ring + s * STG + half * kTcHalf + j * BS * 128, map, PAIR ? 0 : half * 64, y, &full[s],
                            policy);
        }
        ++use;
        return true;
    };
    // A producer leaves only when every copy it issued into this CTA's shared
    // memory has landed.
    auto drain = [&](uint32_t use, uint32_t parity) {
        if (lane == 0) {
            const uint32_t first = use > static_cast<uint32_t>(NS) ? use - NS : 0;
            for (uint32_t u = first; u < use; ++u)
                if ((u & 1u) == parity && !mbar_wait(&full[u % NS], (u / NS) & 1)) atomicOr(p.err, kErrTimeout);
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------------ scheduler
        // Claims items, reads their block-table entries, performs the fused
        // append and publishes each item through the queue, up to kTcQueue
        // ahead of the slowest reader.
        int nclaim = 0;  // queue entries written so far
        bool ok = true;
        if (lane == 0) {
            // sequences with a context length outside 1..max_blocks*BS are skipped; report them once
            for (int s = blockIdx.x; s < B; s += gridDim.x) {
                const int L = s_lens[s];
                if (L < 1 || L > p.max_blocks_per_seq * BS) atomicOr(p.err, kErrBadLen);
            }
        }
        auto table_entry = [&](const TcItem& it) {
            const int n_blk = (it.n_tok + BS - 1) / BS;
            int phys = -1;
            if (lane < n_blk) {
                phys = p.block_tables[it.seq * p.table_seq_stride + it.kvh * p.table_kvh_stride + it.tok_begin / BS +
                                      lane];
                if (phys < 0 || phys >= p.num_blocks) {
                    atomicOr(p.err, kErrBadBlock);
                    phys = -1;
                }
            }
            return phys;
        };
        // Claim the next item for this CTA and pass it to the other roles; false
        // at the end of the work (the end marker is queued) or on an abort.
        auto claim = [&](TcItem& it, int& phys) {
            phys = -1;
            int ci = -1;
            if (lane == 0) {
                ci = atomicAdd(p.work_counter, 1);
                if (ci >= total) ci = -1;
            }
            ci = __shfl_sync(0xffffffffu, ci, 0);
            it.qshift = 0;
            if (ci >= 0) {
                tc_decode_item(ci, p, s_lens, s_prefix, s_order, heads_per_row, it);
                if constexpr (FP8) {
                    // q enters the MMA as E4M3 high and low parts of q x 2^-qshift:
                    // the exact power-of-2 scale puts its largest magnitude in
                    // [128, 256), below the E4M3 maximum of 448
                    const uint16_t* qg = static_cast<const uint16_t*>(p.q) +
                                         (static_cast<int64_t>(it.seq) * p.num_q_heads + it.kvh * G) * kTcD;
                    float m = 0.f;
                    for (int i = lane; i < G * kTcD / 8; i += 32) {
                        const uint4 u = *reinterpret_cast<const uint4*>(qg + i * 8);
                        const uint16_t* e = reinterpret_cast<const uint16_t*>(&u);
#pragma unroll
                        for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(act_to_float<ACT>(e[j])));
                    }
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                    const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xff) - 127;  // floor(log2 m)
                    it.qshift = m > 0.f ? min(120, max(-120, e - 7)) : 0;
                }
                phys = table_entry(it);
                if (p.new_slots != nullptr && it.tok_begin + it.n_tok == s_lens[it.row]) {
                    // fused append: this item holds the new (last) token; write it
                    // before the item is published, so before any copy of its block
#pragma unroll
                    for (int h = 0; h < (PAIR ? 2 : 1); ++h)
                        append_row_warp<ACT, CACHE>(p.k_new, p.v_new, p.new_slots[it.seq], it.seq,
                                                    PAIR ? 2 * it.kvh + h : it.kvh, p.num_kv_heads, BS, HD,
                                                    p.num_blocks, const_cast<void*>(p.k_cache),
                                                    const_cast<void*>(p.v_cache), p.k_scale, p.v_scale, p.err, lane);
                }
            }
            const int slot = nclaim % kTcQueue;
            bool good = true;
            if (lane == 0 && nclaim >= kTcQueue)
                good = tc_wait(&item_empty[slot], ((nclaim / kTcQueue) - 1) & 1, abort_flag, p.err);
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
                ok = false;
                return false;
            }
            item_phys[slot * 32 + lane] = phys;
            if (lane == 0) {
                item_q[slot] = ci;
                item_shift[slot] = it.qshift;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_full[slot]);
            ++nclaim;
            return ci >= 0;
        };
        TcItem it;
        int phys = -1;
        while (ok && claim(it, phys)) {
        }
    } else if (warp >= 6) {
        // ------------------------------------------------------ tile producers
        // Warp 6 arms the even stage uses and writes Q, warp 7 arms the odd
        // uses.  Both read the items from the queue and follow one tile order:
        // K(0), then for each n: K(n+1), V(n).
        const uint32_t parity = static_cast<uint32_t>(warp - 6);
        uint32_t use = 0;  // ring stage uses so far (either parity)
        int nq = 0;        // Q tiles written so far
        int nread = 0;
        if constexpr (Q3) {
            // rows 8-15 of the low-part operand stay zero (made visible to the
            // MMA by the fence before the first Q is published)
            if (parity == 0)
                for (int i = lane; i < 64 * S::QBUFS; i += 32)
                    reinterpret_cast<uint4*>(qbuf + (i >> 6) * S::QBUF + 3072)[i & 63] = make_uint4(0u, 0u, 0u, 0u);
        }
        auto read_item = [&](TcItem& it, int& phys) {
            const int slot = nread % kTcQueue;
            const bool good =
                __all_sync(0xffffffffu, tc_wait(&item_full[slot], (nread / kTcQueue) & 1, abort_flag, p.err));
            ++nread;
            if (!good) return -1;
            const int ci = item_q[slot];
            it.qshift = item_shift[slot];
            phys = item_phys[slot * 32 + lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (ci < 0) return 0;
            // (an appended row of this item was written, and fenced for the copy
            // engine, by the scheduler before it published the item)
            tc_decode_item(ci, p, s_lens, s_prefix, s_order, heads_per_row, it);
            return 1;
        };
        auto issue_q = [&](const TcItem& it, int k) {
            bool good = true;
            if constexpr (FP8) {
                // Q x 2^-qshift = hi + lo, both E4M3 (hi the nearest code, lo the
                // nearest code to the exact remainder: about 8 significant bits in
                // all, so every bfloat16 query is exact), written as the MMA's B
                // operand in the 128-byte swizzled layout: row g holds hi of head
                // g, row 8 + g lo (1 KB further).  Binary16 queries (11 bits) take
                // a third part: rows 8 + g hold the middle part and the low part
                // sits in a second operand 2 KB further, over 8 zero rows, so that a
                // second MMA adds K lo^T into the same accumulator columns.
                // two Q buffers: item k's Q goes in once the S MMAs of item k-2 have read it
                const int qb = k & 1;
                if (lane == 0 && k >= 2) good = tc_wait(&q_empty[qb], ((k >> 1) - 1) & 1, abort_flag, p.err);
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) return false;
                unsigned char* qbuf_k = qbuf + qb * S::QBUF;
                const float f = __uint_as_float(static_cast<uint32_t>(127 - it.qshift) << 23);  // 2^-qshift
                const uint16_t* qg = static_cast<const uint16_t*>(p.q) +
                                     (static_cast<int64_t>(it.seq) * p.num_q_heads + it.kvh * G) * kTcD;
                for (int i = lane; i < G * kTcD / 16; i += 32) {
                    const int g = i >> 3, c = i & 7;  // head, 16-column chunk
                    const uint4 u0 = *reinterpret_cast<const uint4*>(qg + g * kTcD + c * 16);
                    const uint4 u1 = *reinterpret_cast<const uint4*>(qg + g * kTcD + c * 16 + 8);
                    const uint32_t e[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                    uint32_t hw[4], mw[4], lw[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t hb[2], mb[2], lb[2];
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const uint32_t w = e[2 * j + h2];
                            const float x0 = act_to_float<ACT>(static_cast<uint16_t>(w & 0xffffu)) * f;
                            const float x1 = act_to_float<ACT>(static_cast<uint16_t>(w >> 16)) * f;
                            if constexpr (Q3) split3_e4m3x2(x0, x1, hb[h2], mb[h2], lb[h2]);
                            else split_e4m3x2(x0, x1, hb[h2], mb[h2]);
                        }
                        hw[j] = hb[0] | (hb[1] << 16);
                        mw[j] = mb[0] | (mb[1] << 16);
                        if constexpr (Q3) lw[j] = lb[0] | (lb[1] << 16);
                    }
                    const int off = g * 128 + ((c ^ g) * 16);
                    *reinterpret_cast<uint4*>(qbuf_k + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4*>(qbuf_k + 1024 + off) = make_uint4(mw[0], mw[1], mw[2], mw[3]);
                    if constexpr (Q3)
                        *reinterpret_cast<uint4*>(qbuf_k + 2048 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_full[qb]);
                ++nq;
                return true;
            }
            if (lane == 0) {
                // one Q buffer: item k's Q loads once the S MMAs of item k-1 have read it
                if (k >= 1) good = tc_wait(&q_empty[0], (k - 1) & 1, abort_flag, p.err);
                if (good) {
                    mbar_arrive_expect_tx(&q_full[0], 2 * G * 128);
                    if constexpr (PAIR) {
                        // the queries of kv head 2v (rows 0-7 of the first operand) and
                        // of 2v+1 (rows 8-15 of the second, 3 KB in)
                        const int row = it.seq * p.num_q_heads + 2 * it.kvh * G;
                        tc::tma_load_2d(qbuf, &qmap, 0, row, &q_full[0], policy);
                        tc::tma_load_2d(qbuf + 3072, &qmap, 0, row + G, &q_full[0], policy);
                    } else {
                        const int row = it.seq * p.num_q_heads + it.kvh * G;
                        tc::tma_load_2d(qbuf, &qmap, 0, row, &q_full[0], policy);
                        tc::tma_load_2d(qbuf + 1024, &qmap, 64, row, &q_full[0], policy);
                    }
                }
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) return false;
            ++nq;
            return true;
        };

        auto issue_k = [&](const TcItem& it, int phys, int k) {
            // 16-bit: Q first (one TMA issue); E4M3: the K copies first, so that
            // their latency covers the Q conversion
            if (!FP8 && parity == 0 && !issue_q(it, k)) return false;
            for (int t = 0; t < it.n_tiles; ++t)
                if (!issue_tile(use, parity, it, phys, t, &kmap)) return false;
            return !FP8 || parity != 0 || issue_q(it, k);
        };
        TcItem cur, nxt;
        int phys_c = -1, phys_n = -1;
        int rc = read_item(cur, phys_c);
        bool ok = rc >= 0;
        if (rc > 0) ok = issue_k(cur, phys_c, 0);
        for (int k = 0; rc > 0 && ok; ++k) {
            const int rn = read_item(nxt, phys_n);
            if (rn < 0) break;
            if (rn > 0) ok = issue_k(nxt, phys_n, k + 1);
            for (int t = 0; ok && t < cur.n_tiles; ++t) ok = issue_tile(use, parity, cur, phys_c, t, &vmap);
            rc = rn;
            cur = nxt;
            phys_c = phys_n;
        }
        drain(use, parity);
        if (parity == 0 && lane == 0 && nq > 0) {
            const int last = nq - 1;  // the last Q written (16-bit: loaded by TMA) has landed
            const bool landed = S::QBUFS == 2 ? mbar_wait(&q_full[last & 1], (last >> 1) & 1)
                                              : mbar_wait(&q_full[0], last & 1);
            if (!landed) atomicOr(p.err, kErrTimeout);
        }
    } else if (warp == 1) {
        // --------------------------------------------------------------------- MMA
        uint32_t use = 0;
        int nread = 0;
        // 1: an item, 0: end of work, -1: abort
        auto read_item = [&](TcItem& it) {
            const int slot = nread % kTcQueue;
            bool good = true;
            int ci = -1;
            if (lane == 0) {
                good = tc_wait(&item_full[slot], (nread / kTcQueue) & 1, abort_flag, p.err);
                if (good) {
                    ci = item_q[slot];
                    mbar_arrive(&item_empty[slot]);
                }
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            ci = __shfl_sync(0xffffffffu, ci, 0);
            ++nread;
            if (!good) return -1;
            if (ci < 0) return 0;
            tc_decode_item(ci, p, s_lens, s_prefix, s_order, heads_per_row, it);
            return 1;
        };
        auto mma_s = [&](const TcItem& it, int k) {
            const int b = k & 1;
            bool good = true;
            const int qi = S::QBUFS == 2 ? (k & 1) : 0;  // Q buffer of item k
            if (lane == 0) good = tc_wait(&q_full[qi], S::QBUFS == 2 ? (k >> 1) & 1 : k & 1, abort_flag, p.err);
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) return false;
            tc::fence_after_sync();
            const uint32_t qb = smem_addr(qbuf + qi * S::QBUF);
            for (int t = 0; t < it.n_tiles; ++t) {
                const int s = use % NS;
                if (lane == 0) good = tc_wait(&full[s], (use / NS) & 1, abort_flag, p.err);
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) return false;
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t kb = smem_addr(ring + s * STG);
                    if constexpr (FP8) {
                        // K = 32 codes (32 bytes of the 128-byte row) per MMA
#pragma unroll
                        for (int kk = 0; kk < kTcD / 32; ++kk) {
                            tc::mma_f8(tmem + b * kTcSlotCols + t * kTcN, tc::desc_sw128(kb + kk * 32, 16, 1024),
                                       tc::desc_sw128(qb + kk * 32, 16, 1024), IDESC_S, kk > 0);
                            if constexpr (Q3)  // + K lo^T into columns 0-7 (rows 8-15 of this operand are zero)
                                tc::mma_f8(tmem + b * kTcSlotCols + t * kTcN, tc::desc_sw128(kb + kk * 32, 16, 1024),
                                           tc::desc_sw128(qb + 2048 + kk * 32, 16, 1024), IDESC_S, 1u);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < kTcD / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * kTcHalf + (kk & 3) * 32;
                            // PAIR: dimensions 64-127 read the operand 2 KB in (rows 0-7 zero)
                            const uint32_t qoff = (kk >> 2) * (PAIR ? 2048 : 1024) + (kk & 3) * 32;
                            tc::mma_f16(tmem + b * kTcSlotCols + t * kTcN, tc::desc_sw128(kb + off, 16, 1024),
                                        tc::desc_sw128(qb + qoff, 16, 1024), IDESC_S, kk > 0);
                        }
                    }
                    tc::commit(&empty[s]);
                }
                __syncwarp();
                ++use;
            }
            if (lane == 0) {
                tc::commit(&q_empty[qi]);
                tc::commit(&s_full[b]);
            }
            __syncwarp();
            return true;
        };
        auto mma_o = [&](const TcItem& it, int k) {
            const int b = k & 1;
            bool good = true;
            if (lane == 0) {
                good = S::PBUFS == 2 ? tc_wait(&p_full[b], (k >> 1) & 1, abort_flag, p.err)
                                     : tc_wait(&p_full[0], k & 1, abort_flag, p.err);
                if (good && k >= 2) good = tc_wait(&o_free[b], ((k >> 1) - 1) & 1, abort_flag, p.err);
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) return false;
            tc::fence_after_sync();
            const uint32_t pbase = smem_addr(pbuf + (S::PBUFS == 2 ? b * S::PBUF : 0));
            for (int t = 0; t < it.n_tiles; ++t) {
                const int s = use % NS;
                good = __all_sync(0xffffffffu, tc_wait(&full[s], (use / NS) & 1, abort_flag, p.err));
                if (!good) return false;
                unsigned char* vb = ring + s * STG;
                const int valid = min(kTcTile, it.n_tok - t * kTcTile);
                constexpr int KSTEP = FP8 ? 32 : 16;  // tokens per MMA
                constexpr int CHUNKS = FP8 ? 8 : 16;  // 16-byte chunks per token row
                const int ksteps = (valid + KSTEP - 1) / KSTEP;
                // rows past the context inside the last step: zero them so that
                // never-written pool slots cannot turn P = 0 into NaN
                const int zero_rows = ksteps * KSTEP - valid;
                if (zero_rows > 0) {
                    for (int i = lane; i < zero_rows * CHUNKS; i += 32) {
                        const int r = valid + i / CHUNKS;
                        const int c = i % CHUNKS;  // 16-byte chunk of the row (two halves when 16-bit)
                        *reinterpret_cast<uint4*>(vb + (c >> 3) * kTcHalf + r * 128 + (c & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                }
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t vaddr = smem_addr(vb);
                    for (int j = 0; j < ksteps; ++j) {
                        if constexpr (FP8) {
                            // A = V^T: the 128 codes of a token are one 128-byte row, so
                            // M = 128 is a single swizzle atom; 32 tokens = 4 KB per step
                            // B = P: core matrices of 8 tokens x 16 bytes, 128 B apart
                            tc::mma_f8(tmem + b * kTcSlotCols + kTcMaxTiles * kTcN,
                                       tc::desc_sw128(vaddr + j * 4096, kTcStage8, 1024),
                                       tc::desc_noswizzle(pbase + t * 2048 + j * 512, 128, 2048), IDESC_O,
                                       (t > 0 || j > 0) ? 1u : 0u);
                        } else {
                            const uint32_t poff = (2 * t + (j >> 2)) * (PAIR ? 2048 : 1024) + (j & 3) * 32;
                            tc::mma_f16(tmem + b * kTcSlotCols + kTcMaxTiles * kTcN,
                                        tc::desc_sw128(vaddr + j * 2048, kTcHalf, 1024),
                                        tc::desc_sw128(pbase + poff, 16, 1024), IDESC_O, (t > 0 || j > 0) ? 1u : 0u);
                        }
                    }
                    tc::commit(&empty[s]);
                }
                __syncwarp();
                ++use;
            }
            if (lane == 0) tc::commit(&o_full[b]);
            __syncwarp();
            return true;
        };

        TcItem cur, nxt;
        int rc = read_item(cur);
        bool ok = rc >= 0;
        if (rc > 0) ok = mma_s(cur, 0);
        for (int k = 0; rc > 0 && ok; ++k) {
            const int rn = read_item(nxt);
            if (rn < 0) break;
            if (rn > 0) ok = mma_s(nxt, k + 1);
            if (ok) ok = mma_o(cur, k);
            rc = rn;
            cur = nxt;
        }
        // every MMA this thread issued has completed before tensor memory is freed
        if (lane == 0) {
            tc::commit(final_bar);
            if (!mbar_wait(final_bar, 0)) atomicOr(p.err, kErrTimeout);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------ softmax + epilogue
        const int q4 = warp & 3;         // tensor-memory lane quarter of this warp
        const int row = q4 * 32 + lane;  // token of each tile (S) / dimension d (O)
        const int tid = threadIdx.x - 64;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
        int nread = 0;

        // Every wait below is followed by a barrier that all 128 threads reach;
        // a failure is OR-reduced there so that the four warps leave together
        // and no named barrier is left waiting.
        auto read_item = [&](TcItem& it) {
            const int slot = nread % kTcQueue;
            const bool good =
                __all_sync(0xffffffffu, tc_wait(&item_full[slot], (nread / kTcQueue) & 1, abort_flag, p.err));
            const int ci = good ? item_q[slot] : -1;
            const int qshift = good ? item_shift[slot] : 0;
            ++nread;
            if (named_bar_or(3, 128, !good)) return -1;
            if (tid == 0) mbar_arrive(&item_empty[slot]);
            if (ci < 0) return 0;
            tc_decode_item(ci, p, s_lens, s_prefix, s_order, heads_per_row, it);
            it.qshift = qshift;
            return 1;
        };
        auto softmax = [&](const TcItem& it, int k) {
            const int b = k & 1;
            // one P buffer: item k writes it once the O MMAs of item k-1 have read
            // it.  Two (E4M3): buffer b was last read by the O MMAs of item k-2,
            // whose completion the epilogue of k-2 has already waited for.
            const bool good = __all_sync(
                0xffffffffu, tc_wait(&s_full[b], (k >> 1) & 1, abort_flag, p.err) &&
                                 (k == 0 || S::PBUFS == 2 ||
                                  tc_wait(&o_full[(k - 1) & 1], ((k - 1) >> 1) & 1, abort_flag, p.err)));
            // E4M3: S was computed on the stored codes and on q x 2^-qshift
            const float sl = FP8 ? p.scale_log2 * *p.k_scale * __uint_as_float(static_cast<uint32_t>(127 + it.qshift) << 23)
                                 : p.scale_log2;
            unsigned char* pb = pbuf + (S::PBUFS == 2 ? b * S::PBUF : 0);
            // PAIR: columns 0-7 (kv head 2v) and 8-15 (kv head 2v+1) in two
            // passes over the same scores, each as the single-head case
            constexpr int NH = PAIR ? 2 : 1;
#pragma unroll 1
            for (int hh = 0; hh < NH; ++hh) {
                float sc[kTcMaxTiles][G] = {};
                if (good) {
                    tc::fence_after_sync();
                    if constexpr (FP8) {
                        // column g: the high part of q, column 8 + g: the low part
                        float lo[kTcMaxTiles][G] = {};
#pragma unroll
                        for (int t = 0; t < kTcMaxTiles; ++t)
                            if (t < it.n_tiles) {
                                tc::TmemLd<G>::load(lane_addr + b * kTcSlotCols + t * kTcN, sc[t]);
                                tc::TmemLd<G>::load(lane_addr + b * kTcSlotCols + t * kTcN + 8, lo[t]);
                            }
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int t = 0; t < kTcMaxTiles; ++t)
#pragma unroll
                            for (int g = 0; g < G; ++g) sc[t][g] += lo[t][g];
                    } else {
#pragma unroll
                        for (int t = 0; t < kTcMaxTiles; ++t)
                            if (t < it.n_tiles)
                                tc::TmemLd<G>::load(lane_addr + b * kTcSlotCols + t * kTcN + hh * 8, sc[t]);
                        tc::tmem_wait_ld();
                    }
                    tc::fence_before_sync();  // these reads precede the next MMA into this S buffer
                    float mx[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) mx[g] = -INFINITY;
#pragma unroll
                    for (int t = 0; t < kTcMaxTiles; ++t) {
                        const bool valid = t < it.n_tiles && t * kTcTile + row < it.n_tok;
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            sc[t][g] = valid ? sc[t][g] * sl : -INFINITY;
                            mx[g] = fmaxf(mx[g], sc[t][g]);
                        }
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) mx[g] = warp_max(mx[g]);
                    if (lane == 0) {
#pragma unroll
                        for (int g = 0; g < G; ++g) red_max[q4 * 8 + g] = mx[g];
                    }
                }
                if (named_bar_or(1, 128, !good)) return false;
                float M[G], sum[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    M[g] = fmaxf(fmaxf(red_max[g], red_max[8 + g]), fmaxf(red_max[16 + g], red_max[24 + g]));
                    sum[g] = 0.f;
                }
#pragma unroll
                for (int t = 0; t < kTcMaxTiles; ++t) {
                    if (t < it.n_tiles) {
                        if constexpr (FP8) {
                            // P x 2^8 (at most 256) = hi + lo in E4M3; token `row` of
                            // tile t holds 16 bytes: hi of heads 0-7, then lo of heads 0-7
                            uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                            for (int g = 0; g < G; g += 2) {
                                // M is finite (every item has a token); 2^-inf = 0 for masked rows
                                const float p0 = fast_exp2(sc[t][g] - M[g]);
                                const float p1 = fast_exp2(sc[t][g + 1] - M[g + 1]);
                                sum[g] += p0;
                                sum[g + 1] += p1;
                                uint32_t hi, lo;
                                split_e4m3x2(p0 * 256.f, p1 * 256.f, hi, lo);
                                w[g >> 2] |= hi << (8 * (g & 3));
                                w[2 + (g >> 2)] |= lo << (8 * (g & 3));
                            }
                            *reinterpret_cast<uint4*>(pb + t * 2048 + row * 16) = make_uint4(w[0], w[1], w[2], w[3]);
                        } else {
                            // 8-row regions of (tile, 64-token half), 1 KB apart; PAIR:
                            // 16-row regions, 2 KB apart, rows 8-15 for kv head 2v+1
                            unsigned char* pt = pb + (2 * t + (row >> 6)) * (PAIR ? 2048 : 1024) + hh * 1024;
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                const float pv = fast_exp2(sc[t][g] - M[g]);  // 2^-inf = 0 for masked rows
                                sum[g] += pv;
                                const int chunk = ((row & 63) >> 3) ^ g;
                                *reinterpret_cast<uint16_t*>(pt + g * 128 + chunk * 16 + (row & 7) * 2) =
                                    float_to_act<ACT>(pv);
                            }
                        }
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) sum[g] += __shfl_xor_sync(0xffffffffu, sum[g], off);
                }
                if (lane == 0) {
#pragma unroll
                    for (int g = 0; g < G; ++g) red_sum[q4 * 8 + g] = sum[g];
                }
                if (hh == NH - 1) tc::fence_proxy_async_smem();
                asm volatile("bar.sync 2, 128;" ::: "memory");
                if (tid == 0) {
                    float* st = stats + (b * 2 + hh) * 16;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        st[g] = M[g];
                        st[8 + g] = red_sum[g] + red_sum[8 + g] + red_sum[16 + g] + red_sum[24 + g];
                    }
                    if (hh == NH - 1) mbar_arrive(&p_full[S::PBUFS == 2 ? b : 0]);
                }
            }
            return true;
        };
        auto epilogue = [&](const TcItem& it, int k) {
            const int b = k & 1;
            const bool good = __all_sync(0xffffffffu, tc_wait(&o_full[b], (k >> 1) & 1, abort_flag, p.err));
            float o[G] = {};
            // PAIR: dimensions 64-127 (warps of lane quarters 2 and 3) are kv head
            // 2v+1, whose heads are columns 8-15
            const int hh = PAIR ? (q4 >> 1) : 0;
            if (good) {
                tc::fence_after_sync();
                tc::TmemLd<G>::load(lane_addr + b * kTcSlotCols + kTcMaxTiles * kTcN + hh * 8, o);
                if constexpr (FP8) {
                    float lo[G];  // O of the low parts of P
                    tc::TmemLd<G>::load(lane_addr + b * kTcSlotCols + kTcMaxTiles * kTcN + 8, lo);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int g = 0; g < G; ++g) o[g] += lo[g];
                } else {
                    tc::tmem_wait_ld();
                }
                tc::fence_before_sync();
            }
            // also orders the stats written by the softmax of this item before the reads below
            if (named_bar_or(1, 128, !good)) return false;
            if (tid == 0) mbar_arrive(&o_free[b]);
            const int d = PAIR ? (row & 63) : row;
            const bool single = p.max_parts == 1 || s_lens[it.row] <= p.partition_size;
            // E4M3: O was computed on the stored codes and on P x 2^8
            const float vmul = FP8 ? *p.v_scale * (1.0f / 256.f) : 1.0f;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float Mg = stats[(b * 2 + hh) * 16 + g];
                const float Lg = stats[(b * 2 + hh) * 16 + 8 + g];
                // L >= 1 (the max token's weight is 1): one reciprocal per head
                const float val = o[g] * (__frcp_rn(Lg) * vmul);
                const int kvh = PAIR ? 2 * it.kvh + hh : it.kvh;
                const size_t hrow = static_cast<size_t>(it.seq) * p.num_q_heads + kvh * G + g;
                if (single) {
                    static_cast<uint16_t*>(p.out)[hrow * HD + d] = float_to_act<ACT>(val);
                } else {
                    const size_t slot = hrow * p.max_parts + it.part;
                    p.ws_o[slot * HD + d] = val;
                    if (d == 0) {
                        p.ws_ml[slot * 2] = Mg;
                        p.ws_ml[slot * 2 + 1] = Lg;
                    }
                }
            }
            return true;
        };

        TcItem cur, nxt;
        int rc = read_item(cur);
        bool ok = rc >= 0;
        if (rc > 0) ok = softmax(cur, 0);
        for (int k = 0; rc > 0 && ok; ++k) {
            const int rn = read_item(nxt);
            if (rn < 0) break;
            if (rn > 0) ok = softmax(nxt, k + 1);
            if (ok) ok = epilogue(cur, k);
            rc = rn;
            cur = nxt;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, kTcTmemCols);
}

}  // namespace pkv
