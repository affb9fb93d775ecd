/*
 * pagedkv.h -- C ABI of libpagedkv.so: paged KV-cache decode on GB300 (sm_103a).
 *
 * The KV cache lives in fixed-size physical blocks of a shared pool; each
 * sequence owns a block table mapping its logical blocks to physical ones
 * (Ultralytics glossary "PagedAttention", section "How paging works";
 * OptiVerse "Paged KV cache", section "Block table and non-contiguous
 * allocation").  This library provides the device side of that design --
 * slot-mapped append, the attention kernel that reads K/V block by block
 * through the table, the copy-on-write block copy -- and the host-side block
 * manager that produces the tables and slot mappings.
 *
 * Conventions shared by every device entry point
 *  - Pointers named *_cache, q, k, v, out, block_tables, context_lens,
 *    slot_mapping, src_dst_pairs, workspace, k_scale, v_scale are DEVICE
 *    pointers owned by the caller; the library keeps no reference to them
 *    after the call and never frees them.  All device buffers must be
 *    16-byte aligned.
 *  - Cache layout: k_cache and v_cache are separate row-major arrays
 *    [num_blocks][num_kv_heads][block_size][head_dim] of the cache element
 *    type.  One (block, kv-head) tile is block_size*head_dim contiguous
 *    elements.  Flat slot s means block s / block_size, offset s % block_size.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every device call only enqueues work on that stream and
 *    returns; it is ordered with other work on the same stream.
 *  - Return value: PKV_OK, or an error code below with a message available
 *    from pkv_last_error() (per host thread).  An argument error enqueues
 *    nothing.
 *  - Index errors that can only be seen on the device (a block id outside
 *    the pool, a context length outside 1..max_blocks_per_seq*block_size,
 *    a slot outside the pool) make the kernel skip the offending access and
 *    set a bit in a per-device error word, read with pkv_device_error().
 *
 * Element types: PKV_F16 (IEEE binary16), PKV_BF16 (bfloat16), PKV_E4M3
 * (OCP FP8 E4M3, cache only; per-tensor float32 scales, value = code*scale).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum pkv_dtype { PKV_F16 = 0, PKV_BF16 = 1, PKV_E4M3 = 2 };

enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID = 1,   /* null pointer, unsupported type/head_dim/block_size/group, misalignment */
    PKV_ERR_SHAPE = 2,     /* inconsistent sizes (e.g. num_q_heads not a multiple of num_kv_heads) */
    PKV_ERR_CUDA = 3,      /* a CUDA runtime call or kernel launch failed */
    PKV_ERR_NO_SPACE = 4,  /* block manager: not enough free blocks; state unchanged */
    PKV_ERR_NOT_FOUND = 5  /* block manager: unknown or duplicate sequence id */
};

/* Bits of the per-device error word (pkv_device_error). */
enum pkv_device_error_bits {
    PKV_DEV_BAD_BLOCK = 1,       /* decode: block table entry outside [0, num_blocks) */
    PKV_DEV_BAD_CONTEXT_LEN = 2, /* decode: context length outside 1..max_blocks_per_seq*block_size */
    PKV_DEV_BAD_SLOT = 4,        /* append: slot >= num_blocks*block_size */
    PKV_DEV_BAD_PAIR = 8,        /* block copy: src or dst outside [0, num_blocks) */
    PKV_DEV_WAIT_TIMEOUT = 16    /* a kernel gave up waiting on an on-chip barrier (about 2 s) */
};

/* Partition-size selectors for paged_attention_decode. */
#define PKV_PARTITION_SINGLE 0 /* one pass over the whole context per (sequence, kv head) */
#define PKV_PARTITION_AUTO (-1) /* the library picks the partition size */

/*
 * paged_kv_append -- write each new token's K and V into its slot.
 * Defined by the Ultralytics glossary "PagedAttention", section "How paging
 * works" (position pos of a request goes to block_table[pos // block_size],
 * offset pos % block_size) and OptiVerse "Paged KV cache", section "Block
 * table and non-contiguous allocation" (token 41 of a 41-token request goes
 * to the 10th position of its third block).
 *
 *  k, v          [num_tokens][num_kv_heads][head_dim] of act_dtype (device).
 *  slot_mapping  int64 [num_tokens] (device): flat slot of each token;
 *                a negative slot skips the token (padding).
 *  k_cache, v_cache  the pools, cache_dtype (device, written).
 *  cache_dtype   == act_dtype: bytes are copied unchanged (bit-exact);
 *                PKV_E4M3 with act_dtype F16/BF16: each element x is stored
 *                as e4m3(x / scale) -- binary32 division, round to nearest
 *                even, saturating to +-448 -- with scale = *k_scale for K and
 *                *v_scale for V (device float32 scalars; ignored otherwise).
 *  head_dim      a multiple of 8 (any block_size >= 1).
 * Slots >= num_blocks*block_size are skipped and flag PKV_DEV_BAD_SLOT.
 * Two tokens mapped to the same slot in one call race (one of them wins).
 */
int paged_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                    void* k_cache, void* v_cache, int num_blocks, int num_kv_heads, int block_size,
                    int head_dim, int act_dtype, int cache_dtype, const float* k_scale,
                    const float* v_scale, void* stream);

/*
 * paged_attention_decode -- one decode step of attention over a paged cache.
 * The attention kernel gathers each sequence's keys and values block by
 * block through its block table (Ultralytics glossary "PagedAttention",
 * section "How paging works"; OptiVerse "Paged KV cache", section "Block
 * table and non-contiguous allocation"); query heads share KV heads in
 * groups (Ultralytics glossary, section "Related techniques": grouped-query
 * attention).  For sequence b with L = context_lens[b] tokens and query head
 * h (kv head h / (num_q_heads/num_kv_heads)):
 *     s_j = scale * <q[b][h], K_b[j]>,  p = softmax(s),  out[b][h] = sum_j p_j V_b[j]
 * with K_b[j] = k_cache[block_tables[b][j / block_size]][kvh][j % block_size]
 * (times *k_scale for an E4M3 cache; likewise V).  fp32 online softmax and
 * accumulation; the output is rounded once to act_dtype.
 *
 *  q             [num_seqs][num_q_heads][head_dim] of act_dtype (device).
 *  block_tables  int32 [num_seqs][max_blocks_per_seq] (device); only the
 *                first ceil(L/block_size) entries of a row are read.
 *  context_lens  int32 [num_seqs] (device), each in 1..max_blocks_per_seq*block_size.
 *  out           [num_seqs][num_q_heads][head_dim] of act_dtype (written): device
 *                memory, or pinned host memory the device can address (the
 *                kernels then store the result over the host link within the
 *                same launch; measured slower than device memory plus one
 *                copy for a 0.5 MB result).
 *  act_dtype     PKV_F16 or PKV_BF16; cache_dtype == act_dtype or PKV_E4M3.
 *  head_dim      64 or 128; block_size 16 or 32; group num_q_heads/num_kv_heads
 *                in {1, 2, 4, 8}.
 *  partition_size  PKV_PARTITION_SINGLE (0): one pass per (sequence, kv head);
 *                PKV_PARTITION_AUTO (-1): library choice; > 0: split each
 *                context into partitions of that many tokens (a multiple of
 *                32 and of block_size), attended independently and merged by
 *                their log-sum-exp weights (split-K).
 *  workspace     device scratch of at least pkv_workspace_size(...) bytes
 *                (never less than 256: a work counter that the call zeroes
 *                itself, plus the split-K partials when more than one
 *                partition is possible).  Its contents need no
 *                initialisation and are undefined after the call; calls
 *                sharing a workspace must be ordered (same stream).
 */
int paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int block_size, int head_dim, int num_blocks,
                           float scale, void* out, int act_dtype, int cache_dtype,
                           const float* k_scale, const float* v_scale, int partition_size,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * paged_attention_decode_append -- paged_kv_append of one new token per
 * sequence fused into paged_attention_decode, in one launch: the composition
 * of the append (Ultralytics glossary "PagedAttention", section "How paging
 * works": each new key goes to its slot) and the attention kernel that reads
 * the keys back block by block.
 *  k_new, v_new  [num_seqs][num_kv_heads][head_dim] of act_dtype (device):
 *                the K/V of each sequence's newest token.
 *  slot_mapping  int64 [num_seqs] (device): the slot of that token, which
 *                must be position context_lens[b] - 1 of sequence b (the
 *                slot the block manager returns for it); < 0: sequence b has
 *                no new token this step.
 * Everything else as paged_attention_decode: context_lens count the new
 * token.  Result and cache contents are those of paged_kv_append followed by
 * paged_attention_decode; the new token's row is written by the CTA whose
 * partition ends the context, before that CTA's TMA reads of its block.
 */
int paged_attention_decode_append(const void* q, const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int block_size, int head_dim, int num_blocks,
                                  float scale, void* out, int act_dtype, int cache_dtype,
                                  const float* k_scale, const float* v_scale, int partition_size,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * pkv_workspace_size -- bytes of workspace paged_attention_decode needs for
 * these sizes and partition_size: a 256-byte header (the work counter of the
 * tensor-core kernel's dynamic scheduling) and, when more than one partition
 * is possible, room for each (sequence, query head, partition)'s running
 * max, running sum and normalised partial output in float32.  0 only for
 * invalid arguments.  Host only.
 */
size_t pkv_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int max_blocks_per_seq, int block_size, int partition_size);

/*
 * pkv_resolve_partition_size -- the partition size in tokens that
 * paged_attention_decode uses for these arguments (a value >= the longest
 * possible context means a single pass), or -1 if partition_size is not
 * accepted.  PKV_PARTITION_AUTO gives 512 when num_q_heads/num_kv_heads >= 4
 * and head_dim is 128, or 64 with an even num_kv_heads (the shapes the
 * tensor-core kernel serves; batches of more than 2048 sequences run as
 * several of its launches), or 256 when the number of its work items
 * (num_seqs * num_kv_heads, halved at head_dim 64, * the number of 512-token
 * partitions of the longest possible context) is in [256, 1024); else 1024.
 * Host only.
 */
int pkv_resolve_partition_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int max_blocks_per_seq, int block_size, int partition_size);

/*
 * paged_block_copy -- copy whole physical blocks for copy-on-write.
 * iThome "how to store the KV cache", section "Copy-on-Write": when a
 * sequence writes into a shared, partly filled block, it gets a new block
 * holding a copy of the old contents.  For each pair i, block
 * src_dst_pairs[2i] is copied to block src_dst_pairs[2i+1] in both caches
 * (all kv heads, all slots): block_bytes = num_kv_heads*block_size*head_dim*
 * element size of one cache.  Pairs run concurrently: a block must not be
 * both a destination and a source (or two destinations) in one call.
 *  src_dst_pairs int32 [num_pairs][2] (device).  block_bytes must be a
 *                multiple of 16.  num_pairs == 0 enqueues nothing.
 * Pairs with an id outside [0, num_blocks) are skipped and flag PKV_DEV_BAD_PAIR.
 */
int paged_block_copy(void* k_cache, void* v_cache, const int32_t* src_dst_pairs, int num_pairs,
                     int num_blocks, size_t block_bytes, void* stream);

/* Size of the fixed scratch array behind paged_attention_decode_noalloc. */
#define PKV_NOALLOC_MAX_WORKSPACE_BYTES (16u << 20)

/*
 * paged_attention_decode_noalloc -- paged_attention_decode without a
 * caller-provided workspace, for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a library convenience, not a step of
 * the method.
 *
 * Who needs it: an engine that reserves all free device memory up front for
 * its own pool (a further cudaMalloc would fail or compete with it), a host
 * framework that forbids allocation on its decode path because cudaMalloc can
 * block and synchronise the device, or a plain C caller without a device
 * allocator.  Such callers cannot provide the split-K workspace.
 *
 * Arguments and results are those of paged_attention_decode, minus workspace
 * and workspace_bytes.  The caller still passes every input and output.
 * The split-K scratch is a file-scope device array of
 * PKV_NOALLOC_MAX_WORKSPACE_BYTES (16 MiB); every GPU that loads the library
 * holds it until the process exits.  This call allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.
 *  - Requests whose pkv_workspace_size(...) exceeds the limit are rejected
 *    with PKV_ERR_INVALID and a message naming both sizes (nothing is
 *    enqueued).  Larger partitions, fewer sequences or a shorter table
 *    shrink the need.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it.  Make
 *    that first call before any stream capture.
 *  - With lazy module loading (the CUDA runtime's default since 12.2, unless
 *    CUDA_MODULE_LOADING=EAGER), the array's 16 MiB are committed on a device
 *    when the library's device code holding it is first loaded there, which
 *    may be that first call.  An engine that reserves all free device memory
 *    for its pool should make its first call (any valid decode) before that
 *    reservation; later calls take no device memory.
 *  - The cached address belongs to the device's primary context, which the
 *    CUDA runtime uses.  After cudaDeviceReset, or under another context made
 *    current through the driver API, it is stale: do not call this entry
 *    point there.
 *  - Every call on a device shares the one array, and it keeps the previous
 *    call's contents.  Each call zeroes the work counter it needs (an
 *    asynchronous 4-byte memset on the stream) and writes all the partials
 *    it reads, so no clearing is needed between calls.  Calls that overlap on the GPU (different
 *    streams without ordering, or several host threads) race on the array
 *    and give wrong results; order them on one stream.
 */
int paged_attention_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int block_size, int head_dim, int num_blocks,
                                   float scale, void* out, int act_dtype, int cache_dtype,
                                   const float* k_scale, const float* v_scale, int partition_size,
                                   void* stream);

/* Kernel paths of paged_attention_decode (pkv_set_kernel_path). */
enum pkv_kernel_path {
    PKV_PATH_AUTO = 0,        /* library choice (default) */
    PKV_PATH_CUDA_CORE = 1,   /* CUDA-core kernel for every shape */
    PKV_PATH_TENSOR = 2,      /* tensor-core grouped-query kernel, 5 stages, 1 CTA per SM */
    PKV_PATH_TENSOR_2CTA = 3  /* tensor-core grouped-query kernel, 2 stages, 2 CTAs per SM */
};

/*
 * pkv_set_kernel_path -- choose the decode kernel for later calls in this
 * process (all threads, all devices); returns the previous choice, or -1 for
 * an unknown value.  PKV_PATH_AUTO uses the tensor-core kernel (2 CTAs per
 * SM) when num_q_heads/num_kv_heads >= 4, partitions are at most 512 tokens
 * and either head_dim is 128 with a 16-bit or E4M3 cache, or head_dim is 64
 * with a 16-bit cache, an even num_kv_heads and tables shared by a
 * sequence's kv heads (one item then covers kv heads 2v and 2v+1); the
 * CUDA-core kernel otherwise.
 * Forcing a tensor-core path on a shape it does not serve makes
 * paged_attention_decode return PKV_ERR_INVALID.  Both kernels compute the
 * same function; this is a tuning and testing switch.
 */
int pkv_set_kernel_path(int path);

/* Directions of paged_block_swap. */
enum pkv_swap_direction { PKV_SWAP_OUT = 0, PKV_SWAP_IN = 1 };

/*
 * paged_block_swap -- move whole physical blocks between the pools and a
 * staging buffer, for preemption by swapping (the PagedAttention notes page,
 * section on preemption: swapping moves the KV cache of a sequence that is
 * not running to CPU memory and brings it back when there is room; small
 * blocks make many small transfers).
 *  block_ids  int32 [num_ids] (device): physical blocks, in staging order.
 *  staging    [num_ids][2][block_bytes] bytes: for entry i, the K block then
 *             the V block.  Pinned host memory (cudaHostAlloc, or registered
 *             with cudaHostRegister) or device memory; the kernel reads or
 *             writes it directly, in one launch for the whole list.
 *  direction  PKV_SWAP_OUT: staging[i] = block block_ids[i] of k_cache, v_cache;
 *             PKV_SWAP_IN:  block block_ids[i] = staging[i].
 *  block_bytes one block of one cache (num_kv_heads*block_size*head_dim*elem),
 *             a multiple of 16.  Unregistered pageable host memory is
 *             refused (PKV_ERR_INVALID).  Ids outside [0, num_blocks) are
 *             skipped and flag PKV_DEV_BAD_PAIR.  Swap-in ids must be distinct.
 */
int paged_block_swap(void* k_cache, void* v_cache, const int32_t* block_ids, int num_ids,
                     int num_blocks, size_t block_bytes, void* staging, int direction,
                     void* stream);

/* ------------------------------------------------------------------------
 * QUEST query-aware block selection (Tencent Cloud "LLMs serving
 * challenges", section "Query-sparsity attention / QUEST"): per block the
 * channel-wise minimum and maximum key; for a query the upper bound
 * U = sum_c max(q_c * min_c, q_c * max_c) of q.k over the block's keys;
 * attention reads only the K blocks with the largest bounds.
 * kmeta: [num_blocks][num_kv_heads][2][head_dim] of the queries' 16-bit
 * type (min row, then max row, over the block's filled slots).  With a
 * 16-bit cache that is the cache's type.  With an E4M3 cache (Ultralytics
 * glossary, section "Related techniques": an 8-bit cache) kmeta holds the
 * decoded codes without the per-tensor scale -- every E4M3 value is exact in
 * binary16 and bfloat16 -- so the bounds are the true bounds divided by
 * k_scale (> 0), which ranks the blocks identically.
 * ---------------------------------------------------------------------- */

/* Recompute kmeta (of meta_dtype: PKV_F16 or PKV_BF16; cache_dtype is
 * meta_dtype or PKV_E4M3) for every block the given sequences use (their
 * filled slots).  Shared blocks get the same values from each sharer. */
int quest_block_minmax(const void* k_cache, const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int num_seqs, int num_kv_heads, int block_size,
                       int head_dim, int num_blocks, int cache_dtype, int meta_dtype, void* kmeta,
                       void* stream);

/* Update kmeta (of act_dtype) with newly appended keys k_new
 * [num_tokens][num_kv_heads][head_dim] (act_dtype) at slot_mapping (as given
 * to paged_kv_append): a token at offset 0 of its block starts the block's
 * metadata, later offsets widen it.  An E4M3 cache takes each key as the
 * append stores it, e4m3(x / *k_scale) (k_scale: device float32; ignored
 * for 16-bit caches), and the metadata takes that code's value.  At most one
 * token per block per call (one decode step); slots < 0 are skipped.
 * Copy-on-write copies do not carry metadata: recompute it for the copies. */
int quest_append_minmax(const void* k_new, const int64_t* slot_mapping, int num_tokens,
                        int num_kv_heads, int block_size, int head_dim, int num_blocks, int act_dtype,
                        int cache_dtype, const float* k_scale, void* kmeta, void* stream);

/* Select, per (sequence, kv head), the budget_blocks blocks with the largest
 * bounds (the bound of a kv head is the largest over its query heads; equal
 * bounds prefer the lower logical block), in logical order:
 * sel_tables int32 [num_seqs][num_kv_heads][budget_blocks] (unused entries 0)
 * and sel_lens int32 [num_seqs][num_kv_heads] (their token count; the
 * sequence's last block counts its filled slots).  A sequence with at most
 * budget_blocks blocks keeps them all.  Bounds are computed in float32 by
 * one kernel over every block and kept in `workspace` (device, at least
 * quest_workspace_size bytes, no initialisation needed); a second kernel
 * finds each (sequence, kv head)'s K-th largest bound by radix selection
 * over the bounds' order-preserving 32-bit keys in shared memory.
 * head_dim 64 or 128; group 1, 2, 4 or 8; at most 16384 blocks per sequence. */
int quest_select(const void* q, const void* kmeta, const int32_t* block_tables,
                 int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_q_heads,
                 int num_kv_heads, int block_size, int head_dim, int num_blocks, int act_dtype,
                 int budget_blocks, int32_t* sel_tables, int32_t* sel_lens, void* workspace,
                 size_t workspace_bytes, void* stream);

/* Device workspace quest_select needs: one float32 bound per (sequence, kv
 * head, table entry).  Host only. */
size_t quest_workspace_size(int num_seqs, int num_kv_heads, int max_blocks_per_seq);

/* paged_attention_decode over per-(sequence, kv head) block lists, such as
 * quest_select's: tables [num_seqs][num_kv_heads][max_sel_blocks], lengths
 * [num_seqs][num_kv_heads].  Same kernels as paged_attention_decode (the
 * tensor-core kernel takes at most 2048 (sequence, kv head) rows per launch
 * and larger batches in several launches); the workspace
 * is pkv_workspace_size(..., max_sel_blocks, ...). */
int paged_attention_decode_sparse(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* sel_tables, int max_sel_blocks,
                                  const int32_t* sel_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int block_size, int head_dim, int num_blocks,
                                  float scale, void* out, int act_dtype, int cache_dtype,
                                  const float* k_scale, const float* v_scale, int partition_size,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Message of the last failing call on this host thread ("" if none). */
const char* pkv_last_error(void);

/*
 * pkv_device_error -- read (and, if reset != 0, clear) the per-device error
 * word of the current device: an OR of pkv_device_error_bits set by kernels
 * since the last reset.  Synchronises `stream` first.  Returns PKV_OK or
 * PKV_ERR_CUDA.
 */
int pkv_device_error(int* bits, int reset, void* stream);

/*
 * pkv_selftest_wait_timeout -- check of the kernels' bounded waits.  Launches
 * one CTA that waits, through the same bounded-wait routine the kernels use,
 * on a shared-memory barrier that nothing ever arrives at, with a limit of
 * limit_us microseconds (1 .. 2,000,000) instead of the kernels' 2 s.  The
 * wait gives up, the kernel sets PKV_DEV_WAIT_TIMEOUT in the device error word
 * (read it with pkv_device_error) and returns; the context stays usable.
 * Returns PKV_OK, PKV_ERR_INVALID (limit out of range) or PKV_ERR_CUDA.
 */
int pkv_selftest_wait_timeout(int limit_us, void* stream);

/* Library ABI version (major*100 + minor). */
int pkv_version(void);

/* ------------------------------------------------------------------------
 * Host-side block manager (no GPU work).  A free pool of physical block ids
 * popped first-in first-out, a reference count per block, one block table
 * per sequence, copy-on-write of a shared last block.
 *  - Ultralytics glossary "PagedAttention", section "How paging works": a
 *    request of n tokens takes ceil(n / block_size) blocks; a new block is
 *    taken only when the last one is full.
 *  - OptiVerse "Paged KV cache", section "Block table and non-contiguous
 *    allocation": blocks return to the pool when the request ends.
 *  - iThome "how to store the KV cache", sections "Physical Block sharing"
 *    and "Copy-on-Write": forked sequences share blocks with a reference
 *    count; a writer into a shared, partly filled last block gets a new
 *    block (reported as a (src, dst) copy pair) and the old block's count
 *    drops by one; full shared blocks are never copied.
 * Sequence ids are caller-chosen int64 values.  Not thread-safe: one
 * manager per thread, or external locking.
 * ---------------------------------------------------------------------- */
typedef struct pkv_block_manager pkv_block_manager;

/* Create a manager over num_blocks blocks of block_size tokens.  free_list
 * (host, may be NULL) gives the initial free blocks in pop order; NULL means
 * 0..num_blocks-1.  Returns NULL on invalid arguments. */
pkv_block_manager* pkv_bm_create(int num_blocks, int block_size, const int32_t* free_list,
                                 int free_list_len);
void pkv_bm_destroy(pkv_block_manager* bm);

/* Register a new sequence holding num_tokens tokens (>= 0): allocates
 * ceil(num_tokens/block_size) blocks.  PKV_ERR_NO_SPACE leaves no trace. */
int pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, int num_tokens);

/* Reserve the next token's slot for each of n distinct sequences, in array
 * order.  slots_out (host int64 [n]) gets the flat slots; cow_pairs_out
 * (host int32 [2n]) gets the (src, dst) copies to run with paged_block_copy
 * BEFORE the append, and *num_cow_pairs their count.  All or nothing:
 * PKV_ERR_NO_SPACE if the pool cannot cover the whole batch. */
int pkv_bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, int n, int64_t* slots_out,
                        int32_t* cow_pairs_out, int* num_cow_pairs);

/* Child shares all of parent's blocks (counts + 1) and its length. */
int pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id);

/* Release a sequence: counts - 1; blocks reaching 0 go to the back of the free list. */
int pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id);

/* Write the block tables (host int32 [n][max_blocks_per_seq], unused
 * entries = pad) and context lengths (host int32 [n], may be NULL) of n
 * sequences.  PKV_ERR_SHAPE if a table is longer than max_blocks_per_seq. */
int pkv_bm_get_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int n,
                      int32_t* tables_out, int max_blocks_per_seq, int32_t pad,
                      int32_t* context_lens_out);

/* Prefix caching (the PagedAttention notes page, on automatic prefix
 * caching: a block is looked up by a hash of its own tokens and all tokens
 * before it, so a later turn of a dialogue reuses the KV of the earlier
 * turns; Ultralytics glossary, section "Sharing blocks between
 * sequences": hashing full blocks extends sharing across requests).
 * Register a new sequence from its prompt token ids: every full block is
 * keyed by a chained 64-bit FNV-1a hash of (previous block's key, this
 * block's tokens); the blocks of the longest prefix already registered are
 * shared (counts + 1) and *num_cached_tokens (host) receives the number of
 * leading tokens whose K/V are already in the pool (a multiple of
 * block_size); the remaining blocks are taken from the pool and its full
 * blocks registered.  The caller writes K/V for tokens from
 * *num_cached_tokens on.  A key that already names a block keeps it (the
 * first registration stays); a key match counts only if the block's stored
 * token ids and parent key match too.  A registered block whose count drops
 * to 0 keeps its contents on a least-recently-freed list and is reused for
 * new allocations (and unregistered) only when the free list is empty.
 * The sequence keeps its token ids: pkv_bm_append_tokens registers each
 * block that decoding fills; pkv_bm_append_slots (no ids) stops that for
 * the sequence.  Forks inherit the token ids.  PKV_ERR_NO_SPACE leaves no
 * trace. */
int pkv_bm_add_sequence_cached(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                               int num_tokens, int* num_cached_tokens);

/* pkv_bm_append_slots with the id of each appended token (host int32 [n]):
 * for a sequence added by pkv_bm_add_sequence_cached, a token that fills its
 * block registers that block in the prefix cache under the chained key of
 * the sequence's whole token prefix, exactly as a prompt's full blocks are.
 * Sequences without token ids (pkv_bm_add_sequence) ignore the ids.  Slots,
 * copy-on-write pairs, errors and the all-or-nothing rule are those of
 * pkv_bm_append_slots. */
int pkv_bm_append_tokens(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* token_ids, int n,
                         int64_t* slots_out, int32_t* cow_pairs_out, int* num_cow_pairs);
/* Preemption by swapping (the PagedAttention notes page, section on
 * preemption: the KV of a preempted sequence group moves to CPU memory and
 * comes back when there is room; iThome "how to store the KV cache",
 * section "Physical Block sharing": forked samples share blocks).
 *
 * pkv_bm_swap_out_group swaps out n_seqs sequences together (e.g. the
 * samples of one prompt).  It writes their DISTINCT blocks to blocks_out
 * (host int32, capacity cap) and their count to *n, in first-use order
 * (members in the given order, each table in logical order), so a block the
 * members share is listed -- and staged -- once.  Each member remembers its
 * table as positions in that list and its length; then the members release
 * their blocks (counts - 1, in the same order) and hold none.  Run
 * paged_block_swap(PKV_SWAP_OUT) on the listed blocks before any later call
 * reuses them on the same stream.
 *
 * pkv_bm_swap_in_group brings the group back: seq_ids must be exactly the
 * members swapped out together (any order; members freed since are left
 * out).  It takes one fresh block per listed entry, from the front of the
 * free list in list order, writes them to blocks_out in that order (run
 * paged_block_swap(PKV_SWAP_IN) into them with the same staging), and
 * rebuilds every member's table over them: blocks the members shared are
 * shared again, each with a count equal to the number of members holding
 * it, so copy-on-write continues as before the swap.  An entry that no
 * remaining member holds goes straight back to the free list.
 *
 * pkv_bm_swap_out / pkv_bm_swap_in are the group of one.  A swapped-out
 * sequence cannot append, fork or appear in tables; pkv_bm_free_sequence
 * accepts it.  Unknown, repeated or resident ids give PKV_ERR_NOT_FOUND;
 * PKV_ERR_NO_SPACE and PKV_ERR_SHAPE (cap too small) leave no trace. */
int pkv_bm_swap_out_group(pkv_block_manager* bm, const int64_t* seq_ids, int n_seqs, int32_t* blocks_out,
                          int cap, int* n);
int pkv_bm_swap_in_group(pkv_block_manager* bm, const int64_t* seq_ids, int n_seqs, int32_t* blocks_out,
                         int cap, int* n);
int pkv_bm_swap_out(pkv_block_manager* bm, int64_t seq_id, int32_t* blocks_out, int cap, int* n);
int pkv_bm_swap_in(pkv_block_manager* bm, int64_t seq_id, int32_t* blocks_out, int cap, int* n);

/* Blocks registered in the prefix cache (in use or waiting on the LRU list). */
int pkv_bm_num_cached_blocks(const pkv_block_manager* bm);

/* Blocks available for allocation: the free list plus cached blocks with count 0. */
int pkv_bm_num_free(const pkv_block_manager* bm);
int pkv_bm_ref_count(const pkv_block_manager* bm, int block); /* -1 if out of range */
int pkv_bm_context_len(const pkv_block_manager* bm, int64_t seq_id); /* -1 if unknown */
int pkv_bm_num_seq_blocks(const pkv_block_manager* bm, int64_t seq_id); /* -1 if unknown */
/* Copy the free list, in pop order, into out (capacity cap); returns its length. */
int pkv_bm_free_list(const pkv_block_manager* bm, int32_t* out, int cap);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
