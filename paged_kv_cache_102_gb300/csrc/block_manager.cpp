// Host-side block manager of the paged KV cache (no GPU work).
//
// Free pool: physical block ids, popped from the front, returned to the back
// (Ultralytics glossary "PagedAttention", section "How paging works": free
// blocks are scattered across the pool and taken in list order; OptiVerse
// "Paged KV cache", section "Block table and non-contiguous allocation":
// blocks go back to the pool when the request ends).  Each sequence owns a
// block table and a token count; a block is taken only when the last one is
// full.  Forked sequences share blocks through per-block reference counts;
// a writer into a shared, partly filled last block gets a fresh block and a
// (src, dst) copy pair, and the old block's count drops by one (iThome "how
// to store the KV cache", sections "Physical Block sharing" and
// "Copy-on-Write").  Writers are handled in call order; the last holder of
// a block writes in place.
#include <cstdint>
#include <cstring>
#include <deque>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pagedkv.h"
#include "pkv_error.h"

namespace {

struct Sequence {
    std::vector<int32_t> blocks;
    int64_t len = 0;
};

}  // namespace

struct pkv_block_manager {
    int num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_list;
    std::vector<int32_t> ref;
    std::unordered_map<int64_t, Sequence> seqs;

    int32_t take() {
        int32_t b = free_list.front();
        free_list.pop_front();
        ref[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--ref[b] == 0) free_list.push_back(b);
    }
};

extern "C" {

pkv_block_manager* pkv_bm_create(int num_blocks, int block_size, const int32_t* free_list,
                                 int free_list_len) {
    if (num_blocks <= 0 || block_size <= 0) {
        pkv::set_error("pkv_bm_create: num_blocks and block_size must be positive");
        return nullptr;
    }
    auto* bm = new pkv_block_manager();
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->ref.assign(num_blocks, 0);
    if (free_list == nullptr) {
        for (int i = 0; i < num_blocks; ++i) bm->free_list.push_back(i);
    } else {
        std::vector<char> seen(num_blocks, 0);
        for (int i = 0; i < free_list_len; ++i) {
            int32_t b = free_list[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                pkv::set_error("pkv_bm_create: free list holds an id outside the pool or a duplicate");
                delete bm;
                return nullptr;
            }
            seen[b] = 1;
            bm->free_list.push_back(b);
        }
    }
    return bm;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, int num_tokens) {
    if (!bm || num_tokens < 0) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_add_sequence: bad arguments");
    if (bm->seqs.count(seq_id)) return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_add_sequence: sequence id already in use");
    int64_t need = (static_cast<int64_t>(num_tokens) + bm->block_size - 1) / bm->block_size;
    if (need > static_cast<int64_t>(bm->free_list.size()))
        return pkv::fail(PKV_ERR_NO_SPACE, "pkv_bm_add_sequence: not enough free blocks");
    Sequence s;
    s.len = num_tokens;
    for (int64_t i = 0; i < need; ++i) s.blocks.push_back(bm->take());
    bm->seqs.emplace(seq_id, std::move(s));
    return PKV_OK;
}

int pkv_bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, int n, int64_t* slots_out,
                        int32_t* cow_pairs_out, int* num_cow_pairs) {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots_out || !cow_pairs_out)) || !num_cow_pairs)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_append_slots: bad arguments");
    const int bs = bm->block_size;
    // Pass 1: check ids and count the blocks the whole batch needs, replaying
    // the reference-count decrements that earlier writers in the batch make.
    std::unordered_set<int64_t> seen;
    std::unordered_map<int32_t, int32_t> pending_drop;
    int64_t need = 0;
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() || !seen.insert(seq_ids[i]).second)
            return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_append_slots: unknown or repeated sequence id");
        const Sequence& s = it->second;
        if (s.len % bs == 0) {
            ++need;
        } else {
            int32_t last = s.blocks[s.len / bs];
            if (bm->ref[last] - pending_drop[last] > 1) {
                ++need;
                ++pending_drop[last];
            }
        }
    }
    if (need > static_cast<int64_t>(bm->free_list.size()))
        return pkv::fail(PKV_ERR_NO_SPACE, "pkv_bm_append_slots: not enough free blocks for the batch");
    // Pass 2: apply.
    int pairs = 0;
    for (int i = 0; i < n; ++i) {
        Sequence& s = bm->seqs[seq_ids[i]];
        int64_t pos = s.len;
        int64_t lb = pos / bs;
        if (pos % bs == 0) {
            s.blocks.push_back(bm->take());
        } else {
            int32_t last = s.blocks[lb];
            if (bm->ref[last] > 1) {
                int32_t fresh = bm->take();
                --bm->ref[last];
                s.blocks[lb] = fresh;
                cow_pairs_out[2 * pairs] = last;
                cow_pairs_out[2 * pairs + 1] = fresh;
                ++pairs;
            }
        }
        slots_out[i] = static_cast<int64_t>(s.blocks[lb]) * bs + pos % bs;
        s.len = pos + 1;
    }
    *num_cow_pairs = pairs;
    return PKV_OK;
}

int pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_fork: null manager");
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end() || bm->seqs.count(child_id))
        return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_fork: unknown parent or child id in use");
    Sequence child = it->second;
    for (int32_t b : child.blocks) ++bm->ref[b];
    bm->seqs.emplace(child_id, std::move(child));
    return PKV_OK;
}

int pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_free_sequence: null manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_free_sequence: unknown id");
    for (int32_t b : it->second.blocks) bm->release(b);
    bm->seqs.erase(it);
    return PKV_OK;
}

int pkv_bm_get_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int n, int32_t* tables_out,
                      int max_blocks_per_seq, int32_t pad, int32_t* context_lens_out) {
    if (!bm || n < 0 || max_blocks_per_seq < 0 || (n > 0 && (!seq_ids || (!tables_out && max_blocks_per_seq))))
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_get_tables: bad arguments");
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_get_tables: unknown id");
        const Sequence& s = it->second;
        if (static_cast<int64_t>(s.blocks.size()) > max_blocks_per_seq)
            return pkv::fail(PKV_ERR_SHAPE, "pkv_bm_get_tables: a table is longer than max_blocks_per_seq");
        int32_t* row = tables_out + static_cast<size_t>(i) * max_blocks_per_seq;
        for (int j = 0; j < max_blocks_per_seq; ++j)
            row[j] = j < static_cast<int>(s.blocks.size()) ? s.blocks[j] : pad;
        if (context_lens_out) context_lens_out[i] = static_cast<int32_t>(s.len);
    }
    return PKV_OK;
}

int pkv_bm_num_free(const pkv_block_manager* bm) { return bm ? static_cast<int>(bm->free_list.size()) : -1; }

int pkv_bm_ref_count(const pkv_block_manager* bm, int block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    return bm->ref[block];
}

int pkv_bm_context_len(const pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : static_cast<int>(it->second.len);
}

int pkv_bm_num_seq_blocks(const pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : static_cast<int>(it->second.blocks.size());
}

int pkv_bm_free_list(const pkv_block_manager* bm, int32_t* out, int cap) {
    if (!bm) return -1;
    int n = 0;
    for (int32_t b : bm->free_list) {
        if (n < cap && out) out[n] = b;
        ++n;
    }
    return n;
}

}  // extern "C"
