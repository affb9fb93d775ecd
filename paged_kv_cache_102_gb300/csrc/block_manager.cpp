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
//
// Prefix caching (PagedAttention notes, section on Automatic Prefix Caching:
// a KV block is looked up by a hash of its own tokens and all tokens before
// it; equal hashes mean equal blocks; Ultralytics glossary "PagedAttention",
// section "Sharing blocks between sequences": hashing full blocks extends
// sharing across requests).  pkv_bm_add_sequence_cached keys every full
// block of a prompt by a chained 64-bit FNV-1a hash over (previous block's
// hash, this block's token ids), reuses the blocks already registered for
// the longest matching prefix, and registers the new full blocks.  Such a
// sequence keeps the chain hash and the token ids of its partial last block;
// pkv_bm_append_tokens appends with token ids, and a block that becomes full
// is registered the same way, so a later turn of a dialogue finds the
// blocks of the earlier turns' answers as well as their prompts.  A key
// that already names a block keeps it (the first registration stays).  A
// match is confirmed by the block's own token ids and its parent's hash,
// stored at registration.  A freed block that is registered keeps its
// contents and waits on an LRU list; it is taken (and unregistered) only
// when the free list is empty.
#include <cstdint>
#include <cstring>
#include <deque>
#include <list>
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
    bool swapped = false;  // contents staged outside the pool; no blocks held
    int64_t swap_group = -1;          // the group it was swapped out with
    std::vector<int32_t> staged_idx;  // while swapped: its table as positions in the group's staged list
    // prefix caching: set for sequences added from their token ids, cleared by
    // an append without token ids
    bool tracked = false;
    uint64_t chain = 0;         // hash of the last full block (0: none yet)
    std::vector<int32_t> tail;  // token ids of the partly filled last block
};

}  // namespace

namespace {

// FNV-1a, 64-bit: offset basis 14695981039346656037, prime 1099511628211.
constexpr uint64_t kFnvBasis = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

uint64_t fnv1a_bytes(uint64_t h, const void* data, size_t n) {
    const unsigned char* p = static_cast<const unsigned char*>(data);
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= kFnvPrime;
    }
    return h;
}

// Hash of a full block: chained over the previous block's hash and this block's tokens.
uint64_t block_hash(uint64_t parent, const int32_t* tokens, int n) {
    uint64_t h = fnv1a_bytes(kFnvBasis, &parent, sizeof(parent));
    for (int i = 0; i < n; ++i) {
        const uint32_t t = static_cast<uint32_t>(tokens[i]);
        const unsigned char b[4] = {static_cast<unsigned char>(t), static_cast<unsigned char>(t >> 8),
                                    static_cast<unsigned char>(t >> 16), static_cast<unsigned char>(t >> 24)};
        h = fnv1a_bytes(h, b, 4);
    }
    return h;
}

}  // namespace

namespace {

// Sequences swapped out together: their distinct blocks were staged once.
struct SwapGroup {
    std::unordered_set<int64_t> members;
    int n_staged = 0;
};

}  // namespace

struct pkv_block_manager {
    int num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_list;
    std::vector<int32_t> ref;
    std::unordered_map<int64_t, Sequence> seqs;
    std::unordered_map<int64_t, SwapGroup> swap_groups;
    int64_t next_swap_group = 0;
    // prefix cache
    std::unordered_map<uint64_t, int32_t> cached;  // hash -> block
    std::vector<uint64_t> hash_of;                 // per block, valid when registered[b]
    std::vector<uint64_t> parent_of;               // hash of the previous block (0: first block)
    std::vector<int32_t> tokens_of;                // [num_blocks][block_size] token ids of registered blocks
    std::vector<char> registered;
    std::list<int32_t> evictable;  // registered blocks with count 0, least recently freed first
    std::vector<std::list<int32_t>::iterator> evict_pos;

    int available() const { return static_cast<int>(free_list.size() + evictable.size()); }

    void unregister(int32_t b) {
        if (registered[b]) {
            cached.erase(hash_of[b]);
            registered[b] = 0;
        }
    }
    int32_t take() {
        int32_t b;
        if (!free_list.empty()) {
            b = free_list.front();
            free_list.pop_front();
        } else {
            b = evictable.front();
            evictable.pop_front();
            unregister(b);
        }
        ref[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--ref[b] == 0) {
            if (registered[b]) {
                evictable.push_back(b);
                evict_pos[b] = std::prev(evictable.end());
            } else {
                free_list.push_back(b);
            }
        }
    }
    // Register full block b under `hash` unless the key already names a block.
    void register_block(int32_t b, uint64_t hash, uint64_t parent, const int32_t* toks) {
        if (cached.count(hash)) return;
        if (tokens_of.empty()) tokens_of.assign(static_cast<size_t>(num_blocks) * block_size, 0);
        hash_of[b] = hash;
        parent_of[b] = parent;
        std::memcpy(&tokens_of[static_cast<size_t>(b) * block_size], toks, sizeof(int32_t) * block_size);
        registered[b] = 1;
        cached[hash] = b;
    }
    // The registered block for (hash, parent, toks), or -1.
    int32_t lookup(uint64_t hash, uint64_t parent, const int32_t* toks) const {
        auto it = cached.find(hash);
        if (it == cached.end()) return -1;
        const int32_t b = it->second;
        if (parent_of[b] != parent ||
            std::memcmp(&tokens_of[static_cast<size_t>(b) * block_size], toks, sizeof(int32_t) * block_size) != 0)
            return -1;
        return b;
    }
    // A registered block is referenced again.
    void revive(int32_t b) {
        if (ref[b] == 0) evictable.erase(evict_pos[b]);
        ++ref[b];
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
    bm->hash_of.assign(num_blocks, 0);
    bm->parent_of.assign(num_blocks, 0);
    bm->registered.assign(num_blocks, 0);
    bm->evict_pos.resize(num_blocks);
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
    if (need > bm->available())
        return pkv::fail(PKV_ERR_NO_SPACE, "pkv_bm_add_sequence: not enough free blocks");
    Sequence s;
    s.len = num_tokens;
    for (int64_t i = 0; i < need; ++i) s.blocks.push_back(bm->take());
    bm->seqs.emplace(seq_id, std::move(s));
    return PKV_OK;
}

}  // extern "C"

namespace {

// Shared body of pkv_bm_append_slots (token_ids == nullptr) and pkv_bm_append_tokens.
int append_batch(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* token_ids, int n,
                 int64_t* slots_out, int32_t* cow_pairs_out, int* num_cow_pairs, const char* F) {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots_out || !cow_pairs_out)) || !num_cow_pairs)
        return pkv::fail(PKV_ERR_INVALID, std::string(F) + ": bad arguments");
    const int bs = bm->block_size;
    // Pass 1: check ids and count the blocks the whole batch needs, replaying
    // the reference-count decrements that earlier writers in the batch make.
    std::unordered_set<int64_t> seen;
    std::unordered_map<int32_t, int32_t> pending_drop;
    int64_t need = 0;
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() || !seen.insert(seq_ids[i]).second || it->second.swapped)
            return pkv::fail(PKV_ERR_NOT_FOUND, std::string(F) + ": unknown, repeated or swapped-out sequence id");
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
    if (need > bm->available())
        return pkv::fail(PKV_ERR_NO_SPACE, std::string(F) + ": not enough free blocks for the batch");
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
        if (!token_ids) {
            s.tracked = false;  // this token's id is unknown: stop registering
            s.tail.clear();
        } else if (s.tracked) {
            s.tail.push_back(token_ids[i]);
            if (s.len % bs == 0) {  // the token filled its block
                const uint64_t h = block_hash(s.chain, s.tail.data(), bs);
                bm->register_block(s.blocks[lb], h, s.chain, s.tail.data());
                s.chain = h;
                s.tail.clear();
            }
        }
    }
    *num_cow_pairs = pairs;
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, int n, int64_t* slots_out,
                        int32_t* cow_pairs_out, int* num_cow_pairs) {
    return append_batch(bm, seq_ids, nullptr, n, slots_out, cow_pairs_out, num_cow_pairs, "pkv_bm_append_slots");
}

int pkv_bm_append_tokens(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* token_ids, int n,
                         int64_t* slots_out, int32_t* cow_pairs_out, int* num_cow_pairs) {
    if (n > 0 && !token_ids) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_append_tokens: token_ids is null");
    return append_batch(bm, seq_ids, token_ids, n, slots_out, cow_pairs_out, num_cow_pairs, "pkv_bm_append_tokens");
}

int pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_fork: null manager");
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end() || bm->seqs.count(child_id) || it->second.swapped)
        return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_fork: unknown or swapped-out parent, or child id in use");
    Sequence child = it->second;
    for (int32_t b : child.blocks) ++bm->ref[b];
    bm->seqs.emplace(child_id, std::move(child));
    return PKV_OK;
}

int pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_free_sequence: null manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_free_sequence: unknown id");
    for (int32_t b : it->second.blocks) bm->release(b);  // a swapped-out sequence holds none
    if (it->second.swapped) {
        auto g = bm->swap_groups.find(it->second.swap_group);
        if (g != bm->swap_groups.end()) {
            g->second.members.erase(seq_id);
            if (g->second.members.empty()) bm->swap_groups.erase(g);
        }
    }
    bm->seqs.erase(it);
    return PKV_OK;
}

int pkv_bm_get_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int n, int32_t* tables_out,
                      int max_blocks_per_seq, int32_t pad, int32_t* context_lens_out) {
    if (!bm || n < 0 || max_blocks_per_seq < 0 || (n > 0 && (!seq_ids || (!tables_out && max_blocks_per_seq))))
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_get_tables: bad arguments");
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() || it->second.swapped)
            return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_get_tables: unknown or swapped-out id");
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

int pkv_bm_add_sequence_cached(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens, int num_tokens,
                               int* num_cached_tokens) {
    if (!bm || num_tokens < 0 || (num_tokens > 0 && !tokens) || !num_cached_tokens)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_add_sequence_cached: bad arguments");
    if (bm->seqs.count(seq_id))
        return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_add_sequence_cached: sequence id already in use");
    const int bs = bm->block_size;
    const int n_full = num_tokens / bs;
    const int n_blocks = (num_tokens + bs - 1) / bs;
    // longest registered prefix of full blocks
    std::vector<uint64_t> hashes(n_full);
    uint64_t h = 0;
    for (int i = 0; i < n_full; ++i) {
        h = block_hash(h, tokens + static_cast<size_t>(i) * bs, bs);
        hashes[i] = h;
    }
    std::vector<int32_t> hit;
    int revived_from_lru = 0;
    while (static_cast<int>(hit.size()) < n_full) {
        const int i = static_cast<int>(hit.size());
        const int32_t b = bm->lookup(hashes[i], i ? hashes[i - 1] : 0, tokens + static_cast<size_t>(i) * bs);
        if (b < 0) break;
        if (bm->ref[b] == 0) ++revived_from_lru;
        hit.push_back(b);
    }
    const int reused = static_cast<int>(hit.size());
    const int fresh = n_blocks - reused;
    if (fresh > bm->available() - revived_from_lru)
        return pkv::fail(PKV_ERR_NO_SPACE, "pkv_bm_add_sequence_cached: not enough free blocks");
    Sequence s;
    s.len = num_tokens;
    for (int32_t b : hit) {
        bm->revive(b);
        s.blocks.push_back(b);
    }
    for (int i = reused; i < n_blocks; ++i) {
        const int32_t b = bm->take();
        if (i < n_full) bm->register_block(b, hashes[i], i ? hashes[i - 1] : 0, tokens + static_cast<size_t>(i) * bs);
        s.blocks.push_back(b);
    }
    s.tracked = true;
    s.chain = n_full ? hashes[n_full - 1] : 0;
    s.tail.assign(tokens + static_cast<size_t>(n_full) * bs, tokens + num_tokens);
    bm->seqs.emplace(seq_id, std::move(s));
    *num_cached_tokens = reused * bs;
    return PKV_OK;
}

int pkv_bm_swap_out_group(pkv_block_manager* bm, const int64_t* seq_ids, int n_seqs, int32_t* blocks_out, int cap,
                          int* n) {
    if (!bm || !n || cap < 0 || n_seqs < 1 || !seq_ids)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_swap_out_group: bad arguments");
    // distinct blocks in first-use order: members in call order, tables in logical order
    std::unordered_set<int64_t> seen;
    std::unordered_map<int32_t, int32_t> pos;
    std::vector<int32_t> staged;
    for (int i = 0; i < n_seqs; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() || it->second.swapped || !seen.insert(seq_ids[i]).second)
            return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_swap_out_group: unknown, repeated or swapped-out id");
        for (int32_t b : it->second.blocks)
            if (pos.emplace(b, static_cast<int32_t>(staged.size())).second) staged.push_back(b);
    }
    const int ns = static_cast<int>(staged.size());
    if (ns > cap || (ns > 0 && !blocks_out)) return pkv::fail(PKV_ERR_SHAPE, "pkv_bm_swap_out_group: output too small");
    const int64_t gid = bm->next_swap_group++;
    SwapGroup& g = bm->swap_groups[gid];
    g.n_staged = ns;
    for (int i = 0; i < ns; ++i) blocks_out[i] = staged[i];
    for (int i = 0; i < n_seqs; ++i) {
        Sequence& s = bm->seqs[seq_ids[i]];
        s.staged_idx.clear();
        for (int32_t b : s.blocks) {
            s.staged_idx.push_back(pos[b]);
            bm->release(b);
        }
        s.blocks.clear();
        s.swapped = true;
        s.swap_group = gid;
        g.members.insert(seq_ids[i]);
    }
    *n = ns;
    return PKV_OK;
}

int pkv_bm_swap_in_group(pkv_block_manager* bm, const int64_t* seq_ids, int n_seqs, int32_t* blocks_out, int cap,
                         int* n) {
    if (!bm || !n || cap < 0 || n_seqs < 1 || !seq_ids)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_swap_in_group: bad arguments");
    auto first = bm->seqs.find(seq_ids[0]);
    if (first == bm->seqs.end() || !first->second.swapped)
        return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_swap_in_group: unknown or resident id");
    auto git = bm->swap_groups.find(first->second.swap_group);
    if (git == bm->swap_groups.end()) return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_swap_in_group: unknown group");
    SwapGroup& g = git->second;
    std::unordered_set<int64_t> given(seq_ids, seq_ids + n_seqs);
    if (static_cast<int>(given.size()) != n_seqs || given != g.members)
        return pkv::fail(PKV_ERR_NOT_FOUND,
                         "pkv_bm_swap_in_group: the ids must be exactly the sequences swapped out together "
                         "(minus any freed since)");
    const int ns = g.n_staged;
    if (ns > cap || (ns > 0 && !blocks_out)) return pkv::fail(PKV_ERR_SHAPE, "pkv_bm_swap_in_group: output too small");
    if (ns > bm->available()) return pkv::fail(PKV_ERR_NO_SPACE, "pkv_bm_swap_in_group: not enough free blocks");
    std::vector<int32_t> held(ns, 0);
    for (int i = 0; i < n_seqs; ++i)
        for (int32_t k : bm->seqs[seq_ids[i]].staged_idx) ++held[k];
    for (int k = 0; k < ns; ++k) {
        const int32_t b = bm->take();
        blocks_out[k] = b;
        bm->ref[b] = held[k];
        if (held[k] == 0) bm->free_list.push_back(b);  // no member holds this entry any more
    }
    for (int i = 0; i < n_seqs; ++i) {
        Sequence& s = bm->seqs[seq_ids[i]];
        s.blocks.clear();
        for (int32_t k : s.staged_idx) s.blocks.push_back(blocks_out[k]);
        s.staged_idx.clear();
        s.swapped = false;
        s.swap_group = -1;
    }
    bm->swap_groups.erase(git);
    *n = ns;
    return PKV_OK;
}

int pkv_bm_swap_out(pkv_block_manager* bm, int64_t seq_id, int32_t* blocks_out, int cap, int* n) {
    return pkv_bm_swap_out_group(bm, &seq_id, 1, blocks_out, cap, n);
}

int pkv_bm_swap_in(pkv_block_manager* bm, int64_t seq_id, int32_t* blocks_out, int cap, int* n) {
    return pkv_bm_swap_in_group(bm, &seq_id, 1, blocks_out, cap, n);
}

int pkv_bm_num_cached_blocks(const pkv_block_manager* bm) { return bm ? static_cast<int>(bm->cached.size()) : -1; }

int pkv_bm_num_free(const pkv_block_manager* bm) { return bm ? bm->available() : -1; }

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
