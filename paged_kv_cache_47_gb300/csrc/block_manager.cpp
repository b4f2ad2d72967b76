// Host block manager of a paged KV cache (include/pkv_block_manager.h).
//
// Bookkeeping only: which physical block backs each logical block of each
// sequence ("PagedAttention — Math + Memory Model", sections "PagedAttention:
// blocks and the block table" and "Copy-on-write: sharing blocks across
// samples"; prefix sharing: "KV-Cache Optimization & PagedAttention for
// Long-Context Agents", "Key KV-Cache Optimization Principles", item 3).
//
// Data structures, sized for a serving loop that touches every live sequence
// each step: the free pool is a vector used as a stack (take = pop_back,
// free = push_back: the most recently freed block is reused first), counts
// are a flat vector, each sequence's table is a vector of block ids, and
// sequences and prefix hashes live in hash maps. Every call first checks that
// it can complete (free blocks, argument sizes) and only then changes state.
#include <stdint.h>

#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv_block_manager.h"
#include "pkv_internal.h"

struct pkv_block_manager {
    struct Seq {
        std::vector<int32_t> table;
        int64_t len = 0;
    };

    int32_t B = 0, NB = 0;
    std::vector<int32_t> free_blocks;   // stack: back() is taken next
    std::vector<int32_t> ref;
    std::vector<uint64_t> hash_of;
    std::vector<uint8_t> has_hash;
    std::unordered_map<int64_t, Seq> seqs;
    std::unordered_map<uint64_t, int32_t> by_hash;
    int64_t tokens = 0;
    std::mutex mu;

    int32_t take() {
        const int32_t b = free_blocks.back();
        free_blocks.pop_back();
        ref[b] = 1;
        return b;
    }

    void drop(int32_t b) {
        if (--ref[b] == 0) {
            free_blocks.push_back(b);
            if (has_hash[b]) {
                by_hash.erase(hash_of[b]);
                has_hash[b] = 0;
            }
        }
    }
};

namespace {

pkv_status bad(pkv_status st, const char *msg) { return pkv::set_last_error(st, "%s", msg); }

}  // namespace

extern "C" {

pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, pkv_block_manager **out) {
    if (!out) return bad(PKV_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (num_blocks < 1 || block_size < 1)
        return bad(PKV_ERR_INVALID_ARG, "num_blocks and block_size must be >= 1");
    pkv_block_manager *bm = new (std::nothrow) pkv_block_manager();
    if (!bm) return bad(PKV_ERR_INVALID_ARG, "out of host memory");
    bm->B = block_size;
    bm->NB = num_blocks;
    bm->free_blocks.resize(num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) bm->free_blocks[i] = num_blocks - 1 - i;
    bm->ref.assign(num_blocks, 0);
    bm->hash_of.assign(num_blocks, 0);
    bm->has_hash.assign(num_blocks, 0);
    *out = bm;
    return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id,
                               const uint64_t *prefix_hashes, int32_t num_prefix_blocks,
                               uint8_t *hits_out) {
    if (!bm) return bad(PKV_ERR_INVALID_ARG, "manager is NULL");
    if (num_prefix_blocks < 0 || (num_prefix_blocks > 0 && !prefix_hashes))
        return bad(PKV_ERR_INVALID_ARG, "bad prefix arguments");
    std::lock_guard<std::mutex> lk(bm->mu);
    if (bm->seqs.count(seq_id)) return bad(PKV_ERR_INVALID_ARG, "sequence already exists");
    int64_t misses = 0;
    for (int32_t i = 0; i < num_prefix_blocks; ++i)
        if (!bm->by_hash.count(prefix_hashes[i])) ++misses;
    if (misses > (int64_t)bm->free_blocks.size())
        return bad(PKV_ERR_NO_BLOCKS, "not enough free blocks for the prefix");
    pkv_block_manager::Seq sq;
    sq.table.reserve(num_prefix_blocks);
    for (int32_t i = 0; i < num_prefix_blocks; ++i) {
        const uint64_t h = prefix_hashes[i];
        auto it = bm->by_hash.find(h);
        int32_t b;
        if (it != bm->by_hash.end()) {
            b = it->second;
            ++bm->ref[b];
            if (hits_out) hits_out[i] = 1;
        } else {
            b = bm->take();
            bm->by_hash.emplace(h, b);
            bm->hash_of[b] = h;
            bm->has_hash[b] = 1;
            if (hits_out) hits_out[i] = 0;
        }
        sq.table.push_back(b);
    }
    sq.len = (int64_t)num_prefix_blocks * bm->B;
    bm->tokens += sq.len;
    bm->seqs.emplace(seq_id, std::move(sq));
    return PKV_OK;
}

namespace {

// pkv_bm_append with the manager's lock held.
pkv_status append_locked(pkv_block_manager *bm, int64_t seq_id, int32_t num_tokens,
                         int64_t *slots_out, int64_t *copy_pairs_out, int32_t max_copies,
                         int32_t *num_copies_out) {
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return bad(PKV_ERR_INVALID_ARG, "unknown sequence");
    pkv_block_manager::Seq &sq = it->second;
    const int64_t B = bm->B;
    int64_t L = sq.len;
    // blocks this call takes: new blocks past the last one, plus one copy
    // when the first write lands in a block others still share
    const int64_t new_blocks = (L + num_tokens + B - 1) / B - (int64_t)sq.table.size();
    const bool cow = num_tokens > 0 && L % B != 0 && bm->ref[sq.table.back()] > 1;
    if (cow && max_copies < 1) return bad(PKV_ERR_INVALID_ARG, "a copy is needed: max_copies is 0");
    if (new_blocks + (cow ? 1 : 0) > (int64_t)bm->free_blocks.size())
        return bad(PKV_ERR_NO_BLOCKS, "not enough free blocks for the append");
    int32_t copies = 0;
    for (int32_t i = 0; i < num_tokens; ++i) {
        if (L % B == 0) {
            sq.table.push_back(bm->take());
        } else if (bm->ref[sq.table.back()] > 1) {
            const int32_t src = sq.table.back();
            const int32_t dst = bm->take();
            copy_pairs_out[2 * copies] = src;
            copy_pairs_out[2 * copies + 1] = dst;
            ++copies;
            bm->drop(src);
            sq.table.back() = dst;
        }
        slots_out[i] = (int64_t)sq.table[L / B] * B + L % B;
        ++L;
    }
    bm->tokens += L - sq.len;
    sq.len = L;
    if (num_copies_out) *num_copies_out = copies;
    return PKV_OK;
}

}  // namespace

pkv_status pkv_bm_append(pkv_block_manager *bm, int64_t seq_id, int32_t num_tokens,
                         int64_t *slots_out, int64_t *copy_pairs_out, int32_t max_copies,
                         int32_t *num_copies_out) {
    if (!bm) return bad(PKV_ERR_INVALID_ARG, "manager is NULL");
    if (num_tokens < 0 || (num_tokens > 0 && !slots_out) || max_copies < 0 ||
        (max_copies > 0 && !copy_pairs_out))
        return bad(PKV_ERR_INVALID_ARG, "bad append arguments");
    std::lock_guard<std::mutex> lk(bm->mu);
    return append_locked(bm, seq_id, num_tokens, slots_out, copy_pairs_out, max_copies,
                         num_copies_out);
}

pkv_status pkv_bm_append_batch(pkv_block_manager *bm, const int64_t *seq_ids,
                               const int32_t *num_tokens, int32_t num_seqs, int64_t *slots_out,
                               int64_t *copy_pairs_out, int32_t max_copies,
                               int32_t *num_copies_out, int32_t *num_done_out) {
    if (!bm) return bad(PKV_ERR_INVALID_ARG, "manager is NULL");
    if (num_seqs < 0 || (num_seqs > 0 && (!seq_ids || !num_tokens)) || max_copies < 0 ||
        (max_copies > 0 && !copy_pairs_out))
        return bad(PKV_ERR_INVALID_ARG, "bad batch arguments");
    std::lock_guard<std::mutex> lk(bm->mu);
    int64_t nslot = 0;
    int32_t ncopy = 0, done = 0;
    pkv_status st = PKV_OK;
    for (; done < num_seqs; ++done) {
        const int32_t n = num_tokens[done];
        if (n < 0 || (n > 0 && !slots_out)) {
            st = bad(PKV_ERR_INVALID_ARG, "bad token count");
            break;
        }
        int32_t c = 0;
        st = append_locked(bm, seq_ids[done], n, slots_out ? slots_out + nslot : nullptr,
                           copy_pairs_out ? copy_pairs_out + 2 * ncopy : nullptr,
                           max_copies - ncopy, &c);
        if (st != PKV_OK) break;
        nslot += n;
        ncopy += c;
    }
    if (num_copies_out) *num_copies_out = ncopy;
    if (num_done_out) *num_done_out = done;
    return st;
}

pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent_id, int64_t child_id) {
    if (!bm) return bad(PKV_ERR_INVALID_ARG, "manager is NULL");
    std::lock_guard<std::mutex> lk(bm->mu);
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end()) return bad(PKV_ERR_INVALID_ARG, "unknown parent sequence");
    if (bm->seqs.count(child_id)) return bad(PKV_ERR_INVALID_ARG, "child sequence already exists");
    pkv_block_manager::Seq child = it->second;
    for (int32_t b : child.table) ++bm->ref[b];
    bm->tokens += child.len;
    bm->seqs.emplace(child_id, std::move(child));
    return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id) {
    if (!bm) return bad(PKV_ERR_INVALID_ARG, "manager is NULL");
    std::lock_guard<std::mutex> lk(bm->mu);
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return bad(PKV_ERR_INVALID_ARG, "unknown sequence");
    for (int32_t b : it->second.table) bm->drop(b);
    bm->tokens -= it->second.len;
    bm->seqs.erase(it);
    return PKV_OK;
}

pkv_status pkv_bm_block_tables(pkv_block_manager *bm, const int64_t *seq_ids, int32_t num_seqs,
                               int32_t max_blocks_per_seq, int32_t *block_tables_out,
                               int32_t *context_lens_out) {
    if (!bm) return bad(PKV_ERR_INVALID_ARG, "manager is NULL");
    if (num_seqs < 0 || max_blocks_per_seq < 1 ||
        (num_seqs > 0 && (!seq_ids || !block_tables_out || !context_lens_out)))
        return bad(PKV_ERR_INVALID_ARG, "bad table arguments");
    std::lock_guard<std::mutex> lk(bm->mu);
    for (int32_t s = 0; s < num_seqs; ++s) {
        auto it = bm->seqs.find(seq_ids[s]);
        if (it == bm->seqs.end()) return bad(PKV_ERR_INVALID_ARG, "unknown sequence");
        if ((int64_t)it->second.table.size() > max_blocks_per_seq || it->second.len > INT32_MAX)
            return bad(PKV_ERR_INVALID_ARG, "a sequence has more blocks than the table width");
    }
    for (int32_t s = 0; s < num_seqs; ++s) {
        const pkv_block_manager::Seq &sq = bm->seqs.find(seq_ids[s])->second;
        int32_t *row = block_tables_out + (size_t)s * max_blocks_per_seq;
        const int32_t n = (int32_t)sq.table.size();
        for (int32_t j = 0; j < n; ++j) row[j] = sq.table[j];
        for (int32_t j = n; j < max_blocks_per_seq; ++j) row[j] = -1;
        context_lens_out[s] = (int32_t)sq.len;
    }
    return PKV_OK;
}

pkv_status pkv_bm_stats_get(pkv_block_manager *bm, pkv_bm_stats *out) {
    if (!bm || !out) return bad(PKV_ERR_INVALID_ARG, "NULL argument");
    std::lock_guard<std::mutex> lk(bm->mu);
    out->num_blocks = bm->NB;
    out->free_blocks = (int32_t)bm->free_blocks.size();
    int32_t shared = 0;
    for (int32_t r : bm->ref) shared += r > 1;
    out->shared_blocks = shared;
    out->prefix_entries = (int32_t)bm->by_hash.size();
    out->sequences = (int64_t)bm->seqs.size();
    out->tokens = bm->tokens;
    return PKV_OK;
}

int32_t pkv_bm_refcount(pkv_block_manager *bm, int32_t block) {
    if (!bm) return -1;
    std::lock_guard<std::mutex> lk(bm->mu);
    if (block < 0 || block >= bm->NB) return -1;
    return bm->ref[block];
}

pkv_status pkv_bm_simulate_admission(int32_t num_blocks, int32_t block_size,
                                     const int32_t *context_lens, int32_t n,
                                     int32_t reserve_tokens, int32_t *admitted_out,
                                     double *utilisation_out) {
    if (!admitted_out || !utilisation_out || n < 0 || (n > 0 && !context_lens) ||
        reserve_tokens < 0)
        return bad(PKV_ERR_INVALID_ARG, "bad simulation arguments");
    for (int32_t i = 0; i < n; ++i)
        if (context_lens[i] < 0 || (reserve_tokens > 0 && context_lens[i] > reserve_tokens))
            return bad(PKV_ERR_INVALID_ARG, "a request does not fit its reservation");
    pkv_block_manager *bm = nullptr;
    pkv_status st = pkv_bm_create(num_blocks, block_size, &bm);
    if (st != PKV_OK) return st;
    int64_t live = 0;
    int32_t admitted = 0;
    std::vector<int64_t> slots;
    for (int32_t i = 0; i < n; ++i) {
        // a request holds the blocks of its reservation, or of its length
        const int32_t held = reserve_tokens > 0 ? reserve_tokens : context_lens[i];
        slots.resize(held > 0 ? held : 1);
        if ((st = pkv_bm_add_sequence(bm, i, nullptr, 0, nullptr)) != PKV_OK) break;
        int32_t ncopy = 0;
        st = pkv_bm_append(bm, i, held, slots.data(), nullptr, 0, &ncopy);
        if (st == PKV_ERR_NO_BLOCKS) {
            st = PKV_OK;
            break;
        }
        if (st != PKV_OK) break;
        live += context_lens[i];
        ++admitted;
    }
    if (st == PKV_OK) {
        const int64_t used = (int64_t)(num_blocks - (int32_t)bm->free_blocks.size());
        *admitted_out = admitted;
        *utilisation_out = used > 0 ? (double)live / ((double)used * block_size) : 0.0;
    }
    pkv_bm_destroy(bm);
    return st;
}

}  // extern "C"
