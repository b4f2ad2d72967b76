/*
 * libpkv block manager — host bookkeeping of a paged KV cache.
 *
 * The manager decides which physical block backs each logical block of each
 * sequence; the device calls of pkv.h then move the bytes (pkv_append writes
 * at the slots it hands out, pkv_block_copy runs the copies it asks for,
 * pkv_decode_attention reads the tables it fills). Everything here runs on
 * the host and touches no device memory.
 *
 * Passages:
 *  - blocks of B tokens in one pool; a per-sequence block table maps logical
 *    block i (tokens i*B .. i*B+B-1) to a physical block; a sequence takes a
 *    free block when it fills its last one ("PagedAttention — Math + Memory
 *    Model", section "PagedAttention: blocks and the block table");
 *  - sharing by reference with a per-block count; copy-on-write of the one
 *    block a writer hits while others still share it; a block returns to the
 *    free pool when its count reaches zero; samples and beams fork from one
 *    prompt (same page, section "Copy-on-write: sharing blocks across
 *    samples");
 *  - identical prompt prefixes share their blocks across requests
 *    ("KV-Cache Optimization & PagedAttention for Long-Context Agents",
 *    section "Key KV-Cache Optimization Principles", item 3).
 *
 * Policies the pages leave open, fixed here:
 *  - the most recently freed block is taken first; a new manager hands out
 *    blocks 0, 1, 2, ...; a sequence's blocks are freed in table order;
 *  - a full prompt block is identified by a caller-given 64-bit hash of its
 *    prefix; the entry lives while the block is allocated;
 *  - a call that needs more free blocks than there are returns
 *    PKV_ERR_NO_BLOCKS and changes nothing.
 *
 * Thread safety: calls on one manager are serialised by an internal lock.
 * Ownership: the manager owns its memory; pointers passed in are read or
 * written during the call only.
 */
#ifndef PKV_BLOCK_MANAGER_H
#define PKV_BLOCK_MANAGER_H

#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

typedef struct {
    int32_t num_blocks;     /* pool size                                      */
    int32_t free_blocks;    /* blocks with count 0                            */
    int32_t shared_blocks;  /* blocks with count > 1                          */
    int32_t prefix_entries; /* registered prefix hashes                       */
    int64_t sequences;      /* live sequences                                 */
    int64_t tokens;         /* sum of the live sequences' lengths             */
} pkv_bm_stats;

/* New manager over num_blocks blocks of block_size tokens (both >= 1). */
pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, pkv_block_manager **out);

/* Free the manager (NULL is a no-op). */
void pkv_bm_destroy(pkv_block_manager *bm);

/*
 * Add sequence seq_id (which must not exist) whose first num_prefix_blocks
 * blocks are full prompt blocks identified by prefix_hashes[i]. A hash that
 * is registered shares its block (count + 1); any other takes a free block
 * and registers the hash. hits_out (may be NULL) receives 1 per shared block
 * and 0 per new block: the caller must write K/V for the new ones. The
 * sequence's length becomes num_prefix_blocks * block_size.
 */
pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id,
                               const uint64_t *prefix_hashes, int32_t num_prefix_blocks,
                               uint8_t *hits_out);

/*
 * Make room for num_tokens new tokens at the end of seq_id. slots_out
 * [num_tokens] receives slot = block * block_size + offset for each token.
 * copy_pairs_out [max_copies][2] receives the (src, dst) block copies that
 * must run (pkv_block_copy) before the tokens are written; *num_copies_out
 * their number (at most 1 per call). max_copies may be 0 only when no copy
 * can occur; otherwise a needed copy that does not fit is PKV_ERR_INVALID_ARG
 * and nothing changes.
 */
pkv_status pkv_bm_append(pkv_block_manager *bm, int64_t seq_id, int32_t num_tokens,
                         int64_t *slots_out, int64_t *copy_pairs_out, int32_t max_copies,
                         int32_t *num_copies_out);

/*
 * One decode step for a batch: pkv_bm_append(seq_ids[i], num_tokens[i]) for
 * i = 0 .. num_seqs-1 in order, in one call. slots_out receives the slots of
 * all sequences back to back (sum of num_tokens entries); copy_pairs_out
 * [max_copies][2] the copies of all of them, in order. On failure at
 * sequence i (PKV_ERR_NO_BLOCKS, or PKV_ERR_INVALID_ARG for an unknown
 * sequence or too little room for copies) sequences 0 .. i-1 keep their
 * changes, sequence i and later are untouched, and *num_done_out = i.
 */
pkv_status pkv_bm_append_batch(pkv_block_manager *bm, const int64_t *seq_ids,
                               const int32_t *num_tokens, int32_t num_seqs, int64_t *slots_out,
                               int64_t *copy_pairs_out, int32_t max_copies,
                               int32_t *num_copies_out, int32_t *num_done_out);

/* Child child_id (new) shares every block of parent_id (counts + 1). */
pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent_id, int64_t child_id);

/* Drop seq_id: every count - 1; blocks at 0 return to the pool. */
pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id);

/*
 * Decode inputs for a batch: block_tables_out [num_seqs][max_blocks_per_seq]
 * int32 (padded with -1) and context_lens_out [num_seqs] int32, in the
 * layouts of pkv_decode_attention. A sequence with more blocks than
 * max_blocks_per_seq is PKV_ERR_INVALID_ARG.
 */
pkv_status pkv_bm_block_tables(pkv_block_manager *bm, const int64_t *seq_ids, int32_t num_seqs,
                               int32_t max_blocks_per_seq, int32_t *block_tables_out,
                               int32_t *context_lens_out);

pkv_status pkv_bm_stats_get(pkv_block_manager *bm, pkv_bm_stats *out);

/* Reference count of one block (-1 when block is out of range). */
int32_t pkv_bm_refcount(pkv_block_manager *bm, int32_t block);

/*
 * Utilisation simulator: requests of context_lens[i] tokens are admitted in
 * order into a pool of num_blocks blocks of block_size tokens until one does
 * not fit. With reserve_tokens > 0 every request holds
 * ceil(reserve_tokens / block_size) blocks whatever its length (contiguous
 * reserve-for-max in block units); with 0 it holds ceil(L / block_size)
 * (paged). *admitted_out: requests admitted; *utilisation_out: their tokens
 * divided by the token capacity of the blocks they hold.
 */
pkv_status pkv_bm_simulate_admission(int32_t num_blocks, int32_t block_size,
                                     const int32_t *context_lens, int32_t n,
                                     int32_t reserve_tokens, int32_t *admitted_out,
                                     double *utilisation_out);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCK_MANAGER_H */
