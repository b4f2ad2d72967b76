/*
 * libpkv flat spans — a KV cache kept contiguous in virtual memory.
 *
 * Passage: instead of a block table, each sequence reserves one flat virtual
 * range and physical memory is committed into it on demand, so the attention
 * kernel reads a flat span and never gathers through a table
 * ("Contiguous vs Paged KV Cache on RDNA4", section "Why the single-user
 * verdict flipped", on vAttention; the same page's FAQ). This is the
 * alternative to the paged cache of pkv.h, built on the CUDA virtual memory
 * management calls, so that the two can be measured side by side.
 *
 * Layout: one virtual reservation holds num_slots sequence slots. Slot i
 * starts at k_base + i * slot_stride; its K span is [capacity][Hk][D]
 * (token-major: the rows of all kv heads of one token are adjacent) and its V
 * span follows at + v_offset with the same layout. Physical memory is mapped
 * in chunks of the device's allocation granularity (2 MiB on GB300) as a
 * slot grows; a slot that holds L tokens has ceil(L * Hk * D * es /
 * granularity) chunks for K and as many for V.
 *
 * Safety: the library keeps, in device memory, the number of tokens each slot
 * has memory for. The device calls never touch a row past it: the decode
 * clamps a longer context length to it (PKV_DEVERR_CONTEXT) and the append
 * skips a position past it (PKV_DEVERR_SLOT). A slot index out of range sets
 * PKV_DEVERR_BLOCK_ID (decode, length 0) or PKV_DEVERR_SLOT (append).
 *
 * Ownership and ordering: the cache owns its reservation, its physical
 * chunks and the committed-token array. pkv_flat_reserve and
 * pkv_flat_release are synchronous host calls; release a slot only after the
 * kernels that read it have finished (e.g. after a stream synchronise).
 */
#ifndef PKV_FLAT_H
#define PKV_FLAT_H

#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_flat_cache pkv_flat_cache;

typedef struct {
    void *k_base;              /* device address of slot 0's K span            */
    size_t slot_stride;        /* bytes from one slot to the next              */
    size_t v_offset;           /* bytes from a slot's K span to its V span     */
    size_t granularity;        /* bytes per physical chunk                     */
    size_t committed_bytes;    /* physical bytes mapped, K and V, all slots    */
    int32_t *committed_tokens; /* device [num_slots]: tokens each slot holds   */
} pkv_flat_info;

/*
 * New flat cache on the current device: num_slots slots of capacity_tokens
 * tokens (a multiple of 16) of num_kv_heads x head_dim (64 or 128) elements
 * of dtype (PKV_F16 or PKV_BF16), for K and for V. Reserves virtual address
 * space only; no slot holds memory yet.
 */
pkv_status pkv_flat_create(int32_t num_slots, int32_t capacity_tokens, int32_t num_kv_heads,
                           int32_t head_dim, int32_t dtype, pkv_flat_cache **out);

/* Release all memory of the cache (NULL is a no-op). No kernel may still use it. */
void pkv_flat_destroy(pkv_flat_cache *fc);

/* Map physical chunks until slot holds at least tokens tokens (never shrinks). */
pkv_status pkv_flat_reserve(pkv_flat_cache *fc, int32_t slot, int32_t tokens);

/* Unmap every chunk of slot (its kernels must have finished). */
pkv_status pkv_flat_release(pkv_flat_cache *fc, int32_t slot);

pkv_status pkv_flat_get_info(pkv_flat_cache *fc, pkv_flat_info *out);

/*
 * Write token i's K and V rows (k_new, v_new [num_tokens][Hk][D], device, the
 * cache's dtype, 16-byte aligned) at position positions[i] of slot slots[i]
 * (both device int32 [num_tokens]).
 */
pkv_status pkv_flat_append(pkv_flat_cache *fc, const void *k_new, const void *v_new,
                           const int32_t *slots, const int32_t *positions, int32_t num_tokens,
                           void *stream);

/* Workspace bytes for pkv_decode_attention_flat (same contract as pkv_decode_workspace_bytes_ex). */
size_t pkv_flat_decode_workspace_bytes(pkv_flat_cache *fc, int32_t num_q_heads, int32_t num_ctas);

/*
 * pkv_decode_attention_ex over flat spans: sequence s attends over the first
 * context_lens[s] tokens of slot slots[s] (device int32 arrays [num_seqs]).
 * q, out, scale, workspace (zero-filled before first use) and options as in
 * pkv_decode_attention_ex; tensor-core math only (options->consumer 1 is
 * PKV_ERR_UNSUPPORTED).
 */
pkv_status pkv_decode_attention_flat(pkv_flat_cache *fc, const void *q, int32_t num_seqs,
                                     int32_t num_q_heads, const int32_t *slots,
                                     const int32_t *context_lens, float scale, void *out,
                                     int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                     void *stream, const pkv_decode_options *options);

#ifdef __cplusplus
}
#endif

#endif /* PKV_FLAT_H */
