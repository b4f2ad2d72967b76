/*
 * libpkv — paged KV-cache decode for NVIDIA GB300 (sm_103a).
 *
 * C ABI of the hot path: writing each new token's K/V into its slot of a
 * paged pool, decode attention that gathers K/V through per-sequence block
 * tables, and the whole-block copy behind copy-on-write.
 *
 * Data model ("PagedAttention — Math + Memory Model", section "PagedAttention:
 * blocks and the block table"; "KV-cache paging in vLLM", section
 * "PagedAttention: Paging for KV-Caches"): the KV cache is cut into physical
 * blocks of B tokens held in one device pool; a per-sequence block table maps
 * logical block i (tokens i*B .. i*B+B-1) to a physical block id.
 *
 * Layouts (row-major, contiguous, device memory unless stated otherwise):
 *   k_pool, v_pool   [num_blocks][num_kv_heads][block_size][head_dim]   dtype
 *                    One (block, kv head) chunk is block_size*head_dim
 *                    contiguous elements.
 *   q, out           [num_seqs][num_q_heads][head_dim]
 *   k_new, v_new     [num_tokens][num_kv_heads][head_dim]                dtype
 *   block_tables     [num_seqs][max_blocks_per_seq] int32
 *   context_lens     [num_seqs] int32 (tokens, including the one appended
 *                    this step)
 *   slot_mapping     [num_tokens] int64, slot = block_id*block_size + offset
 *
 * Grouped queries: q head h attends with kv head h / (num_q_heads /
 * num_kv_heads).
 *
 * Ownership: every pointer belongs to the caller. Calls that take a `stream`
 * (a cudaStream_t passed as void*, NULL = the legacy default stream) only
 * enqueue work: they return before the GPU runs it, and the caller keeps the
 * buffers alive until the stream has passed that point. The library allocates
 * no device memory on these paths; decode attention uses a caller-provided
 * workspace.
 *
 * Errors: each call returns a pkv_status. Arguments the host can check (null
 * pointers, sizes, alignment, unsupported shapes) are rejected before any
 * launch, with nothing enqueued. Values that live on the device (block ids,
 * slots, context lengths) are checked by the kernels: a bad value sets a bit
 * in a per-device error word and the access is skipped or clamped, never
 * faulting; pkv_get_error reads and clears that word. pkv_last_error_message
 * gives the text of the last failure on the calling thread.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_F32 = 0,
    PKV_F16 = 1,
    PKV_BF16 = 2,
    PKV_INT8 = 3,       /* 8-bit cache codes only (pkv_qcache_desc.code_dtype) */
    PKV_FP8_E4M3 = 4    /* 8-bit cache codes only (pkv_qcache_desc.code_dtype) */
} pkv_dtype;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,   /* null pointer, bad size, misalignment       */
    PKV_ERR_UNSUPPORTED = -2,   /* dtype, head_dim, block_size or shape        */
    PKV_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed        */
    PKV_ERR_OUT_OF_RANGE = -4,  /* the device error word was non-zero          */
    PKV_ERR_TIMEOUT = -5,       /* a bounded on-chip wait gave up              */
    PKV_ERR_WORKSPACE = -6,     /* workspace missing or too small              */
    PKV_ERR_NO_BLOCKS = -7      /* block manager: not enough free blocks; the
                                   call changed nothing                        */
} pkv_status;

/* Bits of the device error word (see pkv_get_error). */
#define PKV_DEVERR_BLOCK_ID   0x1u  /* a block table entry outside [0, num_blocks) */
#define PKV_DEVERR_CONTEXT    0x2u  /* a context length < 0 or > max_blocks*block_size */
#define PKV_DEVERR_TIMEOUT    0x4u  /* an on-chip barrier wait ran out of time */
#define PKV_DEVERR_SLOT       0x8u  /* an append slot outside the pool */

/* Shape of one paged K/V pool pair. */
typedef struct {
    int32_t num_blocks;    /* physical blocks in each pool, >= 1               */
    int32_t block_size;    /* tokens per block B: 8, 16 or 32                  */
    int32_t num_kv_heads;  /* Hk >= 1                                          */
    int32_t head_dim;      /* D: 64 or 128                                     */
    int32_t dtype;         /* pkv_dtype of the pools, q, k_new and v_new       */
} pkv_cache_desc;

/*
 * pkv_append — write one K row and one V row per (token, kv head) into its slot.
 *
 * Passage: blocks are filled as the model generates tokens ("KV-Cache
 * Optimization & PagedAttention for Long-Context Agents", section "Key
 * KV-Cache Optimization Principles", item 1; "PagedAttention — Math + Memory
 * Model", section "PagedAttention: blocks and the block table": a sequence
 * that needs slot B+1 gets a new block appended to its table — the block is
 * allocated by the caller; this call only writes the slot).
 *
 * For token i with s = slot_mapping[i] >= 0, for every kv head g:
 *   k_pool[s / B][g][s % B][:] = k_new[i][g][:]   (same for v)
 * Tokens with s < 0 are skipped. Byte-exact copy. Slots are unique per call
 * (duplicates: one of the writers wins, which one is unspecified). A slot past
 * the pool sets PKV_DEVERR_SLOT and is skipped.
 * Pointers: k_new, v_new, slot_mapping, k_pool, v_pool on the device, 16-byte
 * aligned. num_tokens == 0 is a no-op.
 */
pkv_status pkv_append(const pkv_cache_desc *cache, const void *k_new, const void *v_new,
                      const int64_t *slot_mapping, int32_t num_tokens,
                      void *k_pool, void *v_pool, void *stream);

/* Options of pkv_append_ex. Zero-initialise for the defaults. */
typedef struct {
    int32_t inputs_ready;    /* 1: no kernel that may still be running writes
                                k_new, v_new or slot_mapping (for instance they
                                were copied from the host before the preceding
                                kernel was launched), so the append reads them
                                before it waits for the preceding kernel on
                                `stream`; the pool writes still wait for it.
                                0 (default): everything waits.              */
} pkv_append_options;

/* pkv_append with options (NULL = defaults). Same contract. */
pkv_status pkv_append_ex(const pkv_cache_desc *cache, const void *k_new, const void *v_new,
                         const int64_t *slot_mapping, int32_t num_tokens, void *k_pool,
                         void *v_pool, void *stream, const pkv_append_options *options);

/*
 * pkv_decode_workspace_bytes — bytes of workspace pkv_decode_attention needs.
 *
 * The split-K partials are bounded by the number of CTAs of one launch on the
 * current device, not by the batch or the context length: num_seqs and
 * max_context_len are accepted for a stable signature and do not change the
 * result. Returns 0 if the arguments are invalid or no device is present.
 */
size_t pkv_decode_workspace_bytes(const pkv_cache_desc *cache, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t max_context_len);

/*
 * pkv_decode_attention — one decode step of paged attention, split-K over the
 * context with a log-sum-exp merge.
 *
 * Passage: the attention kernel reads the block table and gathers keys and
 * values from the scattered physical blocks for QK^T and the value-weighted
 * sum ("PagedAttention — Math + Memory Model", section "PagedAttention: blocks
 * and the block table"; "KV-cache paging in vLLM", section "The Attention
 * Kernel Change").
 *
 * For sequence s with L = context_lens[s] and q head h (kv head g = h / G,
 * G = num_q_heads / num_kv_heads):
 *   z_t = scale * <q[s][h], K_t>,  t < L, K_t = k_pool[tab[s][t/B]][g][t%B]
 *   out[s][h] = sum_t softmax(z)_t * V_t
 * computed with fp32 accumulation and written in out_dtype (round to nearest
 * even). L == 0 writes zeros. Pool rows past L in a last block are never used.
 *
 * q, k_pool, v_pool: 16-byte aligned device pointers (dtype cache->dtype).
 * out: device, out_dtype any pkv_dtype. block_tables has max_blocks_per_seq
 * columns; every L must satisfy L <= max_blocks_per_seq * block_size (a larger
 * value is clamped and sets PKV_DEVERR_CONTEXT). Block ids outside the pool
 * set PKV_DEVERR_BLOCK_ID and read as zeros.
 * workspace: device memory of at least pkv_decode_workspace_bytes(...) bytes,
 * 16-byte aligned, owned by the caller, reused by every call on `stream`
 * (two streams need two workspaces). It must be zero-filled before the first
 * call that uses it (e.g. one cudaMemsetAsync after allocating): it holds the
 * arrival counters that let the last CTA holding a piece of a split unit
 * merge the pieces, and every call puts them back to zero. After a call whose
 * device error word reports PKV_DEVERR_TIMEOUT some counters may be left
 * non-zero: zero the workspace again before reusing it.
 * num_q_heads must be a multiple of num_kv_heads. num_seqs == 0 is a no-op.
 */
pkv_status pkv_decode_attention(const pkv_cache_desc *cache, const void *q, int32_t num_seqs,
                                int32_t num_q_heads, const void *k_pool, const void *v_pool,
                                const int32_t *block_tables, int32_t max_blocks_per_seq,
                                const int32_t *context_lens, float scale, void *out,
                                int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                void *stream);

/* Largest num_ctas of pkv_decode_options. The workspace begins with a fixed
 * region of PKV_MAX_DECODE_CTAS x 16 bytes of arrival counters, whatever the
 * launch, so one zero-filled workspace serves launches of any CTA count. */
#define PKV_MAX_DECODE_CTAS 4096

/* Tuning and measurement options for pkv_decode_attention_ex. Zero-initialise
 * for the defaults. */
typedef struct {
    int32_t num_ctas;        /* CTAs of the split-K launch, 0..PKV_MAX_DECODE_CTAS;
                                0 = SMs x occupancy                             */
    int32_t consumer;        /* 0 auto (tensor cores for fp16/bf16, CUDA cores
                                for fp32); 1 CUDA-core (SIMT) math; 2 tensor-
                                core mma (16-bit dtypes only)                   */
    void *timing_events[2];  /* optional cudaEvent_t recorded on `stream` just
                                before and just after the decode kernel of the
                                first 1024 sequences (NULL = not recorded);
                                under stream capture they become event-record
                                nodes */
    float *lse_out;          /* optional device [num_seqs][num_q_heads] fp32:
                                log2 of the softmax denominator of each head,
                                log2 sum_t exp(scale <q, k_t>) (-inf for an
                                empty context), to merge partial attentions
                                computed apart; NULL = not written          */
    int32_t tables_ready;    /* 1: no kernel that may still be running writes
                                context_lens or block_tables (slots for flat
                                spans): they come, say, from host copies that
                                completed before the preceding kernel on
                                `stream` was launched. The decode then reads
                                them while that kernel still runs (it is
                                launched with programmatic dependent launch).
                                q, the pools, the output and the workspace are
                                always touched after that kernel finishes
                                (unless pending_tail says otherwise).
                                0 (default): everything waits for it.       */
    int32_t pending_tail;    /* n >= 0. n > 0 (needs tables_ready): q and every
                                K/V row at positions below L - n of each
                                sequence of context length L may be read before
                                the preceding kernel on `stream` finishes. The
                                caller guarantees that no kernel that may still
                                be running writes them: not the preceding
                                kernel, and not an earlier one either, since
                                with programmatic launch a chain of kernels can
                                overlap. Only the last n rows of a sequence
                                (typically the token the preceding append
                                writes) may be in flight. The decode gathers
                                and attends over the earlier rows at once, and
                                waits for the preceding kernel before the first
                                tile holding one of the last n rows and before
                                its first store to the output or the workspace.
                                In a loop that appends and decodes on one cache
                                each step, the rows of earlier steps' appends
                                count as in flight unless those kernels have
                                certainly completed (the steps use separate
                                cache copies in turn, or an event or host wait
                                separates them); a caller that rewrote other
                                rows (a copy-on-write block copy, say) leaves
                                it 0. Applies to the first 1024 sequences (one
                                launch); a longer batch's later launches wait
                                as with tables_ready. 0 (default): no early
                                rows.                                       */
} pkv_decode_options;

/* Workspace bytes for pkv_decode_attention_ex with options->num_ctas = num_ctas
 * (0 = the default launch). */
size_t pkv_decode_workspace_bytes_ex(const pkv_cache_desc *cache, int32_t num_q_heads,
                                     int32_t num_ctas);

/* pkv_decode_attention with options (NULL = defaults). Same contract. */
pkv_status pkv_decode_attention_ex(const pkv_cache_desc *cache, const void *q, int32_t num_seqs,
                                   int32_t num_q_heads, const void *k_pool, const void *v_pool,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, float scale, void *out,
                                   int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                   void *stream, const pkv_decode_options *options);

/*
 * pkv_append_decode_attention — one decode step in one launch: append each
 * sequence's new token, then attend over the context including it.
 *
 * Passages: the new token's K/V go into the next slot of the sequence's last
 * block ("KV-Cache Optimization & PagedAttention for Long-Context Agents",
 * section "Key KV-Cache Optimization Principles", item 1; "PagedAttention —
 * Math + Memory Model", section "PagedAttention: blocks and the block
 * table"), and the attention gathers the context through the block table
 * (same section; "KV-cache paging in vLLM", section "The Attention Kernel
 * Change").
 *
 * For every sequence s with L = context_lens[s] >= 1 (L counts the new
 * token), the result equals pkv_append with slot_mapping[s] = the slot of
 * position L - 1 (block_tables[s][(L-1)/B] * B + (L-1) % B) followed by
 * pkv_decode_attention:
 *   k_pool[tab[s][(L-1)/B]][g][(L-1)%B][:] = k_new[s][g][:]   (same for v)
 *   out[s][h] = softmax over t < L of scale <q[s][h], K_t>, weighting V_t
 * The attention reads the new rows from k_new / v_new, so the pool rows of
 * position L - 1 are never read (the slot may hold anything before the call);
 * the kernel writes them after its other work, byte-exact. L == 0 appends
 * nothing and writes zeros. A block id outside the pool sets
 * PKV_DEVERR_BLOCK_ID, reads as zeros and is not written.
 * k_new, v_new: device [num_seqs][num_kv_heads][head_dim] in cache->dtype,
 * 16-byte aligned. Everything else, workspace and options included, as for
 * pkv_decode_attention_ex, with one reading of pending_tail: the newest row
 * comes from k_new / v_new, so pending_tail n names the n newest rows of the
 * context as possibly in flight, of which only n - 1 are pool rows
 * (pending_tail 1: none; a loop that decodes one cache every step, each call
 * appending the row the next call reads from the pool, gives 2), and k_new
 * and v_new count as inputs that may be read early, like q.
 */
pkv_status pkv_append_decode_attention(const pkv_cache_desc *cache, const void *q,
                                       int32_t num_seqs, int32_t num_q_heads, const void *k_new,
                                       const void *v_new, void *k_pool, void *v_pool,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *context_lens, float scale, void *out,
                                       int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                       void *stream, const pkv_decode_options *options);

/*
 * pkv_decode_attention_static — pkv_decode_attention for callers that cannot
 * allocate device memory. The pages have no counterpart to this entry point.
 *
 * Some callers cannot provide the split-K workspace: a program that has
 * already given its whole device-memory budget to the KV-cache pool, a
 * plug-in that may only use memory its host framework owns, or code on a
 * path where cudaMalloc (which can synchronise the device) is not allowed.
 * This call takes the same inputs and output as pkv_decode_attention, minus
 * the workspace, and uses instead a fixed scratch array of
 * PKV_STATIC_SCRATCH_BYTES in the library's own device memory (every GPU that
 * loads the library holds it until the process exits). It allocates nothing.
 *
 * It launches one split-K CTA per SM; a shape whose scratch need exceeds
 * PKV_STATIC_SCRATCH_BYTES (need = 16 x PKV_MAX_DECODE_CTAS + SMs x 8 x
 * heads-per-unit x (head_dim + 4) bytes, heads-per-unit = min(16,
 * num_q_heads/num_kv_heads))
 * is rejected with PKV_ERR_WORKSPACE and nothing is enqueued.
 * The first call on a device finds the scratch array's device address (once
 * per device, with that device current); make that first call before any
 * stream capture. All calls on a device share the array. It starts zeroed and
 * every call leaves its arrival counters zero, so it needs no clearing; when
 * pkv_get_error reports PKV_DEVERR_TIMEOUT it zeroes the array of the current
 * device again. Calls whose kernels overlap on the GPU race on it, so order
 * them (e.g. one stream).
 */
#define PKV_STATIC_SCRATCH_BYTES (2u << 20)
pkv_status pkv_decode_attention_static(const pkv_cache_desc *cache, const void *q,
                                       int32_t num_seqs, int32_t num_q_heads,
                                       const void *k_pool, const void *v_pool,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *context_lens, float scale, void *out,
                                       int32_t out_dtype, void *stream);

/*
 * pkv_block_copy — copy whole physical blocks, K and V, all kv heads.
 *
 * Passage: copy-on-write copies the one block a writer hits while others
 * still share it ("PagedAttention — Math + Memory Model", section
 * "Copy-on-write"; the refcount decision and the table update are the
 * caller's).
 *
 * For each pair i: pool[dst_i][:][:][:] = pool[src_i][:][:][:] for both pools.
 * src_dst_pairs is HOST memory, [num_pairs][2] int64 (src, dst); the library
 * reads it during the call and passes the ids to the kernel by value, so the
 * caller may reuse it on return. Rejected with PKV_ERR_INVALID_ARG (nothing
 * enqueued): an id outside [0, num_blocks), two pairs with the same dst, or a
 * dst that is also some pair's src. Byte-exact. num_pairs == 0 is a no-op.
 */
pkv_status pkv_block_copy(const pkv_cache_desc *cache, const int64_t *src_dst_pairs,
                          int32_t num_pairs, void *k_pool, void *v_pool, void *stream);

/* ------------------------------------------------------- prefix-aware decode
 *
 * Passage: identical prompt prefixes are stored once and shared by every
 * request holding them ("KV-Cache Optimization & PagedAttention for
 * Long-Context Agents", section "Key KV-Cache Optimization Principles", item
 * 3). pkv_decode_attention_prefix decodes a group's shared prefix once per
 * unit of several sharers' query heads (8 or 16 heads a unit: 8 / G members
 * for G q heads per kv head) instead of once per sequence, each sequence's
 * private suffix on its own, and merges the two partial attentions by
 * log-sum-exp, all in one launch of the split-K kernel. The result is the
 * plain decode's, up to rounding.
 */
typedef struct {
    int32_t num_groups;
    const int32_t *group_of_seq;         /* host [num_seqs]: group id, or -1     */
    const int32_t *group_prefix_blocks;  /* host [num_groups]: shared leading
                                            table entries (>= 1); every member's
                                            table holds the same ids there and
                                            its length is at least that many
                                            blocks (a shorter one sets
                                            PKV_DEVERR_CONTEXT)                */
} pkv_prefix_groups;

/* Workspace bytes of pkv_decode_attention_prefix (0 on invalid arguments). */
size_t pkv_decode_prefix_workspace_bytes(const pkv_cache_desc *cache, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t max_blocks_per_seq,
                                         const pkv_prefix_groups *groups, int32_t num_ctas);

/*
 * pkv_decode_attention_ex for sequences that share prefixes: same inputs and
 * output, plus the group description (host arrays, read during the call).
 * workspace: at least pkv_decode_prefix_workspace_bytes, zero-filled before
 * its first use; every call leaves its counters zero again. One launch, no
 * host-to-device copy. options: num_ctas (at most PKV_MAX_DECODE_CTAS / 2),
 * consumer, tables_ready, lse_out and timing_events apply; pending_tail is
 * ignored (every read waits for the preceding kernel). The one launch covers
 * fp16 / bf16 caches on the tensor-core math whose q heads per kv head times
 * head_dim is a multiple of 128, and batches whose sequences plus prefix
 * units number at most 1024; any other call is served by the plain decode,
 * with the same result.
 */
pkv_status pkv_decode_attention_prefix(const pkv_cache_desc *cache, const void *q,
                                       int32_t num_seqs, int32_t num_q_heads, const void *k_pool,
                                       const void *v_pool, const int32_t *block_tables,
                                       int32_t max_blocks_per_seq, const int32_t *context_lens,
                                       float scale, const pkv_prefix_groups *groups, void *out,
                                       int32_t out_dtype, void *workspace,
                                       size_t workspace_bytes, void *stream,
                                       const pkv_decode_options *options);

/* ------------------------------------------------------------ 8-bit KV cache
 *
 * Passage: an 8-bit KV cache is the lever that halves the bytes each decode
 * step reads ("Contiguous vs Paged KV Cache on RDNA4", section "The order of
 * the memory levers"; "KV-Cache Optimization & PagedAttention for Long-Context
 * Agents", introduction). The pages fix no format; this library's is:
 *
 *   k_codes, v_codes    [num_blocks][num_kv_heads][block_size][head_dim] uint8
 *                       one code per element: PKV_INT8 (two's complement,
 *                       -127..127) or PKV_FP8_E4M3 (OCP E4M3: bias 7, no
 *                       infinities, largest finite 448)
 *   k_scales, v_scales  [num_blocks][num_kv_heads][block_size] float
 *                       one scale per (token, kv head) row
 *
 * The cached value of element d of a row is scale * value(code[d]). A row x
 * of D activations is quantized at append time: a = max_d |x_d| (fp32),
 * scale = a / Qmax (fp32 division, round to nearest even; Qmax = 127 for
 * int8, 448 for E4M3), code_d = x_d / scale in fp32 rounded to the nearest
 * code value (ties to even), saturated to +-Qmax; a = 0 gives scale 0 and
 * zero codes. Both K and V are stored this way. q, k_new and v_new stay in the
 * activation dtype (PKV_F16 or PKV_BF16).
 */
typedef struct {
    int32_t num_blocks;    /* physical blocks in each pool, >= 1               */
    int32_t block_size;    /* tokens per block B: 8, 16 or 32                  */
    int32_t num_kv_heads;  /* Hk >= 1                                          */
    int32_t head_dim;      /* D: 128                                           */
    int32_t code_dtype;    /* PKV_INT8 or PKV_FP8_E4M3                         */
    int32_t act_dtype;     /* PKV_F16 or PKV_BF16: q, k_new, v_new             */
} pkv_qcache_desc;

/*
 * pkv_append_quant — pkv_append for an 8-bit cache: quantizes each new token's
 * K and V rows and writes codes and scales to slot_mapping[i] (negative
 * slots are skipped; a slot past the pool sets PKV_DEVERR_SLOT and is
 * skipped). k_new, v_new: [num_tokens][num_kv_heads][head_dim] in act_dtype,
 * 16-byte aligned; code pools 16-byte aligned; scale pools 16-byte aligned.
 * Codes and scales equal the rule above bit for bit.
 */
pkv_status pkv_append_quant(const pkv_qcache_desc *cache, const void *k_new, const void *v_new,
                            const int64_t *slot_mapping, int32_t num_tokens, void *k_codes,
                            void *v_codes, float *k_scales, float *v_scales, void *stream);

/* pkv_append_quant with options (NULL = defaults). Same contract. With
 * inputs_ready (see pkv_append_options) each row is read and quantized before
 * the call waits for the preceding kernel on `stream`; only the code and
 * scale stores wait for it. */
pkv_status pkv_append_quant_ex(const pkv_qcache_desc *cache, const void *k_new,
                               const void *v_new, const int64_t *slot_mapping,
                               int32_t num_tokens, void *k_codes, void *v_codes,
                               float *k_scales, float *v_scales, void *stream,
                               const pkv_append_options *options);

/*
 * pkv_append_decode_attention_quant — pkv_append_decode_attention for an
 * 8-bit cache: each sequence's new K/V row k_new[s] / v_new[s]
 * ([num_seqs][num_kv_heads][head_dim] in act_dtype, 16-byte aligned) is
 * quantized by the rule above (the same codes and scales as
 * pkv_append_quant) and written to position context_lens[s] - 1 of its table
 * row, and the decode attention (pkv_decode_attention_quant) runs over the
 * context including it: the quantizing append, then the decode, on `stream`.
 * A sequence with context_lens[s] == 0 has no new row (its output is zeros).
 * The new rows are written after the preceding kernel on `stream` has
 * completed. Other arguments, errors and workspace: as
 * pkv_decode_attention_quant (and pkv_append_quant for the rows).
 */
pkv_status pkv_append_decode_attention_quant(
    const pkv_qcache_desc *cache, const void *q, int32_t num_seqs, int32_t num_q_heads,
    const void *k_new, const void *v_new, void *k_codes, void *v_codes, float *k_scales,
    float *v_scales, const int32_t *block_tables, int32_t max_blocks_per_seq,
    const int32_t *context_lens, float scale, void *out, int32_t out_dtype, void *workspace,
    size_t workspace_bytes, void *stream, const pkv_decode_options *options);

/* Workspace bytes for pkv_decode_attention_quant with num_ctas CTAs (0 = the
 * default launch). Same contract as pkv_decode_workspace_bytes_ex. */
size_t pkv_decode_quant_workspace_bytes(const pkv_qcache_desc *cache, int32_t num_q_heads,
                                        int32_t num_ctas);

/*
 * pkv_decode_attention_quant — pkv_decode_attention_ex over an 8-bit cache:
 * out[s][h] = softmax(scale * q K^T) V with K and V the cached values
 * scale * value(code). q: [num_seqs][num_q_heads][head_dim] in act_dtype.
 * Same contract as pkv_decode_attention_ex for tables, lengths, out, the
 * workspace (zero-filled before first use) and options, except that
 * options->consumer 1 (CUDA-core math) is not available (PKV_ERR_UNSUPPORTED).
 */
pkv_status pkv_decode_attention_quant(const pkv_qcache_desc *cache, const void *q,
                                      int32_t num_seqs, int32_t num_q_heads, const void *k_codes,
                                      const void *v_codes, const float *k_scales,
                                      const float *v_scales, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      float scale, void *out, int32_t out_dtype, void *workspace,
                                      size_t workspace_bytes, void *stream,
                                      const pkv_decode_options *options);

/*
 * pkv_block_copy_quant — pkv_block_copy for an 8-bit cache: copies the codes
 * and the scales of whole blocks. Same pair rules and errors as
 * pkv_block_copy. Byte-exact.
 */
pkv_status pkv_block_copy_quant(const pkv_qcache_desc *cache, const int64_t *src_dst_pairs,
                                int32_t num_pairs, void *k_codes, void *v_codes, float *k_scales,
                                float *v_scales, void *stream);

/*
 * pkv_get_error — synchronise `stream`, then read and clear the device error
 * word of the current device (PKV_DEVERR_* bits) into *device_error_word.
 * Returns PKV_OK when the word was zero, PKV_ERR_OUT_OF_RANGE or
 * PKV_ERR_TIMEOUT (when that bit is set) otherwise. On PKV_DEVERR_TIMEOUT it
 * also zeroes pkv_decode_attention_static's scratch on the current device:
 * the memset is enqueued on `stream` and waited for, so it has completed when
 * the call returns, whatever stream the next call uses. Caller-owned
 * workspaces are the caller's to zero.
 */
pkv_status pkv_get_error(int32_t *device_error_word, void *stream);

/*
 * pkv_debug_set_wait_fault — test hook for the bounded on-chip waits; the
 * pages have no counterpart. It lets a test make a wait run out without
 * faulting or hanging anything.
 *
 * Every wait on an on-chip barrier inside a decode kernel gives up after a
 * limit (2 s by default), sets PKV_DEVERR_TIMEOUT in the device error word
 * and ends its warp's work, so the kernel returns and the context stays
 * usable. After this call, decode launches (pkv_decode_attention*, on any
 * thread and device) use wait_limit_ns as that limit (0 restores the
 * default), and the next drop_arrivals launches each withhold one producer
 * thread's arrival on the first stage of their first CTA: that stage never
 * fills, so its wait runs out. Such a launch leaves the output of the units
 * its first CTA holds unwritten and may leave split-K arrival counters set:
 * zero the workspace before reusing it (pkv_get_error zeroes
 * pkv_decode_attention_static's scratch). Returns PKV_ERR_INVALID_ARG for
 * drop_arrivals < 0. Not for production use: set it back to (0, 0).
 */
pkv_status pkv_debug_set_wait_fault(uint64_t wait_limit_ns, int32_t drop_arrivals);

/* Static text for a status code. */
const char *pkv_status_string(pkv_status status);

/* Text of the last non-OK status returned on the calling thread ("" if none). */
const char *pkv_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
