/*
 * pa_block_manager.h -- host-side page directory of the paged KV cache: the
 * component that produces the block tables and slot mappings the kernels of
 * pa_api.h consume.
 *
 * It follows the BlockManager of "Inference engine: inside nano-vLLM" and
 * "nano-vLLM Part 2: Block Tables, KV Cache, and the Path to the GPU"
 * (sections 2 and 3): fixed-size physical blocks with reference counts, a
 * free list and a used set, and prefix caching through a chained hash of full
 * blocks (h_i = H(h_{i-1}, tokens of block i)) checked against the block's
 * saved token ids.  The calls and their rules, as the pages give them:
 *   - can_allocate: walk the sequence's full blocks except its last logical
 *     block; stop at the first hash miss or token mismatch; a hit on a block
 *     in use needs no free block, a hit on a freed block does; reports the
 *     number of hit blocks, or -1 when the free blocks do not suffice.
 *   - allocate: share the hit blocks (reference count + 1, or revive a freed
 *     block with count 1), then take fresh blocks from the front of the free
 *     list for the rest; num_cached_tokens = hits * block_size.  Taking a
 *     fresh block drops its stale hash entry.
 *   - can_append / may_append: a decode step needs a new block exactly when
 *     the sequence length is 1 mod block_size (its last token starts a page).
 *   - postprocess (the scheduler's hash_blocks + bookkeeping after a model
 *     step): hash the blocks the step completed, register them, and advance
 *     num_cached_tokens by the tokens the step processed.
 *   - deallocate: walk the block table in reverse, decrement, return blocks
 *     whose count reaches 0 to the back of the free list (their hash stays
 *     registered, so a later identical prefix may revive them).
 * The hash H is 64-bit FNV-1a over the previous hash (8 bytes, little
 * endian, absent for the first block) and the block's token ids (4 bytes
 * each, little endian) -- this library's choice; the pages use xxh64.
 *
 * Sequences are identified by caller-chosen 64-bit ids.  A manager is not
 * thread-safe: one owner thread calls it.  Every function returns PA_OK (0)
 * or a negative PA_ERR_* code with a message in pa_last_error(), unless
 * stated otherwise.  No function touches the GPU.
 */
#ifndef PA_BLOCK_MANAGER_H
#define PA_BLOCK_MANAGER_H

#include "pa_api.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_bm pa_bm;

/* A manager of num_blocks blocks of block_size tokens (both > 0); NULL on bad
 * arguments or allocation failure. */
PA_API pa_bm *pa_bm_create(int32_t num_blocks, int32_t block_size);
PA_API void pa_bm_destroy(pa_bm *bm);

/* Register a sequence with its prompt token ids (n >= 1), no blocks yet. */
PA_API int pa_bm_add_sequence(pa_bm *bm, int64_t seq_id, const int32_t *token_ids, int32_t n);
/* Append a sampled token to a sequence (its K/V is computed by the next step). */
PA_API int pa_bm_append_token(pa_bm *bm, int64_t seq_id, int32_t token_id);
/* Forget a sequence, releasing its blocks first if it holds any. */
PA_API int pa_bm_remove_sequence(pa_bm *bm, int64_t seq_id);

/* *num_cached_blocks = the prefix-cache hits (>= 0) if the sequence can be
 * allocated, -1 if the free blocks do not suffice.  The sequence must hold no
 * blocks. */
PA_API int pa_bm_can_allocate(pa_bm *bm, int64_t seq_id, int32_t *num_cached_blocks);
/* Allocate after can_allocate returned num_cached_blocks (>= 0). */
PA_API int pa_bm_allocate(pa_bm *bm, int64_t seq_id, int32_t num_cached_blocks);
PA_API int pa_bm_deallocate(pa_bm *bm, int64_t seq_id);
/* 1 if a decode step of the sequence can get the block it needs, 0 if not. */
PA_API int pa_bm_can_append(pa_bm *bm, int64_t seq_id);
/* Take the block a decode step needs (when the length is 1 mod block_size). */
PA_API int pa_bm_may_append(pa_bm *bm, int64_t seq_id);
/* After a model step that processed num_scheduled_tokens of the sequence:
 * register the blocks it completed and advance num_cached_tokens. */
PA_API int pa_bm_postprocess(pa_bm *bm, int64_t seq_id, int32_t num_scheduled_tokens);

/* Queries: free blocks; a block's reference count; a sequence's block table
 * (its length is returned; at most cap entries are written); its length and
 * cached tokens (negative on error). */
PA_API int pa_bm_num_free_blocks(const pa_bm *bm);
PA_API int pa_bm_ref_count(const pa_bm *bm, int32_t block_id);
PA_API int pa_bm_block_table(const pa_bm *bm, int64_t seq_id, int32_t *out, int32_t cap);
PA_API int64_t pa_bm_seq_len(const pa_bm *bm, int64_t seq_id);
PA_API int64_t pa_bm_num_cached_tokens(const pa_bm *bm, int64_t seq_id);

/* Kernel inputs of a decode step over n sequences (each has had may_append):
 * slot_mapping[i] = slot of the last token (the one this step stores),
 * context_lens[i] = sequence length, block_tables [n, max_blocks] row-major,
 * padded with -1 ("nano-vLLM Part 2", sections 3.1-3.2).  Host buffers. */
PA_API int pa_bm_decode_inputs(const pa_bm *bm, const int64_t *seq_ids, int32_t n, int32_t max_blocks,
                               int32_t *slot_mapping, int32_t *context_lens, int32_t *block_tables);
/* Kernel inputs of a prefill step: sequence i processes num_scheduled[i]
 * tokens from its num_cached_tokens on.  slot_mapping gets sum(num_scheduled)
 * entries (first-page offset and last-page end as in section 2.2),
 * cu_seqlens_q / cu_seqlens_k get n + 1 entries (query tokens / context
 * lengths), block_tables [n, max_blocks] padded with -1.  Host buffers. */
PA_API int pa_bm_prefill_inputs(const pa_bm *bm, const int64_t *seq_ids, const int32_t *num_scheduled, int32_t n,
                                int32_t max_blocks, int32_t *slot_mapping, int32_t *cu_seqlens_q,
                                int32_t *cu_seqlens_k, int32_t *block_tables);

/*
 * pa_prefix_groups -- the shared-prefix groups of a decode batch, the input
 * of the prefix-sharing decode (pa_decode_options of pa_api.h).
 *
 * With prefix caching, sequences with a common prompt prefix point at the
 * same physical pages ("nano-vLLM Part 2", section 2.5: prompt B's table
 * [0, 3, 4, 5] starts with A's page 0; "How vLLM works", prefix caching).
 * The pages define the sharing, not a grouping of a decode batch; this
 * library's rule:
 *   1. a sequence whose context length L is 0 or at most block_size holds no
 *      complete page and is never grouped;
 *   2. the others are grouped by the first entry of their block table, groups
 *      in the order their first member appears in the batch, members in batch
 *      order;
 *   3. a group of two or more shares its first n pages: the number of leading
 *      table entries equal across all members, but at most (L - 1) /
 *      block_size for each member (the page holding a sequence's newest token,
 *      the one a decode step writes, is never shared; only complete pages are,
 *      section 2.4);
 *   4. groups with n < max(min_shared_pages, 1) are dropped, singletons too.
 *   block_tables  host int32 [batch, max_blocks] row-major, -1 padded.
 *   context_lens  host int32 [batch], each in [0, max_blocks * block_size].
 *   group_offsets host int32 [batch / 2 + 1] at least (out): the members of
 *                 group g are group_seqs[group_offsets[g] .. group_offsets[g+1]).
 *   group_seqs    host int32 [batch] (out).
 *   prefix_lens   host int32 [batch] (out): n * block_size for a member of a
 *                 group, 0 for every other sequence.
 *   *num_groups, *max_group_size, *max_prefix_len (out): the host sizes the
 *                 decode options need.
 * Errors: INVALID_ARG for null pointers, negative sizes, a context length
 * outside the table.
 */
PA_API int pa_prefix_groups(const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens,
                            int32_t batch, int32_t block_size, int32_t min_shared_pages, int32_t *group_offsets,
                            int32_t *group_seqs, int32_t *prefix_lens, int32_t *num_groups, int32_t *max_group_size,
                            int32_t *max_prefix_len);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H */
