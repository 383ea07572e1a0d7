/*
 * pa_api.h -- C ABI of the paged-KV attention library (libpa.so, sm_103a).
 *
 * Three operations of one attention layer of a paged-KV inference engine:
 *
 *   pa_store_kv       write this step's new K/V rows into the paged pool
 *   pa_decode         one query token per sequence attending over its paged
 *                     context (split-K over context partitions)
 *   pa_prefill_paged  chunked prefill: new query tokens attending causally over
 *                     a cached paged prefix plus themselves
 * plus the decode step's store fused into decode (pa_store_decode), the same
 * store and decode over an FP8 pool (pa_store_kv_fp8, pa_decode_fp8,
 * pa_store_decode_fp8) and the
 * sampler that turns the step's logits into tokens (pa_sample).  Around them:
 *
 *   pa_decode_ex, pa_store_decode_ex   decode options: split-K plan overrides,
 *                     shared-prefix groups (read each shared page once) and
 *                     operands read at run time (pa_store_decode_fp8_ex: those)
 *   pa_decode_static_workspace  decode for callers that cannot allocate
 *   pa_prefill_paged_ex  prefill with a cap on its persistent grid
 *   pa_sm_split_*, pa_mixed_step  a mixed step's prefill and decode at once
 *                     on disjoint SM partitions
 *   pa_stage_decode_step  the host half of a captured decode step fed from
 *                     the caller's host buffers (through the operands option)
 *   pa_copy_segments  several copies in one launch, from a list read when it
 *                     runs
 *   pa_selftest_wait_timeout  shows the kernels' bounded waits ending
 * and, in pa_block_manager.h, the host-side page directory (pa_bm_*) and the
 * shared-prefix grouping of a decode batch (pa_prefix_groups).
 *
 * Conventions shared by every call
 *   - All tensor arguments are DEVICE pointers to caller-owned memory; the
 *     library allocates nothing and keeps no state besides cached device
 *     properties.  Integer size arguments are host values.  Exception: the
 *     per-step operands of pa_store_kv (k, v, slot_mapping), of
 *     pa_store_decode and pa_store_decode_fp8 (k, v, slot_mapping, q,
 *     block_tables, context_lens and out), of pa_sample (logits,
 *     temperatures, noise, tokens), the output of pa_prefill_paged (out) and
 *     those of pa_mixed_step (k, v, slot_mapping, decode_q,
 *     decode_block_tables, context_lens, prefill_out, decode_out) may instead be
 *     page-locked host memory from cudaHostAlloc / cudaMallocHost, which under
 *     unified addressing is device-accessible through its host pointer: the
 *     kernels then read and write it directly over the CPU-GPU link (zero
 *     copy; NVLink-C2C on a Grace-based GB300), so a step needs no separate
 *     copy.  The pool, the workspace and err_flag stay device memory, and the
 *     caller keeps the host buffers unchanged until the call has completed on
 *     the stream.
 *   - Element type: PA_F16 or PA_BF16 (IEEE binary16 / bfloat16) for every
 *     q/k/v/cache/out buffer of a call (the pool of the *_fp8 calls is E4M3).
 *     Arithmetic is fp32.
 *   - The pool of one layer is two buffers k_cache and v_cache, each
 *     [num_blocks, block_size, num_kv_heads, head_dim] contiguous: physical
 *     block b, token offset o, kv head g, dim d is element
 *     ((b * block_size + o) * num_kv_heads + g) * head_dim + d ("nano-vLLM
 *     Part 2: Block Tables, KV Cache, and the Path to the GPU", section 1).
 *     A slot is the flattened row index b * block_size + o (section 2.2).
 *   - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *   - Supported: head_dim 64 or 128; num_q_heads % num_kv_heads == 0 with a
 *     group size of 1, 2, 4 or 8; block_size a power of two in [8, 1024];
 *     num_blocks * block_size <= INT32_MAX (pool rows are addressed by TMA
 *     with 32-bit coordinates).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Issue pa_store_kv before the attention call of the
 *     same step on the same stream: attention reads the stored rows.
 *   - Return value: PA_OK, or a negative PA_ERR_* code.  Argument checks run
 *     on the host before anything is launched; on PA_ERR_INVALID_ARG and
 *     PA_ERR_UNSUPPORTED no CUDA call has been made.  pa_last_error() gives a
 *     message for the calling thread's most recent failure.  The library never
 *     exits, throws or traps.
 *   - err_flag (nullable DEVICE int32): kernels OR bits into it when the DATA
 *     is invalid -- PA_FLAG_BAD_SLOT (slot outside [-1, num_blocks*block_size)),
 *     PA_FLAG_BAD_BLOCK (a block id inside a context outside [0, num_blocks)),
 *     PA_FLAG_BAD_LENGTH (a negative or over-long context / cu_seqlens),
 *     PA_FLAG_TIMEOUT (a kernel's bounded wait on its own asynchronous copies
 *     or tensor-core work gave up; the kernel drained and returned),
 *     PA_FLAG_INTERNAL (an internal layout invariant did not hold).  The
 *     offending access is skipped or kept inside the pool, so bad metadata
 *     never faults; the corresponding outputs are then unspecified.
 */
#ifndef PA_API_H
#define PA_API_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* PA_F32 is accepted only for the logits of pa_sample; PA_E4M3 (one byte,
 * OCP FP8 E4M3: bias 7, no infinities, 0x7F / 0xFF NaN, largest finite 448)
 * only as the element type of an fp8 pool, which the *_fp8 calls take
 * implicitly. */
typedef enum { PA_F16 = 0, PA_BF16 = 1, PA_F32 = 2, PA_E4M3 = 3 } pa_dtype;

enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,
    PA_ERR_UNSUPPORTED = -2,
    PA_ERR_CUDA = -3,
};

enum {
    PA_FLAG_BAD_SLOT = 1,
    PA_FLAG_BAD_BLOCK = 2,
    PA_FLAG_BAD_LENGTH = 4,
    PA_FLAG_TIMEOUT = 8,
    PA_FLAG_INTERNAL = 16,
    PA_FLAG_BAD_VALUE = 32, /* a value outside its domain (pa_sample: temperature <= 1e-10; an unaligned
                               address in pa_decode_options.operands) */
    PA_FLAG_BAD_GROUP = 64, /* a shared-prefix descriptor breaking its rules (pa_decode_options) */
};

/* Message describing the calling thread's last failed call ("" if none). */
PA_API const char *pa_last_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
PA_API int pa_version(void);

/*
 * pa_store_kv -- slot-mapped store of this step's K/V rows.
 *
 * Follows the store_kvcache kernel of "Inference engine: inside nano-vLLM"
 * (section "Attention in nano-vLLM"): for every token t with
 * s = slot_mapping[t] != -1, copy the num_kv_heads*head_dim elements of row t
 * of k into row s of k_cache, and the same for v; slot -1 (padding, e.g. a
 * CUDA-graph pad row, "nano-vLLM Part 2", section 4.2) is skipped.
 *
 *   k, v          [num_tokens, num_kv_heads, head_dim]; row t starts at
 *                 element t * k_row_stride (v_row_stride); heads and dims of a
 *                 row are contiguous.  Strides are in ELEMENTS and may exceed
 *                 num_kv_heads*head_dim (e.g. k and v as views of a fused qkv).
 *   k_cache/v_cache  the layer's pool (see above), written in place.
 *   slot_mapping  int32 [num_tokens].  Distinct slots are required for a
 *                 deterministic result; duplicated slots race.
 *   The copy is bit-exact (raw 16-bit words).
 * Errors: INVALID_ARG for null pointers, negative sizes, strides smaller than
 * a row; UNSUPPORTED for dtype/head_dim outside the supported set.
 */
PA_API int pa_store_kv(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                void *k_cache, void *v_cache, const int32_t *slot_mapping, int32_t num_tokens,
                int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                pa_dtype dtype, int32_t *err_flag, void *stream);

/*
 * pa_decode_workspace_bytes -- device scratch pa_decode needs for this shape
 * (per-partition softmax partials) on the current device: the split-K plan
 * depends on its SM count, which is queried once per device.  0 on invalid
 * arguments.
 */
PA_API size_t pa_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_blocks_per_seq, int32_t block_size);

/*
 * pa_decode -- paged GQA decode attention, one query token per sequence.
 *
 * The flash_attn_with_kvcache call of "Inference engine: inside nano-vLLM"
 * (section "Attention in nano-vLLM", decode branch) and "From nano-vLLM to
 * vLLM" section 11: sequence b attends over logical positions
 * [0, context_lens[b]) of its context, position j living in cache row
 * block_tables[b][j / block_size] * block_size + j % block_size.
 * out[b, h, :] = softmax_j(scale * q[b,h,:] . K_j) V_j, with K_j/V_j of kv head
 * h / (num_q_heads/num_kv_heads).  context_lens counts the token stored this
 * step ("nano-vLLM Part 2", section 3.1).  A context length of 0 (a padding
 * row) gives an all-zero output row and reads no page.
 *
 *   q             [batch, num_q_heads, head_dim]; row b starts at element
 *                 b * q_row_stride; heads/dims contiguous.
 *   block_tables  int32 [batch, max_blocks_per_seq] row-major, -1 padded;
 *                 entries past ceil(context_len / block_size) are never read.
 *   context_lens  int32 [batch], each in [0, max_blocks_per_seq * block_size].
 *   out           [batch, num_q_heads, head_dim] contiguous, written.
 *   workspace     device scratch of at least pa_decode_workspace_bytes(...)
 *                 bytes; its contents need no initialisation and are
 *                 clobbered.  Two calls in flight at once need two workspaces.
 * The work is split over fixed-size context partitions (one CTA per
 * sequence, kv head and partition); a second kernel merges the partitions'
 * softmax partials by log-sum-exp.  Cache pages are fetched by TMA, so
 * k_cache and v_cache must be 16-byte aligned.
 */
PA_API int pa_decode(const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
              int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
              int32_t num_blocks, int32_t block_size, float scale, void *out, void *workspace,
              size_t workspace_bytes, pa_dtype dtype, int32_t *err_flag, void *stream);

/*
 * pa_store_decode -- pa_store_kv of one decode step fused into pa_decode: one
 * launch stores each sequence's new K/V row and attends over its context.
 *
 * The two calls of the attention layer's decode branch in "Inference engine:
 * inside nano-vLLM" (section "Attention in nano-vLLM": store_kvcache, then
 * flash_attn_with_kvcache), done by one kernel.  Same result as
 *   pa_store_kv(k, v, k_row_stride, v_row_stride, k_cache, v_cache,
 *               slot_mapping, batch, ...) followed by pa_decode(...),
 * for decode steps, where the token stored for sequence b is the last
 * position of its context: slot_mapping[b] must be -1 (nothing stored) or the
 * slot of position context_lens[b] - 1, i.e.
 *   block_tables[b][(L-1) / block_size] * block_size + (L-1) % block_size
 * ("nano-vLLM Part 2", sections 2.2 and 3.1).  Any other slot sets
 * PA_FLAG_BAD_SLOT and that row is not stored.
 *   k, v          [batch, num_kv_heads, head_dim]; row b starts at element
 *                 b * k_row_stride (v_row_stride); strides multiples of 8,
 *                 pointers 16-byte aligned.
 *   slot_mapping  int32 [batch].
 *   other arguments: as pa_decode (k_cache / v_cache are written).
 * The CTA that holds sequence b's last partition for kv head g writes that
 * head's slice of the row before it reads the tile containing it; no other
 * CTA reads that slice.
 */
PA_API int pa_store_decode(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                           const int32_t *slot_mapping, const void *q, int64_t q_row_stride, void *k_cache,
                           void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, void *out,
                           void *workspace, size_t workspace_bytes, pa_dtype dtype, int32_t *err_flag,
                           void *stream);

/*
 * pa_decode_options -- optional settings of pa_decode_ex / pa_store_decode_ex.
 * Zero-initialise it and set only what you need; a NULL pointer or an
 * all-zero struct gives exactly pa_decode / pa_store_decode.  The struct is
 * host memory, read during the call only; the arrays it points to are device
 * memory (or pinned host memory, like the per-step operands), read by the
 * kernels.
 *
 * Split-K plan overrides (tuning and tests; the plan needs no help for
 * ordinary shapes):
 *   partition     tokens per split-K context partition (0: the plan).  A
 *                 multiple of 64 in [64, 2^20]; it is lowered to a multiple of
 *                 64 that keeps a partition within 256 pages of the block
 *                 table.  The result is the same attention up to the fp32
 *                 rounding of the log-sum-exp merge.
 *   stages        TMA ring depth of the partition kernel, 2 or 3 (0: the plan).
 *
 * Shared prefixes (prefix caching: sequences whose block tables begin with the
 * same physical pages, "nano-vLLM Part 2: Block Tables, KV Cache, and the Path
 * to the GPU", section 2.5; "How vLLM works", prefix caching).  Each shared
 * page is then read from memory once per group and kv head for all the group's
 * query heads, instead of once per sequence; the result is the same attention
 * (up to the fp32 rounding of the merge).  pa_prefix_groups
 * (pa_block_manager.h) derives the descriptor from the host block tables.
 *   num_groups      number of groups (0: no sharing; the fields below unused).
 *   max_group_size  host: the most sequences in one group (>= 1).
 *   max_prefix_len  host: the longest prefix_lens entry, tokens (>= 1).
 *   prefix_partition  tokens per partition of a shared prefix (0: the plan;
 *                   else a multiple of 64 in [64, 16384]).
 *   group_offsets   int32 [num_groups + 1], non-decreasing from 0: the members
 *                   of group g are group_seqs[group_offsets[g] ..
 *                   group_offsets[g + 1]).
 *   group_seqs      int32 [batch] (entries past group_offsets[num_groups]
 *                   unused): sequence indices in [0, batch), each at most once;
 *                   every group_offsets entry is at most batch.
 *   prefix_lens     int32 [batch]: the number of leading context tokens of
 *                   sequence b its group's pages hold (0 for a sequence in no
 *                   group).  For a member: a multiple of block_size, the same
 *                   for every member of the group, below context_lens[b]
 *                   (the token a decode step stores is never shared), at most
 *                   max_prefix_len, and the first prefix_lens[b] / block_size
 *                   block-table entries equal across the group.
 * A descriptor breaking these rules sets PA_FLAG_BAD_GROUP where a kernel sees
 * it (outputs of the sequences involved are then unspecified; nothing faults);
 * a sequence with prefix_lens[b] > 0 that is in no group gets an unspecified
 * output without a flag.  Supported for 16-bit pools (pa_decode_ex,
 * pa_store_decode_ex).
 *
 * Operands read at run time (an extension with no counterpart on the pages;
 * it serves the captured decode step of "nano-vLLM Part 2", section 4.2, whose
 * graph has fixed arguments):
 *   operands      NULL, or three addresses {q, k, v} in device-readable memory
 *                 (device memory, or page-locked host memory from cudaHostAlloc /
 *                 cudaMallocHost), read by the kernels when they run in place of
 *                 the call's q, k and v arguments (pa_decode_ex reads only
 *                 entry 0).  Each address must hold a tensor of the shape,
 *                 element type and row stride the call's own arguments
 *                 describe, device-accessible (device or page-locked host
 *                 memory) and 16-byte aligned; a CTA that reads an unaligned
 *                 one sets PA_FLAG_BAD_VALUE and skips its work (the outputs
 *                 are then unspecified).  A CUDA graph of the call is then pointed at a new
 *                 step's buffers by rewriting the three addresses between
 *                 replays; the call's own q, k and v must still be valid
 *                 addresses (they are checked, not read).
 */
typedef struct pa_decode_options {
    int32_t partition;
    int32_t stages;
    int32_t num_groups;
    int32_t max_group_size;
    int32_t max_prefix_len;
    int32_t prefix_partition;
    const int32_t *group_offsets;
    const int32_t *group_seqs;
    const int32_t *prefix_lens;
    const void *const *operands;
} pa_decode_options;

/* Workspace bytes of pa_decode_ex / pa_store_decode_ex with these options
 * (NULL: as pa_decode_workspace_bytes).  0 on invalid arguments. */
PA_API size_t pa_decode_ex_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t max_blocks_per_seq, int32_t block_size,
                                           const pa_decode_options *options);

/* pa_decode with options (see pa_decode_options); the workspace must hold
 * pa_decode_ex_workspace_bytes(..., options) bytes.  Errors as pa_decode, and
 * INVALID_ARG for an option outside its range. */
PA_API int pa_decode_ex(const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                        int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t num_blocks, int32_t block_size, float scale, void *out, void *workspace,
                        size_t workspace_bytes, const pa_decode_options *options, pa_dtype dtype,
                        int32_t *err_flag, void *stream);

/* pa_store_decode with options; as pa_decode_ex for the workspace and errors. */
PA_API int pa_store_decode_ex(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                              const int32_t *slot_mapping, const void *q, int64_t q_row_stride, void *k_cache,
                              void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                              const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                              float scale, void *out, void *workspace, size_t workspace_bytes,
                              const pa_decode_options *options, pa_dtype dtype, int32_t *err_flag, void *stream);

/*
 * pa_decode_static_workspace -- pa_decode for callers that cannot allocate
 * device memory.  The pages describe no such call: it has no counterpart there.
 *
 * Same arguments and result as pa_decode, minus the workspace.  The split-K
 * partials go to scratch memory owned by the library itself: one static
 * 8 MiB device array on every GPU the library is loaded on, held until the
 * process exits.  It serves engines that gave (nearly) all free device memory
 * to their KV pool at start-up, and plugins whose host framework owns every
 * device allocation: neither can cudaMalloc a per-call workspace.  This call
 * allocates nothing.
 *   - A shape whose pa_decode_workspace_bytes(...) exceeds 8 MiB is rejected
 *     with PA_ERR_UNSUPPORTED (see pa_last_error) before any CUDA call.
 *   - Set-up: CUDA loads modules lazily by default, so the 8 MiB array (and
 *     the decode kernels' code) would be placed in device memory only at the
 *     first call on a device.  Call pa_decode_static_workspace once with
 *     batch == 0 (the other pointers may be NULL) on each device, with that
 *     device current, BEFORE reserving the KV pool and before any stream
 *     capture: that call looks up the array's device address
 *     (cudaGetSymbolAddress), loads every kernel this entry point launches,
 *     and computes nothing.  Later calls take no device memory.  The address
 *     is cached per device with the id of its CUDA context, so after a device
 *     reset the next call looks it up again (and places the array again).
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents.  Each call writes every scratch element it later reads, so
 *     nothing needs clearing.  Calls that overlap on the GPU (unordered
 *     streams) race on the scratch: order them on one stream.
 */
PA_API int pa_decode_static_workspace(const void *q, int64_t q_row_stride, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t num_blocks, int32_t block_size,
                                      float scale, void *out, pa_dtype dtype, int32_t *err_flag,
                                      void *stream);

/*
 * FP8 pools.  "Inference engine: inside nano-vLLM" (Appendix B, the KV cache
 * sizing) lists fp8 (1 byte) beside fp16 (2 bytes) as the cache's element
 * type, which halves a pool's bytes and with them what decode streams.  The
 * pages fix no format; this library's reading: the pool holds E4M3 codes
 * (PA_E4M3 above) in the same [num_blocks, block_size, num_kv_heads,
 * head_dim] layout, one byte per element, with one fp32 scale per tensor for K
 * and one for V: element x is stored as the E4M3 code nearest to x / scale
 * (ties to the even code, saturating at +-448) and read back as
 * code_value * scale.  The scales are the caller's (e.g. calibrated amax / 448).
 */

/*
 * pa_store_kv_fp8 -- pa_store_kv into an E4M3 pool: the same slot mapping,
 * padding (-1) and error rules, each element quantised as above (fp32
 * division by the scale, round to nearest even, saturating; NaN stays NaN).
 *   k, v          16-bit rows of dtype (PA_F16 / PA_BF16) as pa_store_kv.
 *   k_cache/v_cache  E4M3 pool, one byte per element, written in place.
 *   k_scale, v_scale  finite and > 0.
 *   num_kv_heads*head_dim and the row strides multiples of 8; k and v
 *   16-byte aligned, the caches 8-byte aligned (16-byte and 8-byte vectors).
 * The result equals the element-wise rule exactly (bit-exact codes).
 */
PA_API int pa_store_kv_fp8(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                    void *k_cache, void *v_cache, const int32_t *slot_mapping, int32_t num_tokens,
                    int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                    pa_dtype dtype, float k_scale, float v_scale, int32_t *err_flag, void *stream);

/* pa_decode_fp8_workspace_bytes -- as pa_decode_workspace_bytes, for pa_decode_fp8. */
PA_API size_t pa_decode_fp8_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t max_blocks_per_seq, int32_t block_size);

/*
 * pa_decode_fp8 -- pa_decode over an E4M3 pool: the same attention with
 * K_j = k_code * k_scale and V_j = v_code * v_scale.
 *   q, out        dtype (PA_F16 / PA_BF16), as pa_decode.
 *   k_cache/v_cache  E4M3 pool, 16-byte aligned.
 *   workspace     at least pa_decode_fp8_workspace_bytes(...) bytes.
 *   other arguments: as pa_decode.
 * head_dim must be 128 (PA_ERR_UNSUPPORTED otherwise).  The codes are
 * widened to fp16 (exactly) for the tensor-core products, q is converted to
 * fp16 (exact for bf16 values of magnitude in [2^-14, 65504]), P is rounded
 * to fp16 and the scales are applied to the fp32 scores and outputs.
 */
PA_API int pa_decode_fp8(const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache,
                  const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                  int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t num_blocks, int32_t block_size, float scale, float k_scale, float v_scale, void *out,
                  void *workspace, size_t workspace_bytes, pa_dtype dtype, int32_t *err_flag, void *stream);

/*
 * pa_store_decode_fp8 -- pa_store_decode over an E4M3 pool: each sequence's
 * new K/V row is quantised as pa_store_kv_fp8 does (same codes) into slot
 * slot_mapping[b], which must be -1 or the slot of position
 * context_lens[b] - 1 (else PA_FLAG_BAD_SLOT and the row is not stored), and
 * the same launch attends as pa_decode_fp8.  Argument rules: those of
 * pa_store_decode for k, v, their strides and slot_mapping, those of
 * pa_decode_fp8 for the rest (workspace: pa_decode_fp8_workspace_bytes).
 */
PA_API int pa_store_decode_fp8(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                        const int32_t *slot_mapping, const void *q, int64_t q_row_stride, void *k_cache,
                        void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                        const int32_t *context_lens, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, float k_scale,
                        float v_scale, void *out, void *workspace, size_t workspace_bytes, pa_dtype dtype,
                        int32_t *err_flag, void *stream);

/*
 * pa_store_decode_fp8_ex -- pa_store_decode_fp8 with decode options, of which
 * an E4M3 pool takes only `operands` (q and the new rows read through three
 * addresses when the kernels run, as for pa_store_decode_ex); every other field
 * must be 0 (PA_ERR_INVALID_ARG otherwise), so the workspace is still
 * pa_decode_fp8_workspace_bytes.  NULL options: pa_store_decode_fp8.
 */
PA_API int pa_store_decode_fp8_ex(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                                  const int32_t *slot_mapping, const void *q, int64_t q_row_stride, void *k_cache,
                                  void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                                  float scale, float k_scale, float v_scale, void *out, void *workspace,
                                  size_t workspace_bytes, const pa_decode_options *options, pa_dtype dtype,
                                  int32_t *err_flag, void *stream);

/*
 * pa_prefill_paged -- causal varlen prefill over a paged prefix.
 *
 * The flash_attn_varlen_func call of "Inference engine: inside nano-vLLM"
 * (section "Attention in nano-vLLM", prefill branch) with the cu_seqlens of
 * "nano-vLLM Part 2", section 4.1.  Sequence i owns query rows
 * [cu_seqlens_q[i], cu_seqlens_q[i+1]) (Lq of them) and a context of
 * Lk = cu_seqlens_k[i+1] - cu_seqlens_k[i] >= Lq tokens whose first
 * P = Lk - Lq are a cached prefix.  Query row r (0-based within the
 * sequence) attends over context positions [0, P + r] (causal, aligned to the
 * end of the context).
 *
 * Where the keys come from, as in the pages' attention layer:
 *   - block_tables != NULL: every context position j in [0, Lk) is read from
 *     the pool through block_tables[i] -- the prefix and this step's rows,
 *     which pa_store_kv must already have written.  k and v are not read.
 *   - block_tables == NULL: no prefix (Lk must equal Lq for every sequence);
 *     keys are rows [cu_seqlens_q[i], cu_seqlens_q[i+1]) of k and v.
 *
 *   q             [total_q, num_q_heads, head_dim] contiguous; total_q (host) is
 *                 its row count, and cu_seqlens_q[num_seqs] must not exceed it.
 *   k, v          [total_q, num_kv_heads, head_dim] contiguous (may be NULL
 *                 when block_tables != NULL).
 *   cu_seqlens_q/k  int32 [num_seqs + 1], DEVICE.
 *   max_seqlen_q/k  host upper bounds on Lq / Lk (size the launch).
 *   out           [total_q, num_q_heads, head_dim] contiguous, written.
 * Buffers q, k, v, k_cache, v_cache must be 16-byte aligned (TMA); scale must
 * be positive (the kernel takes the row maximum of the unscaled scores).
 * QK^T and PV run on the tensor cores (tcgen05, accumulators in TMEM); a work
 * item is 128 query rows of two query heads of one GQA group (one head without
 * GQA), and K/V tiles of 128 keys come through the block table by TMA.  The
 * grid is persistent: one CTA per SM of the device, each working through its
 * share of the items (dealt out longest first) with the K/V stream running on
 * from one item into the next.
 */
PA_API int pa_prefill_paged(const void *q, const void *k, const void *v, const void *k_cache,
                     const void *v_cache, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                     int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
                     const int32_t *block_tables, int32_t max_blocks_per_seq, int32_t num_q_heads,
                     int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                     float scale, void *out, pa_dtype dtype, int32_t *err_flag, void *stream);

/*
 * pa_prefill_paged_ex -- pa_prefill_paged with launch options (opt may be
 * NULL: the defaults, which is pa_prefill_paged).
 *   max_ctas  0: one CTA per SM of the device.  Otherwise the kernel occupies
 *             at most max_ctas SMs (1 <= max_ctas <= 65535): pass the SM count
 *             of the partition when `stream` belongs to a green context with
 *             fewer SMs than the device, or to leave SMs to concurrent work.
 *             The results do not depend on it, bit for bit: an item is
 *             computed the same way whichever CTA takes it.
 * PA_ERR_INVALID_ARG for a max_ctas outside that range.
 */
typedef struct pa_prefill_options {
    int32_t max_ctas;
} pa_prefill_options;
PA_API int pa_prefill_paged_ex(const void *q, const void *k, const void *v, const void *k_cache,
                               const void *v_cache, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                               int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
                               const int32_t *block_tables, int32_t max_blocks_per_seq, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                               float scale, void *out, pa_dtype dtype, int32_t *err_flag,
                               const pa_prefill_options *opt, void *stream);

/*
 * pa_copy_segments -- `count` copies (0 <= count <= 64) in one kernel on `stream`.
 * The list `segments` is read when the kernel runs, from device memory or
 * page-locked host memory (cudaHostAlloc / cudaMallocHost), and each src / dst
 * is a device-accessible address (device memory, or page-locked host memory
 * through its host pointer).  So a CUDA graph that begins with this call reads
 * a new step's inputs where the caller left them once the caller rewrites the
 * list: the step's inputs need no host-side copy into the graph's staging, and
 * all SMs pull them over the CPU-GPU link at once.  Segments must not overlap
 * one another's destinations; the copy uses 16-byte accesses where both
 * addresses are 16-byte aligned.  The pages describe no such call (the
 * library's way of feeding the decode step of "Inference engine: inside
 * nano-vLLM", section "Attention in nano-vLLM", from host buffers).
 * PA_ERR_INVALID_ARG for a count outside [0, 64] or a null list with count > 0.
 */
typedef struct pa_copy_segment {
    const void *src;
    void *dst;
    uint64_t bytes;
} pa_copy_segment;
PA_API int pa_copy_segments(const pa_copy_segment *segments, int32_t count, void *stream);

/*
 * pa_decode_staging -- one bucket of a captured decode step (a CUDA graph of
 * pa_store_decode_ex, optionally preceded by pa_copy_segments): the host
 * arrays its kernels read when it is replayed, all page-locked and owned by
 * the caller.  The pages record one graph per padded decode batch size and
 * have a step write its slot mapping, context lengths and block tables into
 * the graph's fixed buffers, padding the unused rows ("nano-vLLM Part 2",
 * section 4.2); this struct names those buffers for one bucket.
 *   rows            the bucket: rows of every per-sequence array (> 0).
 *   max_blocks      columns of block_tables (> 0).
 *   block_size      tokens per page of the pool (> 0).
 *   slot_mapping    int32 [rows]; context_lens int32 [rows];
 *   block_tables    int32 [rows, max_blocks] row-major.
 *   max_groups, max_group_size, max_prefix_len: the shared-prefix capacities
 *                   the graph was captured for (pa_decode_options), 0 when it
 *                   holds no groups, in which case the three group arrays are
 *                   NULL:
 *   group_offsets   int32 [max_groups + 1]; group_seqs int32 [rows];
 *   prefix_lens     int32 [rows].
 *   segments        the gather list the graph's pa_copy_segments reads, or
 *                   NULL; num_segments (0..4) entries whose dst the caller
 *                   set; segment_row_bytes[i] the bytes of one row of
 *                   segment i (a sequence's q, or its new K or V rows).
 *   operands        the graph's pa_decode_options operands array (three
 *                   entries: q, k, v), or NULL.
 */
typedef struct pa_decode_staging {
    int32_t rows;
    int32_t max_blocks;
    int32_t block_size;
    int32_t *slot_mapping;
    int32_t *context_lens;
    int32_t *block_tables;
    int32_t max_groups;
    int32_t max_group_size;
    int32_t max_prefix_len;
    int32_t *group_offsets;
    int32_t *group_seqs;
    int32_t *prefix_lens;
    pa_copy_segment *segments;
    int32_t num_segments;
    uint64_t segment_row_bytes[4];
    const void **operands;
} pa_decode_staging;

/* shared-prefix groups of a staged step (the `groups` argument below) */
#define PA_STAGE_NO_GROUPS 0     /* no sharing: every group empty, every prefix_lens 0 */
#define PA_STAGE_DERIVE_GROUPS 1 /* pa_prefix_groups over the staged tables (min_shared_pages 1) */
#define PA_STAGE_KEEP_GROUPS 2   /* the group arrays are left as they are (the caller writes them) */

/*
 * pa_stage_decode_step -- writes one decode step of `batch` sequences into a
 * bucket's staging, on the host, with no GPU call: slot_mapping, context_lens
 * and the first table_cols columns of block_tables into the first `batch`
 * rows (the other columns of those rows -1); rows batch..rows-1 padded (slot
 * -1, context length 0, table row untouched: a context of 0 reads no page);
 * the groups as `groups` says, unused group entries empty; and, when
 * `sources` is not NULL, segment i pointed at sources[i] for batch *
 * segment_row_bytes[i] bytes and the operands array set to sources[0..2]
 * (the caller's page-locked q / new K / new V), for whichever of the two the
 * staging holds.
 *   batch           in [0, st->rows].
 *   slot_mapping    host int32 [batch]; context_lens host int32 [batch], each
 *                   in [0, table_cols * block_size].
 *   block_tables    host int32 [batch, table_cols] row-major, table_cols in
 *                   [1, st->max_blocks].
 * Derived groups larger than the captured capacities are an error: the
 * graph's launch shape could not cover them.  Errors: PA_ERR_INVALID_ARG for
 * null pointers, sizes out of range, a context length outside the table, a
 * groups mode the staging cannot hold, derived groups beyond the
 * capacities; the staging's contents are then unspecified.
 */
PA_API int pa_stage_decode_step(const pa_decode_staging *st, int32_t batch, const int32_t *slot_mapping,
                                const int32_t *context_lens, const int32_t *block_tables, int32_t table_cols,
                                int32_t groups, const void *const *sources);

/*
 * pa_selftest_wait_timeout -- a diagnostic with no counterpart on the pages:
 * shows on a live GPU that the library's bounded waits end with a status
 * instead of a hang.  Launches one thread on `stream` that waits on an
 * mbarrier nothing ever arrives on, with the bounded wait the store, decode
 * and prefill kernels use on their own asynchronous copies and tensor-core
 * work; after `max_cycles` SM clock cycles (in (0, 4e9]) it gives up, ORs
 * PA_FLAG_TIMEOUT into the DEVICE int32 *err_flag (required) and returns,
 * and the context stays usable.
 */
PA_API int pa_selftest_wait_timeout(int64_t max_cycles, int32_t *err_flag, void *stream);

/*
 * pa_sm_split -- the GPU's SMs as two disjoint partitions, each with its own
 * stream (CUDA green contexts), for pa_mixed_step.  The pages run a mixed
 * step's chunked prefill and decode as one batch ("nano-vLLM Part 2", section
 * 4; "From nano-vLLM to vLLM", section 6.3); here the prefill, bound by
 * the tensor cores, runs on the first partition while the decode, bound by
 * HBM bandwidth (which it reaches with well under half of the SMs), runs on
 * the second.  This split is this library's choice; the pages describe none.
 *
 * pa_sm_split_create(first_sms, &split) partitions the current device:
 * first_sms SMs for the first partition, the rest for the second.  first_sms
 * must be a multiple of the device's co-scheduling granularity (8 on GB300),
 * at least its minimum partition (8), and leave at least that many SMs;
 * otherwise PA_ERR_INVALID_ARG.  PA_ERR_UNSUPPORTED when the driver lacks
 * green contexts.  It creates driver objects (two green contexts, two
 * streams, three events) and no device buffer: make one per device at
 * start-up and reuse it.  pa_sm_split_info returns the two SM counts and the
 * two streams (cudaStream_t; the split owns them: do not destroy them).
 * pa_sm_split_destroy waits for the split's streams and releases everything.
 * A split serves one step at a time: steps issued concurrently from several
 * threads on one split race on its events.
 */
typedef struct pa_sm_split pa_sm_split;
PA_API int pa_sm_split_create(int32_t first_sms, pa_sm_split **split);
PA_API int pa_sm_split_info(const pa_sm_split *split, int32_t *first_sms, int32_t *second_sms, void **first_stream,
                            void **second_stream);
PA_API void pa_sm_split_destroy(pa_sm_split *split);

/*
 * pa_mixed_step -- one mixed chunked-prefill step of an attention layer: the
 * store of every new token of the step (the prefill chunks' and the decode
 * sequences'), then the chunked prefill of the prefill sequences over their
 * cached prefixes and the decode of the others ("Inference engine: inside
 * nano-vLLM", section "Attention in nano-vLLM": store_kvcache, then
 * flash_attn_varlen_func or flash_attn_with_kvcache).  Same results, bit for
 * bit, as
 *   pa_store_kv(k, v, k_row_stride, v_row_stride, k_cache, v_cache,
 *               slot_mapping, num_tokens, ...);
 *   pa_prefill_paged(prefill_q, NULL, NULL, k_cache, v_cache, cu_seqlens_q,
 *                    cu_seqlens_k, num_prefill_seqs, total_prefill_q,
 *                    max_seqlen_q, max_seqlen_k, prefill_block_tables,
 *                    prefill_max_blocks, ..., prefill_out, ...);
 *   pa_decode(decode_q, decode_q_row_stride, k_cache, v_cache,
 *             decode_block_tables, decode_max_blocks, context_lens,
 *             decode_batch, ..., decode_out, workspace, workspace_bytes, ...);
 * on `stream` (the prefill reads its chunk's keys from the pool, so the store
 * comes first), the argument rules being those of the three calls; a prefill
 * with num_prefill_seqs == 0 or a decode with decode_batch == 0 is skipped.
 * With `split` (nullable) the store runs on `stream`, then the prefill on the
 * split's first partition and the decode on its second, at the same time,
 * and `stream` waits for both before anything issued on it later; the split
 * must belong to the current device.  Every argument is checked before
 * anything is launched.  16-bit pools only (dtype PA_F16 or PA_BF16; the
 * E4M3 pool has no prefill and so no mixed step).
 */
PA_API int pa_mixed_step(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                         const int32_t *slot_mapping, int32_t num_tokens, const void *prefill_q,
                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int32_t num_prefill_seqs,
                         int32_t total_prefill_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
                         const int32_t *prefill_block_tables, int32_t prefill_max_blocks, void *prefill_out,
                         const void *decode_q, int64_t decode_q_row_stride, const int32_t *decode_block_tables,
                         int32_t decode_max_blocks, const int32_t *context_lens, int32_t decode_batch,
                         void *decode_out, void *workspace, size_t workspace_bytes, void *k_cache, void *v_cache,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                         int32_t block_size, float scale, pa_dtype dtype, int32_t *err_flag,
                         const pa_sm_split *split, void *stream);

/*
 * pa_sample -- one token per row by temperature sampling, written as the
 * exponential race of "From nano-vLLM to vLLM: Scheduler, Paged KV Cache,
 * Prefill/Decode, Tensor Parallelism, and Sampling", section 17 (17.1, 17.4,
 * 17.6).  For row b, in fp32:
 *   a_i = logits[b, i] / temperatures[b];   p = softmax(a)
 *   tokens[b] = argmax_i  p_i / max(E_i, 1e-10)   (the first index on ties)
 * with E_i ~ Exp(1) independent, which selects token i with probability p_i.
 *
 *   logits        [batch, vocab], dtype PA_F32, PA_BF16 or PA_F16; row b
 *                 starts at element b * logits_row_stride (>= vocab).  Rows
 *                 that start on a 16-byte boundary are read with 16-byte
 *                 vectors, others element by element.
 *   temperatures  fp32 [batch], DEVICE; each must exceed 1e-10 (the pages'
 *                 sampler has no greedy path): a row whose temperature does
 *                 not gets token -1 and PA_FLAG_BAD_VALUE.
 *   noise         fp32 [batch, vocab] contiguous, DEVICE: the E_i (drawn by
 *                 the caller, e.g. torch's exponential_); or NULL: the kernel
 *                 draws them from Philox4x32-10 (Salmon et al., SC'11) keyed
 *                 by `seed`, counter (i / 4, b, offset low, offset high),
 *                 u = ((x >> 8) + 1) * 2^-24 in (0, 1], E = -log(u).  Pass a
 *                 new offset for every call that needs fresh samples.
 *   tokens        int32 [batch], DEVICE, written.
 * The kernel takes the decision in the race's log form, argmax_i
 * logits[b, i] / T - log(max(E_i, 1e-10)), which section 17.5 of the same
 * page shows selects the same token (the softmax denominator is common to all
 * i); only near-ties can resolve differently from the fp32 ratio form.  A row
 * is split over a cluster of 8 CTAs that compare their winners through
 * distributed shared memory; batch <= 65535.  A row with no finite logit
 * gets -1.
 */
PA_API int pa_sample(const void *logits, int64_t logits_row_stride, int32_t batch, int32_t vocab, pa_dtype dtype,
                     const float *temperatures, const float *noise, uint64_t seed, uint64_t offset,
                     int32_t *tokens, int32_t *err_flag, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_API_H */
