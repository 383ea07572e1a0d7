// C ABI of the paged-KV attention library: argument validation on the host,
// then a launch on the caller's stream.  No call allocates memory.
#include <math.h>
#include <stdint.h>
#include <stdarg.h>
#include <stdio.h>

#include "pa_common.cuh"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) {
        g_err[0] = '\0';
        return PA_OK;
    }
    return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
bool aligned(const void *p, int bytes) { return reinterpret_cast<uintptr_t>(p) % bytes == 0; }
bool valid_dtype(int d) { return d == PA_F16 || d == PA_BF16; }

bool valid_scales(const pa::Fp8Scales &sc) {
    return isfinite(sc.k_scale) && sc.k_scale > 0.f && isfinite(sc.v_scale) && sc.v_scale > 0.f;
}

// Checks shared by the attention calls.  Returns PA_OK or an error code.
int check_attention_shape(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                          int32_t block_size, float scale, pa_dtype dtype) {
    if (!valid_dtype(dtype)) return fail(PA_ERR_UNSUPPORTED, "dtype %d is not PA_F16 or PA_BF16", (int)dtype);
    if (num_q_heads <= 0 || num_kv_heads <= 0)
        return fail(PA_ERR_INVALID_ARG, "head counts must be positive (H_q=%d, H_kv=%d)", num_q_heads,
                    num_kv_heads);
    if (num_q_heads % num_kv_heads)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                    num_kv_heads);
    const int group = num_q_heads / num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8)
        return fail(PA_ERR_UNSUPPORTED, "GQA group size %d (supported: 1, 2, 4, 8)", group);
    if (head_dim != 64 && head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
    if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks must be positive (%d)", num_blocks);
    if (!is_pow2(block_size) || block_size < 8 || block_size > 1024)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: powers of two in [8, 1024])", block_size);
    if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
        return fail(PA_ERR_UNSUPPORTED, "pool of %lld rows (TMA row coordinates are 32-bit)",
                    (long long)num_blocks * block_size);
    if (!isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale is not finite");
    return PA_OK;
}

}  // namespace

namespace pa {
// Records `msg` as the calling thread's last error and returns `code`.
int set_last_error(int code, const char *msg) { return fail(code, "%s", msg); }
}  // namespace pa

namespace {

// Checks of the optional settings of pa_decode_ex / pa_store_decode_ex (NULL: none).
int check_options(const pa_decode_options *opt) {
    if (!opt) return PA_OK;
    if (opt->partition && (opt->partition < 64 || opt->partition % 64 || opt->partition > (1 << 20)))
        return fail(PA_ERR_INVALID_ARG, "options.partition %d must be 0 or a multiple of 64 in [64, 2^20]",
                    opt->partition);
    if (opt->stages && opt->stages != 2 && opt->stages != 3)
        return fail(PA_ERR_INVALID_ARG, "options.stages %d must be 0, 2 or 3", opt->stages);
    if (opt->num_groups < 0) return fail(PA_ERR_INVALID_ARG, "options.num_groups %d is negative", opt->num_groups);
    if (opt->num_groups > 0) {
        if (!opt->group_offsets || !opt->group_seqs || !opt->prefix_lens)
            return fail(PA_ERR_INVALID_ARG, "options: group_offsets, group_seqs and prefix_lens are required");
        if (opt->max_group_size < 1 || opt->max_prefix_len < 1)
            return fail(PA_ERR_INVALID_ARG, "options: max_group_size %d and max_prefix_len %d must be positive",
                        opt->max_group_size, opt->max_prefix_len);
        if (opt->prefix_partition &&
            (opt->prefix_partition < 64 || opt->prefix_partition % 64 || opt->prefix_partition > 16384))
            return fail(PA_ERR_INVALID_ARG, "options.prefix_partition %d must be 0 or a multiple of 64 in [64, 16384]",
                        opt->prefix_partition);
    }
    return PA_OK;
}

// Checks of pa_decode's arguments (also those of pa_store_decode); PA_OK or an error code.
int check_decode(const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache,
                 const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                 float scale, void *out, void *workspace, size_t workspace_bytes, pa_dtype dtype,
                 pa::DecodePlan *plan, const pa::Fp8Scales *fp8 = nullptr,
                 const pa_decode_options *opt = nullptr) {
    int rc = check_attention_shape(num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, dtype);
    if (rc) return rc;
    if (fp8) {
        if (head_dim != 128) return fail(PA_ERR_UNSUPPORTED, "pa_decode_fp8: head_dim %d (supported: 128)", head_dim);
        if (!valid_scales(*fp8))
            return fail(PA_ERR_INVALID_ARG, "k_scale and v_scale must be finite and positive (%g, %g)",
                        fp8->k_scale, fp8->v_scale);
    }
    if (batch < 0) return fail(PA_ERR_INVALID_ARG, "batch is negative (%d)", batch);
    rc = check_options(opt);
    if (rc) return rc;
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
    if (static_cast<int64_t>(max_blocks_per_seq) * block_size > (1LL << 30))
        return fail(PA_ERR_INVALID_ARG, "max context of %lld tokens is too large",
                    (long long)max_blocks_per_seq * block_size);
    if (batch == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
        return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (q_row_stride < static_cast<int64_t>(num_q_heads) * head_dim || q_row_stride % 2)
        return fail(PA_ERR_INVALID_ARG, "q_row_stride %lld must be even and at least H_q*D",
                    (long long)q_row_stride);
    if (!aligned(q, 4) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 2) ||
        !aligned(workspace, 256))
        return fail(PA_ERR_INVALID_ARG, "alignment: q 4 B, caches 16 B, out 2 B, workspace 256 B");
    if (opt && opt->num_groups > 0) {
        if (fp8) return fail(PA_ERR_UNSUPPORTED, "shared-prefix groups need a 16-bit pool");
        if (opt->max_prefix_len > static_cast<int64_t>(max_blocks_per_seq) * block_size)
            return fail(PA_ERR_INVALID_ARG, "options.max_prefix_len %d is longer than a block table",
                        opt->max_prefix_len);
    }
    *plan = pa::plan_decode(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
                            fp8 != nullptr, opt);
    if (plan->prefix_ctas + batch > 65535)
        return fail(PA_ERR_UNSUPPORTED, "batch %d plus %lld shared-prefix CTAs per kv head exceed 65535", batch,
                    (long long)plan->prefix_ctas);
    if (workspace_bytes < plan->ws_bytes)
        return fail(PA_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes,
                    plan->ws_bytes);
    return PA_OK;
}


// Checks of pa_store_kv's (or with scales pa_store_kv_fp8's) arguments; PA_OK or an error code.
int check_store(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride, const void *k_cache,
                const void *v_cache, const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                int32_t head_dim, int32_t num_blocks, int32_t block_size, pa_dtype dtype, const pa::Fp8Scales *fp8) {
    if (!valid_dtype(dtype)) return fail(PA_ERR_UNSUPPORTED, "dtype %d is not PA_F16 or PA_BF16", (int)dtype);
    if (fp8 && !valid_scales(*fp8))
        return fail(PA_ERR_INVALID_ARG, "k_scale and v_scale must be finite and positive (%g, %g)", fp8->k_scale,
                    fp8->v_scale);
    if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens is negative (%d)", num_tokens);
    if (num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 || block_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "sizes must be positive (H_kv=%d, D=%d, N=%d, bs=%d)", num_kv_heads,
                    head_dim, num_blocks, block_size);
    if (!k_cache || !v_cache) return fail(PA_ERR_INVALID_ARG, "k_cache/v_cache is NULL");
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping) return fail(PA_ERR_INVALID_ARG, "k, v or slot_mapping is NULL");
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (row > (1 << 30)) return fail(PA_ERR_INVALID_ARG, "row of %lld elements is too large", (long long)row);
    if (k_row_stride < row || v_row_stride < row)
        return fail(PA_ERR_INVALID_ARG, "row strides (%lld, %lld) are smaller than a row (%lld)",
                    (long long)k_row_stride, (long long)v_row_stride, (long long)row);
    if (!aligned(k, 2) || !aligned(v, 2) || !aligned(k_cache, 2) || !aligned(v_cache, 2))
        return fail(PA_ERR_INVALID_ARG, "buffers must be 2-byte aligned");
    if (fp8 && (row % 8 || k_row_stride % 8 || v_row_stride % 8 || !aligned(k, 16) || !aligned(v, 16) ||
                !aligned(k_cache, 8) || !aligned(v_cache, 8)))
        return fail(PA_ERR_INVALID_ARG,
                    "pa_store_kv_fp8: rows and strides must be multiples of 8 elements, k/v 16-byte and the "
                    "caches 8-byte aligned");
    return PA_OK;
}

// pa_store_kv, or pa_store_kv_fp8 when fp8 is given (an E4M3 pool).
int store_kv(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride, void *k_cache, void *v_cache,
             const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
             int32_t num_blocks, int32_t block_size, pa_dtype dtype, int32_t *err_flag, void *stream,
             const pa::Fp8Scales *fp8) {
    const int rc = check_store(k, v, k_row_stride, v_row_stride, k_cache, v_cache, slot_mapping, num_tokens,
                               num_kv_heads, head_dim, num_blocks, block_size, dtype, fp8);
    if (rc) return rc;
    if (num_tokens == 0) {
        g_err[0] = '\0';
        return PA_OK;
    }
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    const int64_t slots = static_cast<int64_t>(num_blocks) * block_size;
    if (fp8)
        return cuda_status(pa::launch_store_kv_fp8(k, v, k_row_stride, v_row_stride, k_cache, v_cache, slot_mapping,
                                                   num_tokens, static_cast<int32_t>(row), slots, dtype,
                                                   fp8->k_scale, fp8->v_scale, err_flag,
                                                   static_cast<cudaStream_t>(stream)),
                           "pa_store_kv_fp8 launch");
    return cuda_status(pa::launch_store_kv(k, v, k_row_stride, v_row_stride, k_cache, v_cache, slot_mapping,
                                           num_tokens, static_cast<int32_t>(row), slots, err_flag,
                                           static_cast<cudaStream_t>(stream)),
                       "pa_store_kv launch");
}


size_t decode_workspace(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t max_blocks_per_seq, int32_t block_size, bool fp8,
                        const pa_decode_options *opt = nullptr) {
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
        !is_pow2(block_size))
        return 0;
    if (check_options(opt)) return 0;
    return pa::plan_decode(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size, fp8, opt)
        .ws_bytes;
}

// pa_store_decode, or with scales pa_store_decode_fp8 (E4M3 pool).
int store_decode(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                 const int32_t *slot_mapping, const void *q, int64_t q_row_stride, void *k_cache, void *v_cache,
                 const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                 float scale, void *out, void *workspace, size_t workspace_bytes, pa_dtype dtype, int32_t *err_flag,
                 void *stream, const pa::Fp8Scales *fp8, const pa_decode_options *opt = nullptr) {
    pa::DecodePlan plan{};
    const int rc = check_decode(q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                batch, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, out,
                                workspace, workspace_bytes, dtype, &plan, fp8, opt);
    if (rc) return rc;
    if (batch == 0) {
        g_err[0] = '\0';
        return PA_OK;
    }
    if (!k || !v || !slot_mapping) return fail(PA_ERR_INVALID_ARG, "k, v and slot_mapping are required");
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (k_row_stride < row || v_row_stride < row || k_row_stride % 8 || v_row_stride % 8)
        return fail(PA_ERR_INVALID_ARG, "k/v row strides (%lld, %lld) must be multiples of 8 and at least H_kv*D",
                    (long long)k_row_stride, (long long)v_row_stride);
    if (!aligned(k, 16) || !aligned(v, 16)) return fail(PA_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
    const pa::FusedStore fused{k, v, k_row_stride, v_row_stride, slot_mapping};
    return cuda_status(pa::launch_decode(q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                         context_lens, batch, num_q_heads, num_kv_heads, head_dim, num_blocks,
                                         block_size, scale, out, workspace, plan, dtype, err_flag,
                                         static_cast<cudaStream_t>(stream), &fused, fp8, opt),
                       fp8 ? "pa_store_decode_fp8 launch" : "pa_store_decode launch");
}

}  // namespace

extern "C" {

const char *pa_last_error(void) { return g_err; }

int pa_version(void) { return 100; }

int pa_store_kv(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride, void *k_cache,
                void *v_cache, const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                int32_t head_dim, int32_t num_blocks, int32_t block_size, pa_dtype dtype, int32_t *err_flag,
                void *stream) {
    return store_kv(k, v, k_row_stride, v_row_stride, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads,
                    head_dim, num_blocks, block_size, dtype, err_flag, stream, nullptr);
}

int pa_store_kv_fp8(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride, void *k_cache,
                    void *v_cache, const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                    int32_t head_dim, int32_t num_blocks, int32_t block_size, pa_dtype dtype, float k_scale,
                    float v_scale, int32_t *err_flag, void *stream) {
    const pa::Fp8Scales sc{k_scale, v_scale};
    return store_kv(k, v, k_row_stride, v_row_stride, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads,
                    head_dim, num_blocks, block_size, dtype, err_flag, stream, &sc);
}

size_t pa_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t max_blocks_per_seq, int32_t block_size) {
    return decode_workspace(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size, false);
}

size_t pa_decode_fp8_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                     int32_t max_blocks_per_seq, int32_t block_size) {
    return decode_workspace(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size, true);
}

int pa_decode(const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
              float scale, void *out, void *workspace, size_t workspace_bytes, pa_dtype dtype, int32_t *err_flag,
              void *stream) {
    return pa_decode_ex(q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch,
                        num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, out, workspace,
                        workspace_bytes, nullptr, dtype, err_flag, stream);
}

size_t pa_decode_ex_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t max_blocks_per_seq, int32_t block_size,
                                    const pa_decode_options *options) {
    return decode_workspace(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size, false,
                            options);
}

int pa_decode_ex(const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache,
                 const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                 int32_t block_size, float scale, void *out, void *workspace, size_t workspace_bytes,
                 const pa_decode_options *options, pa_dtype dtype, int32_t *err_flag, void *stream) {
    pa::DecodePlan plan{};
    const int rc = check_decode(q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                batch, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, out,
                                workspace, workspace_bytes, dtype, &plan, nullptr, options);
    if (rc) return rc;
    if (batch == 0) {
        g_err[0] = '\0';
        return PA_OK;
    }
    return cuda_status(pa::launch_decode(q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                         context_lens, batch, num_q_heads, num_kv_heads, head_dim, num_blocks,
                                         block_size, scale, out, workspace, plan, dtype, err_flag,
                                         static_cast<cudaStream_t>(stream), nullptr, nullptr, options),
                       "pa_decode launch");
}

int pa_store_decode_ex(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                       const int32_t *slot_mapping, const void *q, int64_t q_row_stride, void *k_cache,
                       void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                       const int32_t *context_lens, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, void *out,
                       void *workspace, size_t workspace_bytes, const pa_decode_options *options, pa_dtype dtype,
                       int32_t *err_flag, void *stream) {
    return store_decode(k, v, k_row_stride, v_row_stride, slot_mapping, q, q_row_stride, k_cache, v_cache,
                        block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                        num_blocks, block_size, scale, out, workspace, workspace_bytes, dtype, err_flag, stream,
                        nullptr, options);
}

int pa_store_decode(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                    const int32_t *slot_mapping, const void *q, int64_t q_row_stride, void *k_cache, void *v_cache,
                    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                    int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                    int32_t block_size, float scale, void *out, void *workspace, size_t workspace_bytes,
                    pa_dtype dtype, int32_t *err_flag, void *stream) {
    return store_decode(k, v, k_row_stride, v_row_stride, slot_mapping, q, q_row_stride, k_cache, v_cache,
                        block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                        num_blocks, block_size, scale, out, workspace, workspace_bytes, dtype, err_flag, stream,
                        nullptr);
}

int pa_store_decode_fp8(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                        const int32_t *slot_mapping, const void *q, int64_t q_row_stride, void *k_cache,
                        void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                        const int32_t *context_lens, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, float k_scale,
                        float v_scale, void *out, void *workspace, size_t workspace_bytes, pa_dtype dtype,
                        int32_t *err_flag, void *stream) {
    const pa::Fp8Scales sc{k_scale, v_scale};
    return store_decode(k, v, k_row_stride, v_row_stride, slot_mapping, q, q_row_stride, k_cache, v_cache,
                        block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                        num_blocks, block_size, scale, out, workspace, workspace_bytes, dtype, err_flag, stream, &sc);
}

int pa_store_decode_fp8_ex(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                           const int32_t *slot_mapping, const void *q, int64_t q_row_stride, void *k_cache,
                           void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, float k_scale,
                           float v_scale, void *out, void *workspace, size_t workspace_bytes,
                           const pa_decode_options *options, pa_dtype dtype, int32_t *err_flag, void *stream) {
    // an E4M3 pool takes the operands alone: its plan (and so its workspace) has no overrides
    if (options && (options->partition || options->stages || options->num_groups || options->max_group_size ||
                    options->max_prefix_len || options->prefix_partition || options->group_offsets ||
                    options->group_seqs || options->prefix_lens))
        return fail(PA_ERR_INVALID_ARG, "pa_store_decode_fp8_ex takes options.operands only");
    const pa::Fp8Scales sc{k_scale, v_scale};
    return store_decode(k, v, k_row_stride, v_row_stride, slot_mapping, q, q_row_stride, k_cache, v_cache,
                        block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                        num_blocks, block_size, scale, out, workspace, workspace_bytes, dtype, err_flag, stream, &sc,
                        options);
}

int pa_decode_fp8(const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache,
                  const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                  int32_t block_size, float scale, float k_scale, float v_scale, void *out, void *workspace,
                  size_t workspace_bytes, pa_dtype dtype, int32_t *err_flag, void *stream) {
    pa::DecodePlan plan{};
    const pa::Fp8Scales sc{k_scale, v_scale};
    const int rc = check_decode(q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                batch, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, out,
                                workspace, workspace_bytes, dtype, &plan, &sc);
    if (rc) return rc;
    if (batch == 0) {
        g_err[0] = '\0';
        return PA_OK;
    }
    return cuda_status(pa::launch_decode(q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                         context_lens, batch, num_q_heads, num_kv_heads, head_dim, num_blocks,
                                         block_size, scale, out, workspace, plan, dtype, err_flag,
                                         static_cast<cudaStream_t>(stream), nullptr, &sc),
                       "pa_decode_fp8 launch");
}

}  // extern "C"

namespace {

// Checks of pa_prefill_paged's arguments; PA_OK or an error code (*work: something to compute).
int check_prefill(const void *q, const void *k, const void *v, const void *k_cache, const void *v_cache,
                  const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                  int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t *block_tables, int32_t max_blocks_per_seq,
                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                  float scale, const void *out, pa_dtype dtype, bool *work) {
    *work = false;
    int rc = check_attention_shape(num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, dtype);
    if (rc) return rc;
    if (!(scale > 0.f)) return fail(PA_ERR_INVALID_ARG, "pa_prefill_paged needs scale > 0 (got %g)", scale);
    if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < max_seqlen_q)
        return fail(PA_ERR_INVALID_ARG, "sizes: num_seqs %d, total_q %d, max_seqlen_q %d, max_seqlen_k %d", num_seqs,
                    total_q, max_seqlen_q, max_seqlen_k);
    if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return PA_OK;
    // work items: (sequence, 128-row q tile, query head pair), counted in 32-bit in the kernel
    if (static_cast<int64_t>(num_seqs) * ((max_seqlen_q + 127) / 128) * num_q_heads >= (1LL << 31))
        return fail(PA_ERR_INVALID_ARG, "num_seqs %d x max_seqlen_q %d x num_q_heads %d is too large", num_seqs,
                    max_seqlen_q, num_q_heads);
    if (!q || !k_cache || !v_cache || !cu_seqlens_q || !cu_seqlens_k || !out)
        return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!block_tables && (!k || !v)) return fail(PA_ERR_INVALID_ARG, "k and v are required without block_tables");
    if (block_tables && max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive with block_tables");
    if (block_tables && static_cast<int64_t>(max_blocks_per_seq) * block_size > (1LL << 30))
        return fail(PA_ERR_INVALID_ARG, "max context of %lld tokens is too large",
                    (long long)max_blocks_per_seq * block_size);
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        (!block_tables && (!aligned(k, 16) || !aligned(v, 16))))
        return fail(PA_ERR_INVALID_ARG, "q, k, v, caches and out must be 16-byte aligned");
    *work = true;
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_prefill_paged_ex(const void *q, const void *k, const void *v, const void *k_cache, const void *v_cache,
                        const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                        int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t *block_tables,
                        int32_t max_blocks_per_seq, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t num_blocks, int32_t block_size, float scale, void *out, pa_dtype dtype,
                        int32_t *err_flag, const pa_prefill_options *opt, void *stream) {
    const int32_t max_ctas = opt ? opt->max_ctas : 0;
    if (max_ctas < 0 || max_ctas > 65535)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_paged_ex: max_ctas %d is not in [0, 65535]", max_ctas);
    bool work = false;
    const int rc = check_prefill(q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q,
                                 max_seqlen_q, max_seqlen_k, block_tables, max_blocks_per_seq, num_q_heads,
                                 num_kv_heads, head_dim, num_blocks, block_size, scale, out, dtype, &work);
    if (rc) return rc;
    if (!work) {
        g_err[0] = '\0';
        return PA_OK;
    }
    const char *why = nullptr;
    const cudaError_t e = pa::launch_prefill(q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, num_seqs,
                                             total_q, max_seqlen_q, block_tables, max_blocks_per_seq, num_q_heads,
                                             num_kv_heads, head_dim, num_blocks, block_size, scale, out, dtype,
                                             err_flag, max_ctas, static_cast<cudaStream_t>(stream), &why);
    if (why) return fail(PA_ERR_CUDA, "pa_prefill_paged: %s", why);
    return cuda_status(e, "pa_prefill_paged launch");
}

int pa_prefill_paged(const void *q, const void *k, const void *v, const void *k_cache, const void *v_cache,
                     const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                     int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t *block_tables,
                     int32_t max_blocks_per_seq, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t num_blocks, int32_t block_size, float scale, void *out, pa_dtype dtype,
                     int32_t *err_flag, void *stream) {
    return pa_prefill_paged_ex(q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q,
                               max_seqlen_q, max_seqlen_k, block_tables, max_blocks_per_seq, num_q_heads,
                               num_kv_heads, head_dim, num_blocks, block_size, scale, out, dtype, err_flag, nullptr,
                               stream);
}

int pa_copy_segments(const pa_copy_segment *segments, int32_t count, void *stream) {
    if (count < 0 || count > 64 || (count > 0 && !segments))
        return fail(PA_ERR_INVALID_ARG, "pa_copy_segments: count %d (0..64) with a segment list", count);
    if (count == 0) {
        g_err[0] = '\0';
        return PA_OK;
    }
    static int sms[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (!sms[dev] && (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                      sms[dev] <= 0))
        sms[dev] = 148;
    return cuda_status(pa::launch_copy_segments(segments, count, 2 * sms[dev], static_cast<cudaStream_t>(stream)),
                       "pa_copy_segments launch");
}

int pa_sample(const void *logits, int64_t logits_row_stride, int32_t batch, int32_t vocab, pa_dtype dtype,
              const float *temperatures, const float *noise, uint64_t seed, uint64_t offset, int32_t *tokens,
              int32_t *err_flag, void *stream) {
    if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_F16)
        return fail(PA_ERR_UNSUPPORTED, "logits dtype %d is not PA_F32, PA_BF16 or PA_F16", (int)dtype);
    if (batch < 0 || batch > 65535 || vocab <= 0)
        return fail(PA_ERR_INVALID_ARG, "batch %d (at most 65535), vocab %d", batch, vocab);
    if (batch == 0) {
        g_err[0] = '\0';
        return PA_OK;
    }
    if (!logits || !temperatures || !tokens) return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (logits_row_stride < vocab)
        return fail(PA_ERR_INVALID_ARG, "logits_row_stride %lld is shorter than vocab", (long long)logits_row_stride);
    if (!aligned(logits, dtype == PA_F32 ? 4 : 2) || (noise && !aligned(noise, 4)))
        return fail(PA_ERR_INVALID_ARG, "logits and noise must be aligned to their element size");
    return cuda_status(pa::launch_sample(logits, logits_row_stride, batch, vocab, dtype, temperatures, noise, seed,
                                         offset, tokens, err_flag, static_cast<cudaStream_t>(stream)),
                       "pa_sample launch");
}

int pa_mixed_step(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                  const int32_t *slot_mapping, int32_t num_tokens, const void *prefill_q, const int32_t *cu_seqlens_q,
                  const int32_t *cu_seqlens_k, int32_t num_prefill_seqs, int32_t total_prefill_q,
                  int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t *prefill_block_tables,
                  int32_t prefill_max_blocks, void *prefill_out, const void *decode_q, int64_t decode_q_row_stride,
                  const int32_t *decode_block_tables, int32_t decode_max_blocks, const int32_t *context_lens,
                  int32_t decode_batch, void *decode_out, void *workspace, size_t workspace_bytes, void *k_cache,
                  void *v_cache, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                  int32_t block_size, float scale, pa_dtype dtype, int32_t *err_flag, const pa_sm_split *split,
                  void *stream) {
    // every check first: nothing is launched unless all three parts are valid
    int rc = check_store(k, v, k_row_stride, v_row_stride, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads,
                         head_dim, num_blocks, block_size, dtype, nullptr);
    if (rc) return rc;
    bool prefill = false;
    if (num_prefill_seqs != 0) {
        if (!prefill_block_tables)
            return fail(PA_ERR_INVALID_ARG, "pa_mixed_step: the prefill reads its keys through prefill_block_tables");
        rc = check_prefill(prefill_q, nullptr, nullptr, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k,
                           num_prefill_seqs, total_prefill_q, max_seqlen_q, max_seqlen_k, prefill_block_tables,
                           prefill_max_blocks, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale,
                           prefill_out, dtype, &prefill);
        if (rc) return rc;
    }
    pa::DecodePlan plan{};
    if (decode_batch != 0) {
        rc = check_decode(decode_q, decode_q_row_stride, k_cache, v_cache, decode_block_tables, decode_max_blocks,
                          context_lens, decode_batch, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                          scale, decode_out, workspace, workspace_bytes, dtype, &plan);
        if (rc) return rc;
    }
    const bool decode = decode_batch > 0;
    if (split) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev != pa::split_device(split))
            return fail(PA_ERR_INVALID_ARG, "pa_mixed_step: the split belongs to device %d, not the current one",
                        pa::split_device(split));
    }
    const cudaStream_t main = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (num_tokens > 0)
        e = pa::launch_store_kv(k, v, k_row_stride, v_row_stride, k_cache, v_cache, slot_mapping, num_tokens,
                                num_kv_heads * head_dim, static_cast<int64_t>(num_blocks) * block_size, err_flag,
                                main);
    const bool both = split && prefill && decode;
    if (e == cudaSuccess && both) e = pa::split_fork(split, main);
    const cudaStream_t s_prefill = both ? pa::split_stream(split, 0) : main;
    const cudaStream_t s_decode = both ? pa::split_stream(split, 1) : main;
    if (e == cudaSuccess && prefill) {
        const char *why = nullptr;
        e = pa::launch_prefill(prefill_q, nullptr, nullptr, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k,
                               num_prefill_seqs, total_prefill_q, max_seqlen_q, prefill_block_tables,
                               prefill_max_blocks, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale,
                               prefill_out, dtype, err_flag, both ? pa::split_sms(split, 0) : 0, s_prefill, &why);
        if (why) return fail(PA_ERR_CUDA, "pa_mixed_step: %s", why);
    }
    if (e == cudaSuccess && decode)
        e = pa::launch_decode(decode_q, decode_q_row_stride, k_cache, v_cache, decode_block_tables, decode_max_blocks,
                              context_lens, decode_batch, num_q_heads, num_kv_heads, head_dim, num_blocks,
                              block_size, scale, decode_out, workspace, plan, dtype, err_flag, s_decode);
    if (e == cudaSuccess && both) e = pa::split_join(split, main);
    return cuda_status(e, "pa_mixed_step launch");
}

}  // extern "C"
