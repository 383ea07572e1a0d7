// pa_stage_decode_step: the host half of a captured decode step, behind the C
// ABI of pa_api.h.  "nano-vLLM Part 2: Block Tables, KV Cache, and the Path to
// the GPU", section 4.2: a decode step writes its slot mapping, context
// lengths and block tables into the fixed buffers of the graph recorded for
// its padded batch size and pads the rows past the batch.  Doing that, the
// shared-prefix grouping and the addresses of the caller's buffers (a gather
// list, or the decode's operands array) in one call keeps a step's host work to
// plain memory copies.  Plain C++, no GPU.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "pa_api.h"
#include "pa_block_manager.h"

namespace pa {
int set_last_error(int code, const char *msg);
}

namespace {

int fail(const char *fmt, long long a = 0, long long b = 0, long long c = 0) {
    char msg[256];
    snprintf(msg, sizeof msg, fmt, a, b, c);
    return pa::set_last_error(PA_ERR_INVALID_ARG, msg);
}

void fill(int32_t *p, int64_t n, int32_t v) {
    for (int64_t i = 0; i < n; ++i) p[i] = v;
}

}  // namespace

extern "C" {

int pa_stage_decode_step(const pa_decode_staging *st, int32_t batch, const int32_t *slot_mapping,
                         const int32_t *context_lens, const int32_t *block_tables, int32_t table_cols,
                         int32_t groups, const void *const *sources) {
    if (!st || st->rows <= 0 || st->max_blocks <= 0 || st->block_size <= 0 || !st->slot_mapping ||
        !st->context_lens || !st->block_tables)
        return fail("bad decode staging");
    if (batch < 0 || batch > st->rows) return fail("batch %lld outside [0, %lld]", batch, st->rows);
    if (batch > 0 && (!slot_mapping || !context_lens || !block_tables))
        return fail("a step of %lld sequences needs its slot mapping, context lengths and block tables", batch);
    if (batch > 0 && (table_cols < 1 || table_cols > st->max_blocks))
        return fail("table_cols %lld outside [1, %lld]", table_cols, st->max_blocks);
    const bool has_groups = st->group_offsets && st->group_seqs && st->prefix_lens && st->max_groups > 0 &&
                            st->max_group_size > 0 && st->max_prefix_len > 0;
    if (groups != PA_STAGE_NO_GROUPS && groups != PA_STAGE_DERIVE_GROUPS && groups != PA_STAGE_KEEP_GROUPS)
        return fail("unknown groups mode %lld", groups);
    if (groups == PA_STAGE_DERIVE_GROUPS && !has_groups) return fail("this staging holds no shared-prefix groups");
    if (sources && !st->operands && !st->segments)
        return fail("this staging holds neither a gather list nor an operands array");
    if (sources && st->segments && (st->num_segments < 0 || st->num_segments > 4))
        return fail("num_segments %lld outside [0, 4]", st->num_segments);
    const int64_t cap = static_cast<int64_t>(table_cols) * st->block_size;
    for (int32_t b = 0; b < batch; ++b)
        if (context_lens[b] < 0 || context_lens[b] > cap)
            return fail("context length %lld of sequence %lld is outside its %lld-token table", context_lens[b], b,
                        cap);

    const int32_t pad = st->rows - batch;
    memcpy(st->slot_mapping, slot_mapping, sizeof(int32_t) * batch);
    fill(st->slot_mapping + batch, pad, -1);
    memcpy(st->context_lens, context_lens, sizeof(int32_t) * batch);
    fill(st->context_lens + batch, pad, 0);
    if (table_cols == st->max_blocks) {
        memcpy(st->block_tables, block_tables, sizeof(int32_t) * batch * static_cast<size_t>(table_cols));
    } else {
        for (int32_t b = 0; b < batch; ++b) {
            int32_t *row = st->block_tables + static_cast<int64_t>(b) * st->max_blocks;
            memcpy(row, block_tables + static_cast<int64_t>(b) * table_cols, sizeof(int32_t) * table_cols);
            fill(row + table_cols, st->max_blocks - table_cols, -1);
        }
    }

    if (has_groups && groups == PA_STAGE_NO_GROUPS) {
        fill(st->group_offsets, st->max_groups + 1, 0);
        fill(st->prefix_lens, st->rows, 0);
    } else if (groups == PA_STAGE_DERIVE_GROUPS) {
        // the derived offsets may outnumber the captured groups: counted in a scratch first
        thread_local std::vector<int32_t> offsets;
        offsets.resize(static_cast<size_t>(batch) / 2 + 1);
        int32_t n = 0, largest = 0, longest = 0;
        const int rc = pa_prefix_groups(st->block_tables, st->max_blocks, st->context_lens, batch, st->block_size, 1,
                                        offsets.data(), st->group_seqs, st->prefix_lens, &n, &largest, &longest);
        if (rc != PA_OK) return rc;
        if (n > st->max_groups || largest > st->max_group_size || longest > st->max_prefix_len)
            return fail("the step's groups (%lld groups, %lld members, %lld prefix tokens) exceed the captured "
                        "capacities",
                        n, largest, longest);
        memcpy(st->group_offsets, offsets.data(), sizeof(int32_t) * (n + 1));
        fill(st->group_offsets + n + 1, st->max_groups - n, offsets[n]);
        fill(st->prefix_lens + batch, pad, 0);
    }

    if (sources && st->segments) {
        for (int32_t i = 0; i < st->num_segments; ++i) {
            st->segments[i].src = sources[i];
            st->segments[i].bytes = static_cast<uint64_t>(batch) * st->segment_row_bytes[i];
        }
    }
    if (sources && st->operands)
        for (int i = 0; i < 3; ++i) st->operands[i] = sources[i];
    return PA_OK;
}

}  // extern "C"
