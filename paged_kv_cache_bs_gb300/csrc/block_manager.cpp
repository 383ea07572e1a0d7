// Host-side page directory of the paged KV cache (prefix-cached block
// allocation), behind the C ABI of pa_block_manager.h.  The rules are the
// BlockManager's of "Inference engine: inside nano-vLLM" and "nano-vLLM
// Part 2: Block Tables, KV Cache, and the Path to the GPU" (sections 2-3);
// the header lists them.  Plain C++, no GPU.
#include <stdio.h>

#include <algorithm>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_block_manager.h"

namespace pa {
int set_last_error(int code, const char *msg);
}

namespace {

int fail(int code, const char *fmt, long long a = 0, long long b = 0) {
    char msg[256];
    snprintf(msg, sizeof msg, fmt, a, b);
    return pa::set_last_error(code, msg);
}

// 64-bit FNV-1a (Fowler, Noll, Vo): offset basis and prime of the published definition.
struct Fnv1a64 {
    uint64_t h = 14695981039346656037ull;
    void byte(uint8_t b) {
        h ^= b;
        h *= 1099511628211ull;
    }
    void u64(uint64_t v) {
        for (int i = 0; i < 8; ++i) byte(static_cast<uint8_t>(v >> (8 * i)));
    }
    void u32(uint32_t v) {
        for (int i = 0; i < 4; ++i) byte(static_cast<uint8_t>(v >> (8 * i)));
    }
};

// Chained block hash: the previous full block's hash (if any), then the token ids.
uint64_t block_hash(const int32_t *tokens, int32_t n, bool has_prev, uint64_t prev) {
    Fnv1a64 f;
    if (has_prev) f.u64(prev);
    for (int32_t i = 0; i < n; ++i) f.u32(static_cast<uint32_t>(tokens[i]));
    return f.h;
}

struct Block {
    int32_t ref_count = 0;
    bool hashed = false;
    uint64_t hash = 0;
    std::vector<int32_t> tokens;  // the block's token ids, saved when it is hashed
};

struct Sequence {
    std::vector<int32_t> tokens;
    std::vector<int32_t> block_table;
    int64_t num_cached_tokens = 0;
};

}  // namespace

struct pa_bm {
    int32_t bs;
    std::vector<Block> blocks;
    std::deque<int32_t> free_ids;  // taken from the front, returned to the back
    std::vector<char> used;        // used[b]: referenced by a live sequence
    std::unordered_map<uint64_t, int32_t> hash_to_block;
    std::unordered_map<int64_t, Sequence> seqs;

    int32_t num_logical_blocks(const Sequence &s) const {
        return static_cast<int32_t>((s.tokens.size() + bs - 1) / bs);
    }
    // tokens of logical block i of s (a full block unless it is the last one)
    const int32_t *block_tokens(const Sequence &s, int32_t i, int32_t *n) const {
        const size_t b = static_cast<size_t>(i) * bs;
        *n = static_cast<int32_t>(std::min<size_t>(bs, s.tokens.size() - b));
        return s.tokens.data() + b;
    }
    // the registered block holding exactly these tokens under this hash, or -1
    int32_t lookup(uint64_t h, const int32_t *tok, int32_t n) const {
        const auto it = hash_to_block.find(h);
        if (it == hash_to_block.end()) return -1;
        const Block &blk = blocks[it->second];
        if (static_cast<int32_t>(blk.tokens.size()) != n || !std::equal(tok, tok + n, blk.tokens.begin())) return -1;
        return it->second;
    }
    int32_t take_fresh_block() {
        const int32_t id = free_ids.front();
        free_ids.pop_front();
        Block &blk = blocks[id];
        if (blk.hashed) {  // repurposed for new content: its old prefix entry goes
            const auto it = hash_to_block.find(blk.hash);
            if (it != hash_to_block.end() && it->second == id) hash_to_block.erase(it);
        }
        blk.hashed = false;
        blk.tokens.clear();
        blk.ref_count = 1;
        used[id] = 1;
        return id;
    }
    void release(Sequence &s) {
        for (auto it = s.block_table.rbegin(); it != s.block_table.rend(); ++it) {
            Block &blk = blocks[*it];
            if (--blk.ref_count == 0) {
                used[*it] = 0;
                free_ids.push_back(*it);
            }
        }
        s.block_table.clear();
        s.num_cached_tokens = 0;
    }
};

namespace {

Sequence *find(pa_bm *bm, int64_t id) {
    if (!bm) return nullptr;
    const auto it = bm->seqs.find(id);
    return it == bm->seqs.end() ? nullptr : &it->second;
}
const Sequence *find(const pa_bm *bm, int64_t id) {
    if (!bm) return nullptr;
    const auto it = bm->seqs.find(id);
    return it == bm->seqs.end() ? nullptr : &it->second;
}
// Leading entries equal in rows a and b, at most n: 8-entry blocks compared whole first (an OR
// of XORs, which the compiler turns into vector code), then entry by entry.
int32_t common_prefix(const int32_t *a, const int32_t *b, int32_t n) {
    int32_t k = 0;
    for (; k + 8 <= n; k += 8) {
        uint32_t diff = 0;
        for (int j = 0; j < 8; ++j) diff |= static_cast<uint32_t>(a[k + j] ^ b[k + j]);
        if (diff) break;
    }
    while (k < n && a[k] == b[k]) ++k;
    return k;
}

// Open-addressing map from a page id to an int32 value (-1: absent), linear probing over a
// power-of-two table at most half full.  A slot belongs to the current call when its stamp is
// the call's generation, so starting a call clears nothing.
class PageSlots {
  public:
    void reset(int32_t max_keys) {
        size_t cap = 16;
        int bits = 4;
        while (cap < 2 * static_cast<size_t>(max_keys)) cap <<= 1, ++bits;
        if (cap > keys_.size()) {
            bits_ = bits;
            keys_.assign(cap, 0);
            vals_.assign(cap, -1);
            stamps_.assign(cap, 0);
            gen_ = 0;
        }
        if (++gen_ == 0) {  // the stamps wrapped: clear them once
            std::fill(stamps_.begin(), stamps_.end(), 0u);
            gen_ = 1;
        }
    }
    int32_t &find_or_add(int32_t key) {
        const size_t mask = keys_.size() - 1;
        // multiplicative hashing (Knuth): the top bits of the id times 2^32 / golden ratio
        size_t i = (static_cast<uint32_t>(key) * 2654435769u) >> (32 - bits_);
        while (stamps_[i] == gen_ && keys_[i] != key) i = (i + 1) & mask;
        if (stamps_[i] != gen_) {
            stamps_[i] = gen_;
            keys_[i] = key;
            vals_[i] = -1;
        }
        return vals_[i];
    }

  private:
    std::vector<int32_t> keys_, vals_;
    std::vector<uint32_t> stamps_;
    uint32_t gen_ = 0;
    int bits_ = 0;
};

int no_seq(int64_t id) { return fail(PA_ERR_INVALID_ARG, "no sequence %lld in this block manager", id); }

}  // namespace

extern "C" {

pa_bm *pa_bm_create(int32_t num_blocks, int32_t block_size) {
    if (num_blocks <= 0 || block_size <= 0) {
        fail(PA_ERR_INVALID_ARG, "num_blocks %lld and block_size %lld must be positive", num_blocks, block_size);
        return nullptr;
    }
    pa_bm *bm = new (std::nothrow) pa_bm;
    if (!bm) return nullptr;
    bm->bs = block_size;
    bm->blocks.resize(num_blocks);
    bm->used.assign(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) bm->free_ids.push_back(i);
    return bm;
}

void pa_bm_destroy(pa_bm *bm) { delete bm; }

int pa_bm_add_sequence(pa_bm *bm, int64_t seq_id, const int32_t *token_ids, int32_t n) {
    if (!bm || !token_ids || n <= 0) return fail(PA_ERR_INVALID_ARG, "a sequence needs at least one token");
    if (bm->seqs.count(seq_id)) return fail(PA_ERR_INVALID_ARG, "sequence %lld already exists", seq_id);
    Sequence s;
    s.tokens.assign(token_ids, token_ids + n);
    bm->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
}

int pa_bm_append_token(pa_bm *bm, int64_t seq_id, int32_t token_id) {
    Sequence *s = find(bm, seq_id);
    if (!s) return no_seq(seq_id);
    s->tokens.push_back(token_id);
    return PA_OK;
}

int pa_bm_remove_sequence(pa_bm *bm, int64_t seq_id) {
    Sequence *s = find(bm, seq_id);
    if (!s) return no_seq(seq_id);
    bm->release(*s);
    bm->seqs.erase(seq_id);
    return PA_OK;
}

int pa_bm_can_allocate(pa_bm *bm, int64_t seq_id, int32_t *num_cached_blocks) {
    Sequence *s = find(bm, seq_id);
    if (!s) return no_seq(seq_id);
    if (!num_cached_blocks) return fail(PA_ERR_INVALID_ARG, "num_cached_blocks is NULL");
    if (!s->block_table.empty()) return fail(PA_ERR_INVALID_ARG, "sequence %lld already holds blocks", seq_id);
    const int32_t nb = bm->num_logical_blocks(*s);
    int32_t hits = 0, need = nb;
    bool has = false;
    uint64_t h = 0;
    for (int32_t i = 0; i + 1 < nb; ++i) {  // never the last logical block
        int32_t n;
        const int32_t *tok = bm->block_tokens(*s, i, &n);
        h = block_hash(tok, n, has, h);
        has = true;
        const int32_t id = bm->lookup(h, tok, n);
        if (id < 0) break;
        ++hits;
        if (bm->used[id]) --need;  // shared with a live sequence: no free block consumed
    }
    *num_cached_blocks = static_cast<int32_t>(bm->free_ids.size()) < need ? -1 : hits;
    return PA_OK;
}

int pa_bm_allocate(pa_bm *bm, int64_t seq_id, int32_t num_cached_blocks) {
    Sequence *s = find(bm, seq_id);
    if (!s) return no_seq(seq_id);
    const int32_t nb = bm->num_logical_blocks(*s);
    if (!s->block_table.empty()) return fail(PA_ERR_INVALID_ARG, "sequence %lld already holds blocks", seq_id);
    if (num_cached_blocks < 0 || num_cached_blocks > nb - 1)
        return fail(PA_ERR_INVALID_ARG, "num_cached_blocks %lld out of range for %lld blocks", num_cached_blocks, nb);
    // check before changing anything: the hits are still registered and enough blocks are free
    {
        bool has = false;
        uint64_t h = 0;
        int32_t need = nb;
        for (int32_t i = 0; i < num_cached_blocks; ++i) {
            int32_t n;
            const int32_t *tok = bm->block_tokens(*s, i, &n);
            h = block_hash(tok, n, has, h);
            has = true;
            const int32_t id = bm->lookup(h, tok, n);
            if (id < 0) return fail(PA_ERR_INVALID_ARG, "block %lld of sequence %lld is not cached", i, seq_id);
            if (bm->used[id]) --need;
        }
        if (static_cast<int32_t>(bm->free_ids.size()) < need)
            return fail(PA_ERR_INVALID_ARG, "%lld free blocks, %lld needed", (long long)bm->free_ids.size(), need);
    }
    bool has = false;
    uint64_t h = 0;
    for (int32_t i = 0; i < num_cached_blocks; ++i) {
        int32_t n;
        const int32_t *tok = bm->block_tokens(*s, i, &n);
        h = block_hash(tok, n, has, h);
        has = true;
        const int32_t id = bm->lookup(h, tok, n);
        Block &blk = bm->blocks[id];
        if (bm->used[id]) {
            ++blk.ref_count;
        } else {  // a freed block whose contents are still valid: revive it
            blk.ref_count = 1;
            bm->free_ids.erase(std::find(bm->free_ids.begin(), bm->free_ids.end(), id));
            bm->used[id] = 1;
        }
        s->block_table.push_back(id);
    }
    for (int32_t i = num_cached_blocks; i < nb; ++i) s->block_table.push_back(bm->take_fresh_block());
    s->num_cached_tokens = static_cast<int64_t>(num_cached_blocks) * bm->bs;
    return PA_OK;
}

int pa_bm_deallocate(pa_bm *bm, int64_t seq_id) {
    Sequence *s = find(bm, seq_id);
    if (!s) return no_seq(seq_id);
    bm->release(*s);
    return PA_OK;
}

int pa_bm_can_append(pa_bm *bm, int64_t seq_id) {
    Sequence *s = find(bm, seq_id);
    if (!s) return no_seq(seq_id);
    const int32_t need = ((s->tokens.size() - 1) % bm->bs) == 0 ? 1 : 0;  // the last token starts a page
    return static_cast<int32_t>(bm->free_ids.size()) >= need ? 1 : 0;
}

int pa_bm_may_append(pa_bm *bm, int64_t seq_id) {
    Sequence *s = find(bm, seq_id);
    if (!s) return no_seq(seq_id);
    if (s->block_table.empty()) return fail(PA_ERR_INVALID_ARG, "sequence %lld holds no blocks", seq_id);
    if (((s->tokens.size() - 1) % bm->bs) == 0) {  // length 1 mod block_size: the last token starts a page
        if (bm->free_ids.empty()) return fail(PA_ERR_INVALID_ARG, "no free block for sequence %lld", seq_id);
        s->block_table.push_back(bm->take_fresh_block());
    }
    return PA_OK;
}

int pa_bm_postprocess(pa_bm *bm, int64_t seq_id, int32_t num_scheduled_tokens) {
    Sequence *s = find(bm, seq_id);
    if (!s) return no_seq(seq_id);
    const int64_t done = s->num_cached_tokens + num_scheduled_tokens;
    if (num_scheduled_tokens < 0 || done > static_cast<int64_t>(s->tokens.size()) ||
        (done + bm->bs - 1) / bm->bs > static_cast<int64_t>(s->block_table.size()))
        return fail(PA_ERR_INVALID_ARG, "sequence %lld cannot have processed %lld more tokens", seq_id,
                    num_scheduled_tokens);
    const int64_t start = s->num_cached_tokens / bm->bs, end = done / bm->bs;
    if (start < end) {
        bool has = start > 0;
        uint64_t h = has ? bm->blocks[s->block_table[start - 1]].hash : 0;
        for (int64_t i = start; i < end; ++i) {
            int32_t n;
            const int32_t *tok = bm->block_tokens(*s, static_cast<int32_t>(i), &n);
            h = block_hash(tok, n, has, h);
            has = true;
            const int32_t id = s->block_table[i];
            Block &blk = bm->blocks[id];
            blk.hashed = true;
            blk.hash = h;
            blk.tokens.assign(tok, tok + n);
            bm->hash_to_block[h] = id;
        }
    }
    s->num_cached_tokens = done;
    return PA_OK;
}

int pa_bm_num_free_blocks(const pa_bm *bm) {
    return bm ? static_cast<int32_t>(bm->free_ids.size()) : fail(PA_ERR_INVALID_ARG, "null block manager");
}

int pa_bm_ref_count(const pa_bm *bm, int32_t block_id) {
    if (!bm || block_id < 0 || block_id >= static_cast<int32_t>(bm->blocks.size()))
        return fail(PA_ERR_INVALID_ARG, "no block %lld", block_id);
    return bm->blocks[block_id].ref_count;
}

int pa_bm_block_table(const pa_bm *bm, int64_t seq_id, int32_t *out, int32_t cap) {
    const Sequence *s = find(bm, seq_id);
    if (!s) return no_seq(seq_id);
    const int32_t n = static_cast<int32_t>(s->block_table.size());
    for (int32_t i = 0; i < n && i < cap && out; ++i) out[i] = s->block_table[i];
    return n;
}

int64_t pa_bm_seq_len(const pa_bm *bm, int64_t seq_id) {
    const Sequence *s = find(bm, seq_id);
    return s ? static_cast<int64_t>(s->tokens.size()) : no_seq(seq_id);
}

int64_t pa_bm_num_cached_tokens(const pa_bm *bm, int64_t seq_id) {
    const Sequence *s = find(bm, seq_id);
    return s ? s->num_cached_tokens : no_seq(seq_id);
}

int pa_bm_decode_inputs(const pa_bm *bm, const int64_t *seq_ids, int32_t n, int32_t max_blocks,
                        int32_t *slot_mapping, int32_t *context_lens, int32_t *block_tables) {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !slot_mapping || !context_lens || !block_tables)) || max_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "bad decode-input arguments");
    for (int32_t i = 0; i < n; ++i) {
        const Sequence *s = find(bm, seq_ids[i]);
        if (!s) return no_seq(seq_ids[i]);
        const int64_t len = static_cast<int64_t>(s->tokens.size());
        const int32_t nb = static_cast<int32_t>(s->block_table.size());
        if (nb > max_blocks) return fail(PA_ERR_INVALID_ARG, "block table of %lld entries, room for %lld", nb, max_blocks);
        if ((len + bm->bs - 1) / bm->bs > nb)
            return fail(PA_ERR_INVALID_ARG, "sequence %lld needs a block (call may_append first)", seq_ids[i]);
        slot_mapping[i] = s->block_table[(len - 1) / bm->bs] * bm->bs + static_cast<int32_t>((len - 1) % bm->bs);
        context_lens[i] = static_cast<int32_t>(len);
        for (int32_t j = 0; j < max_blocks; ++j)
            block_tables[static_cast<int64_t>(i) * max_blocks + j] = j < nb ? s->block_table[j] : -1;
    }
    return PA_OK;
}

int pa_bm_prefill_inputs(const pa_bm *bm, const int64_t *seq_ids, const int32_t *num_scheduled, int32_t n,
                         int32_t max_blocks, int32_t *slot_mapping, int32_t *cu_seqlens_q, int32_t *cu_seqlens_k,
                         int32_t *block_tables) {
    if (!bm || n < 0 || !cu_seqlens_q || !cu_seqlens_k || max_blocks <= 0 ||
        (n > 0 && (!seq_ids || !num_scheduled || !slot_mapping || !block_tables)))
        return fail(PA_ERR_INVALID_ARG, "bad prefill-input arguments");
    const int32_t bs = bm->bs;
    int64_t t = 0;
    cu_seqlens_q[0] = cu_seqlens_k[0] = 0;
    for (int32_t i = 0; i < n; ++i) {
        const Sequence *s = find(bm, seq_ids[i]);
        if (!s) return no_seq(seq_ids[i]);
        const int64_t start = s->num_cached_tokens, end = start + num_scheduled[i];
        const int32_t nb = static_cast<int32_t>(s->block_table.size());
        if (num_scheduled[i] <= 0 || end > static_cast<int64_t>(s->tokens.size()) || (end + bs - 1) / bs > nb)
            return fail(PA_ERR_INVALID_ARG, "sequence %lld cannot process %lld tokens", seq_ids[i], num_scheduled[i]);
        if (nb > max_blocks) return fail(PA_ERR_INVALID_ARG, "block table of %lld entries, room for %lld", nb, max_blocks);
        // the slots of positions [start, end), page by page
        const int64_t first = start / bs, last = (end + bs - 1) / bs;
        for (int64_t pg = first; pg < last; ++pg) {
            const int64_t base = static_cast<int64_t>(s->block_table[pg]) * bs;
            const int64_t lo = pg == first ? start % bs : 0;
            const int64_t hi = pg == last - 1 ? end - pg * bs : bs;
            for (int64_t o = lo; o < hi; ++o) slot_mapping[t++] = static_cast<int32_t>(base + o);
        }
        cu_seqlens_q[i + 1] = cu_seqlens_q[i] + num_scheduled[i];
        cu_seqlens_k[i + 1] = cu_seqlens_k[i] + static_cast<int32_t>(end);
        for (int32_t j = 0; j < max_blocks; ++j)
            block_tables[static_cast<int64_t>(i) * max_blocks + j] = j < nb ? s->block_table[j] : -1;
    }
    return PA_OK;
}

int pa_prefix_groups(const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens, int32_t batch,
                     int32_t block_size, int32_t min_shared_pages, int32_t *group_offsets, int32_t *group_seqs,
                     int32_t *prefix_lens, int32_t *num_groups, int32_t *max_group_size, int32_t *max_prefix_len) {
    if (batch < 0 || max_blocks <= 0 || block_size <= 0 || !group_offsets || !num_groups || !max_group_size ||
        !max_prefix_len || (batch > 0 && (!block_tables || !context_lens || !group_seqs || !prefix_lens)))
        return fail(PA_ERR_INVALID_ARG, "bad prefix-group arguments");
    const int64_t cap_tokens = static_cast<int64_t>(max_blocks) * block_size;
    for (int32_t b = 0; b < batch; ++b)
        if (context_lens[b] < 0 || context_lens[b] > cap_tokens)
            return fail(PA_ERR_INVALID_ARG, "context length %lld of sequence %lld is outside the table",
                        context_lens[b], b);
    const int32_t min_pages = min_shared_pages > 1 ? min_shared_pages : 1;
    // candidates keyed by the first page of their table, groups in order of first appearance,
    // members in batch order (a counting sort); the buffers are reused from call to call
    thread_local PageSlots slot_of_page;
    thread_local std::vector<int32_t> cand_of, pages_of, count, first, members_of;
    slot_of_page.reset(batch);
    cand_of.assign(static_cast<size_t>(batch), -1);
    pages_of.resize(static_cast<size_t>(batch));
    count.clear();
    const bool pow2 = (block_size & (block_size - 1)) == 0;
    const int shift = pow2 ? __builtin_ctz(static_cast<unsigned>(block_size)) : 0;
    int32_t eligible = 0;
    for (int32_t b = 0; b < batch; ++b) {
        const int32_t len = context_lens[b];
        if (len <= 0) continue;
        // pages before the newest token's page
        const int32_t complete = pow2 ? (len - 1) >> shift : (len - 1) / block_size;
        if (complete < 1) continue;
        pages_of[b] = complete;
        int32_t &c = slot_of_page.find_or_add(block_tables[static_cast<int64_t>(b) * max_blocks]);
        if (c < 0) {
            c = static_cast<int32_t>(count.size());
            count.push_back(0);
        }
        cand_of[b] = c;
        ++count[c];
        ++eligible;
    }
    const int32_t ncand = static_cast<int32_t>(count.size());
    first.assign(static_cast<size_t>(ncand) + 1, 0);
    for (int32_t c = 0; c < ncand; ++c) first[c + 1] = first[c] + count[c];
    members_of.resize(static_cast<size_t>(eligible));
    for (int32_t c = 0; c < ncand; ++c) count[c] = first[c];  // next free position of candidate c
    for (int32_t b = 0; b < batch; ++b)
        if (cand_of[b] >= 0) members_of[count[cand_of[b]]++] = b;
    for (int32_t b = 0; b < batch; ++b) prefix_lens[b] = 0;
    int32_t groups = 0, members = 0, largest = 0, longest = 0;
    group_offsets[0] = 0;
    for (int32_t c = 0; c < ncand; ++c) {
        const int32_t *m = members_of.data() + first[c];
        const int32_t size = first[c + 1] - first[c];
        if (size < 2) continue;
        int32_t n = INT32_MAX;  // leading table entries equal across the members, within every cap
        for (int32_t i = 0; i < size; ++i) n = std::min(n, pages_of[m[i]]);
        const int32_t *lead = block_tables + static_cast<int64_t>(m[0]) * max_blocks;
        for (int32_t i = 1; i < size && n > 0; ++i)
            n = common_prefix(lead, block_tables + static_cast<int64_t>(m[i]) * max_blocks, n);
        if (n < min_pages) continue;
        for (int32_t i = 0; i < size; ++i) {
            group_seqs[members++] = m[i];
            prefix_lens[m[i]] = n * block_size;
        }
        group_offsets[++groups] = members;
        largest = std::max(largest, size);
        longest = std::max(longest, n * block_size);
    }
    *num_groups = groups;
    *max_group_size = largest;
    *max_prefix_len = longest;
    return PA_OK;
}

}  // extern "C"
