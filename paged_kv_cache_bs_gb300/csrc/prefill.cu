// Chunked prefill over a paged prefix on the 5th-generation tensor cores.
//
// What is computed is the prefill branch of the attention layer in
// "Inference engine: inside nano-vLLM" (flash_attn_varlen_func with
// cu_seqlens_q / cu_seqlens_k and a block table): sequence i owns
// Lq = cu_q[i+1]-cu_q[i] query rows and a context of Lk = cu_k[i+1]-cu_k[i]
// tokens, the first P = Lk - Lq of them a cached prefix; query r attends over
// context positions 0..P+r ("nano-vLLM Part 2", sections 2.5 and 4.1).  With
// a block table every context position is read from the pool (prefix and the
// rows pa_store_kv wrote this step, as the pages' layer does with
// k, v = k_cache, v_cache); without one, keys are the packed k/v rows.
//
// A work item = the same 128 query rows of two query heads of one GQA group
// (one head without GQA), so every 128-key K/V tile serves two Q tiles.  The
// grid is persistent: one CTA per SM, each working through its share of the
// items (ranked longest first and dealt out boustrophedon); TMEM and the
// barriers are set up once, and the K/V tile stream runs on from one item
// into the next (an item's last stage carries the next item's first K tile,
// and a head's next Q tile is loaded as soon as its last S of the item is
// done), so an item costs its key tiles and little else.
// Warp-specialised: warp 9 issues every TMA load, warp 8 every tcgen05.mma
// (one thread each); warpgroups 0 and 1 run the softmax of heads A and B
// (TMEM lane r = query row r); all hand-offs are mbarriers.  Back-to-back
// tcgen05.mma instructions issue at about their execution time (the tensor
// core queues one or two), so the issuing thread is the critical path: S
// MMAs use N = 128 keys, and per key tile the issuer does one wait and one
// commit for the K/V tiles (V_t and K_(t+1) share a stage barrier).  The heads
// ping-pong: while head A's softmax runs, the tensor core does head B's PV and
// next S, and vice versa.  Each head's S tile is overwritten in TMEM by its P,
// which the PV MMA reads from TMEM.
//   * Q and each 128-key K/V tile arrive by TMA with the 128-byte
//     swizzle the MMA descriptors expect; K/V tiles are double-buffered and
//     fetched page by page through the block table (one box per page when a
//     page is shorter than the tile); stage t = {V_t, K_(t+1)} is refilled
//     once the MMAs of step t-2 are done, and the tile two ahead is brought
//     into L2 meanwhile (its first copy then needs no trip to HBM).
//   * S = Q K^T: 128x128x16 tcgen05.mma steps, fp32 accumulator in TMEM.
//   * Softmax: each thread owns one row; it loads its S row from TMEM, masks
//     (causal, bottom-right aligned, and past the context), and exponentiates
//     in the log2 domain against a running maximum that is only moved when a
//     tile's maximum exceeds it by more than 2^8, so the TMEM accumulator O
//     is rescaled rarely; P is written back to TMEM as bf16/fp16.
//   * O += P V: tcgen05.mma with A = P in TMEM and V as an N-major
//     (D-contiguous) shared-memory operand, accumulating in TMEM.
//   * Every mbarrier wait is bounded; a wait that gives up flags
//     PA_FLAG_TIMEOUT, drains what this CTA has in flight (bounded again),
//     frees TMEM and returns.
#include <math.h>

#include <algorithm>

#include "tc_common.cuh"

namespace pa {
namespace {

constexpr int kBM = 128;  // query rows per Q tile
constexpr int kBN = 128;  // keys per K/V tile (the N of every S MMA)
constexpr int kWgThreads = 128;    // one softmax warpgroup: thread = query row = TMEM lane
constexpr int kMmaWarp = 8;        // warps 0-3: head A softmax, 4-7: head B softmax
constexpr int kTmaWarp = 9;        // warp 8: MMA issuer, warp 9: TMA producer
constexpr int kThreads = 2 * kWgThreads + 64;
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMaxRanked = 128;            // (sequence, q tile) items ordered longest first in-kernel

struct PrefillMaps {
    CUtensorMap q;  // [total_q rows, H_q*D cols], 128-row boxes
    CUtensorMap k;  // pool [N*bs rows, H_kv*D cols] (or packed [total_q, H_kv*D]), boxes of min(bs, 128) rows
    CUtensorMap v;
};

struct PrefillArgs {
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *block_tables;  // null: keys are the packed k/v rows
    int32_t max_blocks;
    int32_t num_blocks;
    int32_t log2_bs;
    int32_t box_rows;  // rows per K/V TMA box: min(block_size, kBN)
    int32_t num_q_heads;
    int32_t group;
    int32_t heads_per_cta;  // 2: two query heads of one GQA group share K/V; 1 without GQA
    int32_t total_q;
    int32_t qtiles;
    int32_t num_seqs;
    float scale_log2;
    void *out;
    int32_t *err_flag;
};

// Shared memory, every tile 1024-byte aligned with the 128-byte swizzle and
// stored as 64-column "halves" of 128-byte rows:
//   Q tile A, Q tile B [128 x D] | K slots 0, 1 [128 x D] | V slots 0, 1 [128 x D] | barriers
// 192 KB at D = 128: one CTA per SM.  TMEM (512 columns): per head, S/P
// [0, 128) (S_kt in fp32, then P_kt packed to 16 bits in its first 64
// columns) and O [128, 128 + D).
template <int D> struct PShape {
    static constexpr int kHalves = D / 64;
    static constexpr int kHalf = 128 * 128;  // one 64-column half of a 128-row tile
    static constexpr int kTile = kHalves * kHalf;
    static constexpr int kOffQ = 0;                 // + head * kTile
    static constexpr int kOffK = 2 * kTile;         // + slot * kTile
    static constexpr int kOffV = 4 * kTile;         // + slot * kTile
    static constexpr int kOffBar = 6 * kTile;
    static constexpr int kSmem = kOffBar + 256;
    static constexpr uint32_t kTmemCols = 512;
};

__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];\n" ::"l"(p));
}

template <typename T> struct IsBf16 { static constexpr bool value = false; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

// One unit of work: the 128 query rows of q tile q0 / kBM of one sequence, for the query
// heads h0 .. h0 + heads_per_cta - 1.
struct Item {
    int seq, h0, q_start, Lq, Lk, P, q0;
    int nkt;  // key tiles to stream; 0: nothing to do (tile past the chunk, or bad lengths)
};

// The item of schedule rank r.  The (sequence, q tile) groups are ranked longest first when
// the kernel ranked them (s_inv), else taken by sequence with the last q tile first; the head
// pairs of one group hold consecutive ranks.  With `report`, lengths that break the call's
// rules raise PA_FLAG_BAD_LENGTH (once per sequence: by the item of q tile 0, head pair 0).
__device__ __forceinline__ Item item_at(const PrefillArgs &a, const int *s_inv, bool ranked, int hps, int r,
                                        bool report) {
    Item it;
    int e = r / hps;
    const int hp = r - e * hps;
    if (ranked) e = s_inv[e];
    const int qt = ranked ? e % a.qtiles : a.qtiles - 1 - e % a.qtiles;
    it.seq = e / a.qtiles;
    it.h0 = hp * a.heads_per_cta;
    it.q_start = a.cu_q[it.seq];
    const int q_end = a.cu_q[it.seq + 1];
    it.Lq = q_end - it.q_start;
    it.Lk = a.cu_k[it.seq + 1] - a.cu_k[it.seq];
    it.P = it.Lk - it.Lq;
    it.q0 = qt * kBM;
    it.nkt = 0;
    const bool paged = a.block_tables != nullptr;
    const bool bad = it.Lq < 0 || it.P < 0 || it.q_start < 0 || q_end > a.total_q || (!paged && it.P != 0) ||
                     (paged && static_cast<int64_t>(it.Lk) > (static_cast<int64_t>(a.max_blocks) << a.log2_bs));
    if (bad) {
        if (report && qt == 0 && hp == 0) raise_flag(a.err_flag, PA_FLAG_BAD_LENGTH);
        return it;
    }
    if (report && qt == a.qtiles - 1 && hp == 0 && it.Lq > a.qtiles * kBM) raise_flag(a.err_flag, PA_FLAG_BAD_LENGTH);
    if (it.q0 >= it.Lq) return it;
    it.nkt = (min(it.Lk, it.P + it.q0 + kBM) + kBN - 1) / kBN;  // keys [0, hi) are visible to some row
    return it;
}

// This CTA's share of the items: CTA c of m takes, in round k, rank k*m + c (k even) or
// k*m + m-1-c (k odd) -- the ranks dealt out longest first, boustrophedon, so each CTA's
// rounds alternate between the long and the short end of a round.  Advances k to the next
// position of this CTA's list whose item has work; false when the list is done.
__device__ __forceinline__ int sched_rank(int k) {
    const int m = gridDim.x, c = blockIdx.x;
    return k * m + ((k & 1) ? m - 1 - c : c);
}
__device__ __forceinline__ bool next_item(const PrefillArgs &a, const int *s_inv, bool ranked, int hps, int total,
                                          int &k, Item &it, bool report) {
    for (; k * static_cast<int>(gridDim.x) < total; ++k) {
        const int r = sched_rank(k);
        if (r >= total) continue;
        it = item_at(a, s_inv, ranked, hps, r, report);
        if (it.nkt > 0) return true;
    }
    return false;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillMaps maps,
                                                              const PrefillArgs a) {
    using S = PShape<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    // launched as a programmatic dependent of the store of this step: wait for it first
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nwg = a.heads_per_cta;
    if (sb & 1023u) {  // the swizzled tiles need 1024-byte alignment
        if (tid == 0) raise_flag(a.err_flag, PA_FLAG_INTERNAL);
        return;
    }

    // Rank the (sequence, q tile) groups by their number of key tiles, longest first (every
    // CTA the same way); the CTAs then deal the items out among themselves (next_item).
    __shared__ int s_cost[kMaxRanked];
    __shared__ int s_inv[kMaxRanked];
    const int n_groups = a.num_seqs * a.qtiles;
    const bool ranked = n_groups <= kMaxRanked;
    const int hps = a.num_q_heads / a.heads_per_cta;
    const int total = n_groups * hps;
    if (ranked) {
        for (int e = tid; e < n_groups; e += kThreads) {
            const int sq = e / a.qtiles, t = e % a.qtiles;
            const int lq = a.cu_q[sq + 1] - a.cu_q[sq], lk = a.cu_k[sq + 1] - a.cu_k[sq];
            const int base = (lk - lq) + t * kBM;  // prefix + first row of the tile
            s_cost[e] = (t * kBM < lq && lk >= lq) ? (min(lk, base + kBM) + kBN - 1) / kBN : 0;
        }
        __syncthreads();
        for (int e = tid; e < n_groups; e += kThreads) {
            int r = 0;
            for (int f = 0; f < n_groups; ++f) r += s_cost[f] > s_cost[e] || (s_cost[f] == s_cost[e] && f < e);
            s_inv[r] = e;
        }
    }

    // mbarriers (8 bytes each) after the tiles.  Tiles are numbered u = 0, 1, ... across all
    // the items of this CTA, and stage u = {V_u, K_(u+1)} lands on one barrier (K_(u+1) is the
    // next item's first K tile after an item's last V tile): per key tile, one wait and one
    // commit for the tiles, and the stream of tiles runs on from one item into the next.
    const uint32_t bar0 = sb + S::kOffBar;
    auto bar_q = [&](int w) { return bar0 + (w ? 48 : 0); };           // Q tile of head w of an item landed
    const uint32_t bar_k0 = bar0 + 8;                                 // the first K tile landed
    auto bar_st = [&](int u) { return bar0 + 16 + 8 * (u & 1); };     // stage u landed (2 arrivals)
    auto bar_done = [&](int i) { return bar0 + 32 + 8 * (i & 1); };   // MMAs of step i-1 done (see below)
    auto bar_s = [&](int w) { return bar0 + 72 + 8 * w; };            // S_w in TMEM
    auto bar_p = [&](int w) { return bar0 + 88 + 8 * w; };            // P_w in TMEM (128 arrivals)
    auto bar_o = [&](int w) { return bar0 + 104 + 8 * w; };           // last PV_w of an item done
    const uint32_t tmem_slot = bar0 + 120;
    volatile int *abort_word = reinterpret_cast<volatile int *>(smem + S::kOffBar + 124);
    const uint32_t bar_drain = bar0 + 128;                            // MMA drain on abort

    if (tid == 0) {
        tc::mbar_init(bar_q(0), 1);
        tc::mbar_init(bar_q(1), 1);
        tc::mbar_init(bar_k0, 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar_st(i), 2);  // the V part and the K part (or a plain arrival)
            tc::mbar_init(bar_done(i), 1);
            tc::mbar_init(bar_s(i), 1);
            tc::mbar_init(bar_p(i), kWgThreads);
            tc::mbar_init(bar_o(i), 1);
        }
        tc::mbar_init(bar_drain, 1);
        tc::mbar_fence_init();
        *abort_word = 0;
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tmem_slot, S::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + S::kOffBar + 120);
    auto tS = [&](int w) { return tmem + 256 * w; };
    auto tO = [&](int w) { return tmem + 256 * w + 128; };
    auto wait = [&](uint32_t bar, uint32_t phase) {
        return tc::mbar_wait_or_abort(bar, phase, kWaitCycles, abort_word);
    };
    const bool paged = a.block_tables != nullptr;

    if (warp == kTmaWarp) {
        // ================= TMA producer: one thread =================
        if (lane == 0) {
            const bool one_box = a.box_rows == kBN;  // block_size >= kBN: a key tile lies in one page
            // physical page of logical page lp of item `it`
            auto page_of = [&](const Item &it, int lp) {
                int page = a.block_tables[static_cast<int64_t>(it.seq) * a.max_blocks + lp];
                if (page < 0 || page >= a.num_blocks) {
                    raise_flag(a.err_flag, PA_FLAG_BAD_BLOCK);
                    page = 0;  // stay inside the pool; the sequence's output is then unspecified
                }
                return page;
            };
            // keys [t*kBN, t*kBN + kBN) of item `it`'s K or V into `dst`, page by page through the block
            // table; with one box per tile its page `page0` was read beforehand
            auto load = [&](const Item &it, const CUtensorMap *map, uint32_t dst, uint32_t bar, int t, int page0) {
                const int j0 = t * kBN;
                const int x = (it.h0 / a.group) * D;  // both heads of the item read one kv head
                if (!paged) {
                    tc::mbar_arrive_expect_tx(bar, S::kTile);
                    for (int hf = 0; hf < S::kHalves; ++hf)
                        tc::tma_load_2d(dst + hf * S::kHalf, map, x + hf * 64, it.q_start + j0, bar);
                    return;
                }
                const int pages_in_ctx = (it.Lk + (1 << a.log2_bs) - 1) >> a.log2_bs;
                const int rows = a.box_rows;
                const int npg = kBN / rows;
                int n = 0;
                for (int p = 0; p < npg; ++p)
                    if (((j0 + p * rows) >> a.log2_bs) < pages_in_ctx) ++n;
                tc::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * rows * 128 * S::kHalves));
                for (int p = 0; p < npg; ++p) {
                    const int jp = j0 + p * rows;
                    const int lp = jp >> a.log2_bs;
                    if (lp >= pages_in_ctx) break;
                    const int page = one_box ? page0 : page_of(it, lp);
                    const int y = (page << a.log2_bs) + (jp & ((1 << a.log2_bs) - 1));
                    for (int hf = 0; hf < S::kHalves; ++hf)
                        tc::tma_load_2d(dst + hf * S::kHalf + p * rows * 128, map, x + hf * 64, y, bar);
                }
            };
            auto load_q = [&](const Item &it, int w) {  // the Q tile of the item's head w
                tc::mbar_arrive_expect_tx(bar_q(w), S::kTile);
                for (int hf = 0; hf < S::kHalves; ++hf)
                    tc::tma_load_2d(sb + S::kOffQ + w * S::kTile + hf * S::kHalf, &maps.q, (it.h0 + w) * D + hf * 64,
                                    it.q_start + it.q0, bar_q(w));
            };
            tc::prefetch_tmap(&maps.q);
            tc::prefetch_tmap(&maps.k);
            tc::prefetch_tmap(&maps.v);
            int k = 0;
            Item cur;
            bool have = next_item(a, s_inv, ranked, hps, total, k, cur, true);
            const bool started = have;
            int u = 0, issued = 0;
            int nq[2] = {0, 0};  // stages and Q tiles loaded, for the drain on abort
            int vpage = 0;       // one box per tile: the page of the next V tile (that of the K tile before)
            bool ok = true;
            if (have) {
                for (int w = 0; w < nwg; ++w) {
                    load_q(cur, w);
                    nq[w] = 1;
                }
                if (paged && one_box) vpage = page_of(cur, 0);
                load(cur, &maps.k, sb + S::kOffK, bar_k0, 0, vpage);
            }
            while (have && ok) {
                int kn = k + 1;
                Item nxt;
                const bool more = next_item(a, s_inv, ranked, hps, total, kn, nxt, true);
                if (more)  // the next item's Q tiles into L2 now; they are loaded at its first tile
                    for (int w = 0; w < nwg; ++w)
                        for (int hf = 0; hf < S::kHalves; ++hf)
                            tc::tma_prefetch_2d(&maps.q, (nxt.h0 + w) * D + hf * 64, nxt.q_start + nxt.q0);
                for (int t = 0; t < cur.nkt; ++t, ++u) {
                    // The block-table entry of the K tile this stage carries is read before the waits
                    // below, so its latency overlaps them instead of delaying the copies (one box per
                    // tile; with several, the entries are brought into L1 now and read after the wait).
                    int kpage = 0;
                    if (paged && (t + 1 < cur.nkt || more)) {
                        const Item &kit = t + 1 < cur.nkt ? cur : nxt;
                        const int lp = ((t + 1 < cur.nkt ? t + 1 : 0) * kBN) >> a.log2_bs;
                        if (one_box)
                            kpage = page_of(kit, lp);
                        else
                            prefetch_l1(a.block_tables + static_cast<int64_t>(kit.seq) * a.max_blocks + lp);
                    }
                    if (u >= 1) {
                        if (t == 0) {
                            // a head's Q tile is free once its last S of the item before is done
                            // (S_w(u-1): completion u-1 of bar_s(w); the next one needs this Q tile)
                            for (int w = 0; w < nwg && ok; ++w) {
                                ok = wait(bar_s(w), (u - 1) & 1);
                                if (!ok) break;
                                load_q(cur, w);
                                ++nq[w];
                            }
                            if (!ok) break;
                        }
                        // V_u goes to V slot u&1 (last read by PV(u-2)), K_(u+1) to K slot (u+1)&1
                        // (last read by S(u-1)): both are free once step u-2's MMAs are done (for
                        // u = 1: S(0))
                        ok = wait(bar_done(u - 1), ((u - 1) >> 1) & 1);
                        if (!ok) break;
                    }
                    load(cur, &maps.v, sb + S::kOffV + (u & 1) * S::kTile, bar_st(u), t, vpage);
                    // the K and V boxes of the item's tile t + 2 into L2 now: the first copy of a tile
                    // then finds it there instead of waiting on HBM (one box per tile)
                    if (paged && one_box && t + 2 < cur.nkt) {
                        const int jp = (t + 2) * kBN;
                        const int y = (page_of(cur, jp >> a.log2_bs) << a.log2_bs) + (jp & ((1 << a.log2_bs) - 1));
                        const int x = (cur.h0 / a.group) * D;
                        for (int hf = 0; hf < S::kHalves; ++hf) {
                            tc::tma_prefetch_2d(&maps.k, x + hf * 64, y);
                            tc::tma_prefetch_2d(&maps.v, x + hf * 64, y);
                        }
                    }
                    const uint32_t kdst = sb + S::kOffK + ((u + 1) & 1) * S::kTile;
                    if (t + 1 < cur.nkt)
                        load(cur, &maps.k, kdst, bar_st(u), t + 1, kpage);
                    else if (more)
                        load(nxt, &maps.k, kdst, bar_st(u), 0, kpage);
                    else
                        tc::mbar_arrive(bar_st(u));
                    vpage = kpage;
                    issued = u + 1;
                }
                k = kn;
                cur = nxt;
                have = more;
            }
            if (!ok) {  // let the copies this thread started land (bounded) before the CTA exits
                raise_flag(a.err_flag, PA_FLAG_TIMEOUT);
                *abort_word = 1;
                // a Q tile or stage is loaded only once the MMAs reading the one before it are
                // done, so only the last Q tile of each head and the last two stages can be in flight
                for (int w = 0; w < nwg; ++w)
                    if (nq[w]) tc::mbar_wait(bar_q(w), (nq[w] - 1) & 1, kWaitCycles);
                if (started) tc::mbar_wait(bar_k0, 0, kWaitCycles);
                for (int t = max(0, issued - 2); t < issued; ++t) tc::mbar_wait(bar_st(t), (t >> 1) & 1, kWaitCycles);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ================= MMA issuer: one thread =================
        if (lane == 0) {
            constexpr uint32_t kIdS = tc::idesc_f16(kBM, kBN, IsBf16<T>::value, false);
            constexpr uint32_t kIdO = tc::idesc_f16(kBM, D, IsBf16<T>::value, true);
            // descriptors built once; a k-step or slot moves only the start-address field
            const uint64_t dQ0 = tc::smem_desc_sw128(sb + S::kOffQ, 16, 1024);
            const uint64_t dK0 = tc::smem_desc_sw128(sb + S::kOffK, 16, 1024);
            const uint64_t dV0 = tc::smem_desc_sw128(sb + S::kOffV, S::kHalf, 1024);
            auto issue_s = [&](int w, int slot) {  // S_w = Q_w K^T, K in slot `slot`
                const uint64_t dq = dQ0 + static_cast<uint64_t>((w * S::kTile) >> 4);
                const uint64_t dk = dK0 + static_cast<uint64_t>((slot * S::kTile) >> 4);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = ((ks / 4) * S::kHalf + (ks % 4) * 32) >> 4;
                    tc::umma_f16(tS(w), dq + off, dk + off, kIdS, ks > 0);
                }
            };
            auto issue_pv = [&](int w, int slot, bool acc) {  // O_w (+)= P_w V, P_w from TMEM, V in `slot`
                const uint64_t dv = dV0 + static_cast<uint64_t>((slot * S::kTile) >> 4);
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks)
                    tc::umma_f16_ts(tO(w), tS(w) + ks * 8, dv + ((ks * 16 * 128) >> 4), kIdO,
                                    (acc || ks > 0) ? 1u : 0u);
            };
            // bar_done(i) completes when the MMAs issued before its i-th commit are done: i = 0
            // after S(0) of both heads, i = u + 1 after PV(u) and S(u+1) of both heads
            int k = 0, u = 0, j = 0;
            Item cur;
            bool have = next_item(a, s_inv, ranked, hps, total, k, cur, false);
            bool ok = true;
            if (have) {
                ok = wait(bar_k0, 0);
                for (int w = 0; w < nwg && ok; ++w) {
                    ok = wait(bar_q(w), 0);
                    if (!ok) break;
                    tc::fence_after_sync();
                    issue_s(w, 0);
                    tc::umma_commit(bar_s(w));
                }
                if (ok) tc::umma_commit(bar_done(0));
            }
            while (have && ok) {
                int kn = k + 1;
                Item nxt;
                const bool more = next_item(a, s_inv, ranked, hps, total, kn, nxt, false);
                for (int t = 0; t < cur.nkt && ok; ++t, ++u) {
                    // Per head: O += P V_u as soon as its softmax is done, then S for the next
                    // tile (it overwrites P, which the PV just issued reads first: MMAs run in
                    // issue order).  After an item's last tile the next S is the next item's first.
                    ok = wait(bar_st(u), (u >> 1) & 1);
                    const bool last = t + 1 == cur.nkt;
                    for (int w = 0; w < nwg && ok; ++w) {
                        ok = wait(bar_p(w), u & 1);
                        if (!ok) break;
                        tc::fence_after_sync();
                        issue_pv(w, u & 1, t > 0);
                        if (last) tc::umma_commit(bar_o(w));
                        if (last && !more) continue;
                        if (last) {  // the next item's Q tile of this head
                            ok = wait(bar_q(w), (j + 1) & 1);
                            if (!ok) break;
                            tc::fence_after_sync();
                        }
                        issue_s(w, (u + 1) & 1);
                        tc::umma_commit(bar_s(w));
                    }
                    if (!ok) break;
                    tc::umma_commit(bar_done(u + 1));
                }
                k = kn;
                cur = nxt;
                have = more;
                ++j;
            }
            if (!ok) {
                raise_flag(a.err_flag, PA_FLAG_TIMEOUT);
                *abort_word = 1;
                // one more commit covers every MMA this thread issued
                tc::umma_commit(bar_drain);
                tc::mbar_wait(bar_drain, 0, kWaitCycles);
            }
        }
        __syncwarp();
    } else if (warp / 4 < nwg) {
        // ================= softmax: thread = query row = TMEM lane =================
        // Scores stay raw (unscaled) until the single FFMA feeding the
        // exponential: scale > 0 keeps the raw maximum the scaled maximum.
        const int w = warp / 4;
        const int row = tid & (kWgThreads - 1);
        const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const float c = a.scale_log2;
        int k = 0, u = 0, j = 0;
        bool ok = true;
        for (;; ++k, ++j) {
            // only what the tile loop needs stays live across it; the epilogue looks the item up again
            int pq, Lk, nkt;  // prefix + first row of the tile, context length, key tiles
            {
                Item cur;
                if (!next_item(a, s_inv, ranked, hps, total, k, cur, false)) break;
                pq = cur.P + cur.q0;
                Lk = cur.Lk;
                nkt = cur.nkt;
            }
            const int limit = pq + row;  // last visible context position of this row
            float m_used = -INFINITY, l_sum = 0.f;  // m_used in scaled log2 units
            for (int t = 0; t < nkt && ok; ++t, ++u) {
                const int j0 = t * kBN;
                // S_w(u) ready; it was issued after PV_w(u-1), so O is stable too
                ok = __all_sync(0xffffffffu, wait(bar_s(w), u & 1));
                if (!ok) break;
                tc::fence_after_sync();
                const bool masked = (j0 + kBN - 1 > pq) || (j0 + kBN > Lk);  // diagonal or last tile
                const int lim = min(limit, Lk - 1) - j0;                            // last visible column
                // the row of S, read from TMEM once, masked in place
                uint32_t sr[kBN];
                tc::tmem_ld128(tS(w) + lane_base, sr);
                if (masked) {
#pragma unroll
                    for (int e = 0; e < kBN; ++e)
                        if (e > lim) sr[e] = __float_as_uint(-INFINITY);
                }
                // row maximum: three-input maxima, eight independent chains
                // (columns 0-7 start the chains, 8-119 go in pairs, 120-127 last)
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) m8[e] = __uint_as_float(sr[e]);
#pragma unroll
                for (int e = 8; e < kBN - 8; e += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        m8[i] = tc::max3(m8[i], __uint_as_float(sr[e + i]), __uint_as_float(sr[e + 8 + i]));
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], __uint_as_float(sr[kBN - 8 + i]));
                const float mx = tc::max3(tc::max3(m8[0], m8[1], m8[2]), tc::max3(m8[3], m8[4], m8[5]),
                                          fmaxf(m8[6], m8[7])) * c;
                // running maximum, moved only when this tile exceeds it by more than 2^8
                const float m_new = fmaxf(m_used, mx);
                float alpha = 1.f;
                bool rescale = false;
                if (t == 0) {
                    m_used = m_new;
                } else if (m_new > m_used + kRescaleThreshold) {
                    alpha = tc::ex2_approx(m_used - m_new);
                    m_used = m_new;
                    rescale = true;
                }
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tc::tmem_ld32(tO(w) + lane_base + 32 * cc, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::tmem_st32(tO(w) + lane_base + 32 * cc, o);
                    }
                }
                // P = 2^(c*s - m), packed to 16 bits over the first 64 columns of S, stored 8
                // columns (16 scores) at a time so that few registers hold packed P; the stores are
                // issued back to back and waited for once.
                // scale and shift two scores per instruction (packed fp32 pairs), sum P in pairs too
                const unsigned long long cc2 = tc::f32x2(c, c), nm2 = tc::f32x2(-m_used, -m_used);
                unsigned long long l2[2] = {0ull, 0ull};
#pragma unroll
                for (int ch = 0; ch < kBN / 16; ++ch) {
                    uint32_t pw[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const unsigned long long x = tc::fma_f32x2(
                            tc::f32x2(__uint_as_float(sr[16 * ch + e]), __uint_as_float(sr[16 * ch + e + 1])), cc2,
                            nm2);
                        const float p0 = tc::ex2_approx(tc::f32x2_lo(x));
                        const float p1 = tc::ex2_approx(tc::f32x2_hi(x));
                        l2[(e >> 1) & 1] = tc::add_f32x2(l2[(e >> 1) & 1], tc::f32x2(p0, p1));
                        pw[e >> 1] = Dt<T>::pack(p0, p1);
                    }
                    tc::tmem_st8_nowait(tS(w) + lane_base + 8 * ch, pw);  // P columns [8*ch, 8*ch + 8)
                }
                tc::tmem_wait_st();
                const unsigned long long ls = tc::add_f32x2(l2[0], l2[1]);
                l_sum = l_sum * alpha + (tc::f32x2_lo(ls) + tc::f32x2_hi(ls));
                const int valid = min(kBN, Lk - j0);
                if (w == 0 && valid < kBN) {
                    // V rows past the context may hold anything (NaN included): zero them so P V
                    // stays finite.  Head A does it; head B's PV is issued after head A's.
                    ok = __all_sync(0xffffffffu, wait(bar_st(u), (u >> 1) & 1));
                    if (!ok) break;
                    const int per_half = (kBN - valid) * 8;
                    uint4 *vz = reinterpret_cast<uint4 *>(smem + S::kOffV + (u & 1) * S::kTile);
                    for (int i = row; i < per_half * S::kHalves; i += kWgThreads) {
                        const int hf = i / per_half, rem = i % per_half;
                        vz[(hf * S::kHalf + (valid + rem / 8) * 128) / 16 + rem % 8] = make_uint4(0, 0, 0, 0);
                    }
                    tc::fence_async_smem();
                }
                // the P store (and, at an item's first tile, the last item's O read in the
                // epilogue below) is done before the PV that reads P and overwrites O is issued
                tc::fence_before_sync();
                tc::mbar_arrive(bar_p(w));
            }
            if (ok) ok = wait(bar_o(w), j & 1);  // committed once per item, after its last PV
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            {
                tc::fence_after_sync();
                const Item cur = item_at(a, s_inv, ranked, hps, sched_rank(k), false);
                const int qrow = cur.q0 + row;
                const float inv_l = 1.f / l_sum;
                T *dst = static_cast<T *>(a.out) +
                         (static_cast<int64_t>(cur.q_start + qrow) * a.num_q_heads + cur.h0 + w) * D;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tc::tmem_ld32(tO(w) + lane_base + 32 * cc, o);
                    if (qrow < cur.Lq) {
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) {
                            uint4 v;
                            v.x = Dt<T>::pack(__uint_as_float(o[q8 * 8 + 0]) * inv_l, __uint_as_float(o[q8 * 8 + 1]) * inv_l);
                            v.y = Dt<T>::pack(__uint_as_float(o[q8 * 8 + 2]) * inv_l, __uint_as_float(o[q8 * 8 + 3]) * inv_l);
                            v.z = Dt<T>::pack(__uint_as_float(o[q8 * 8 + 4]) * inv_l, __uint_as_float(o[q8 * 8 + 5]) * inv_l);
                            v.w = Dt<T>::pack(__uint_as_float(o[q8 * 8 + 6]) * inv_l, __uint_as_float(o[q8 * 8 + 7]) * inv_l);
                            *reinterpret_cast<uint4 *>(dst + 32 * cc + 8 * q8) = v;
                        }
                    }
                }
            }
        }
    }

    // teardown: every role is done with TMEM (the MMA issuer drained on abort)
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, S::kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

int ilog2(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

// SMs of the current device (cached per device)
int device_sms() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
        cached[dev] = sms;
    }
    return cached[dev];
}

template <typename T, int D>
cudaError_t run(const PrefillMaps &maps, const PrefillArgs &a, int ctas, cudaStream_t stream) {
    using S = PShape<D>;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = S::kSmem;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_kernel<T, D>, maps, a);
}

}  // namespace

cudaError_t launch_prefill(const void *q, const void *k, const void *v, const void *k_cache, const void *v_cache,
                           const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int32_t num_seqs,
                           int32_t total_q, int32_t max_seqlen_q, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t num_blocks, int32_t block_size, float scale, void *out, pa_dtype dtype,
                           int32_t *err_flag, int32_t sms, cudaStream_t stream, const char **why) {
    *why = nullptr;
    if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return cudaSuccess;
    PrefillMaps maps;
    const int64_t kv_cols = static_cast<int64_t>(num_kv_heads) * head_dim;
    bool ok = make_tmap_rows(&maps.q, q, dtype, static_cast<int64_t>(num_q_heads) * head_dim, total_q, kBM);
    int box_rows = kBN;
    if (block_tables) {
        box_rows = block_size < kBN ? block_size : kBN;
        const int64_t rows = static_cast<int64_t>(num_blocks) * block_size;
        ok = ok && make_tmap_rows(&maps.k, k_cache, dtype, kv_cols, rows, box_rows) &&
             make_tmap_rows(&maps.v, v_cache, dtype, kv_cols, rows, box_rows);
    } else {
        ok = ok && make_tmap_rows(&maps.k, k, dtype, kv_cols, total_q, kBN) &&
             make_tmap_rows(&maps.v, v, dtype, kv_cols, total_q, kBN);
    }
    if (!ok) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or tensor too large)";
        return cudaErrorInvalidValue;
    }
    PrefillArgs a;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.log2_bs = ilog2(block_size);
    a.box_rows = box_rows;
    a.num_q_heads = num_q_heads;
    a.group = num_q_heads / num_kv_heads;
    a.heads_per_cta = a.group >= 2 ? 2 : 1;
    a.total_q = total_q;
    a.qtiles = (max_seqlen_q + kBM - 1) / kBM;
    a.num_seqs = num_seqs;
    a.scale_log2 = scale * kLog2e;
    a.out = out;
    a.err_flag = err_flag;
    // persistent: one CTA per SM the kernel may use (it holds a whole SM), at most one per item
    const int64_t items = static_cast<int64_t>(num_seqs) * a.qtiles * (num_q_heads / a.heads_per_cta);
    const int ctas = static_cast<int>(std::min<int64_t>(items, sms > 0 ? sms : device_sms()));
    if (dtype == PA_BF16)
        return head_dim == 128 ? run<__nv_bfloat16, 128>(maps, a, ctas, stream)
                               : run<__nv_bfloat16, 64>(maps, a, ctas, stream);
    return head_dim == 128 ? run<__half, 128>(maps, a, ctas, stream) : run<__half, 64>(maps, a, ctas, stream);
}

}  // namespace pa
