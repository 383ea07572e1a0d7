"""GPU parity of the prefix-sharing decode (pa_decode_ex / pa_store_decode_ex with
shared-prefix groups from pa_prefix_groups) against the oracle: the full
Qwen3-8B-like workload (groups of 8 sharing a 512-token prefix), GQA group sizes
1..8 (prefix CTAs serving 4 to 32 sequences, groups split over several CTAs),
both head dims and dtypes, block sizes 8..256, prefixes split over several
partitions and ending inside a tile, batches mixing groups, unshared sequences
and padding rows, private parts split over several partitions, and descriptors
that break the rules (flagged, never faulting).  The sharing changes which CTA
reads a page, not the attention: every case is also compared with the plain
decode of the same step."""

import pytest
import torch

import oracle
from tests import inputs
from tests.gpu_cases import TOL, assert_bit_equal, max_err

pytestmark = pytest.mark.gpu


def _groups(pa, st, min_pages=1):
    from paged_kv_cache_bs_gb300.block_manager import prefix_groups
    return prefix_groups(st.block_tables, st.context_lens, st.pool.block_size, min_pages).to("cuda")


def _run(pa, st, options, fused=False, err_flag=None):
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    q, kn, vn, sm = st.q.cuda(), st.k_new.cuda(), st.v_new.cuda(), st.slot_mapping.cuda()
    bt, cl = st.block_tables.cuda(), st.context_lens.cuda()
    if fused:
        out = pa.store_decode(kn, vn, sm, q, kc, vc, bt, cl, st.scale, err_flag=err_flag, options=options)
    else:
        pa.store_kv(kn, vn, kc, vc, sm, err_flag=err_flag)
        out = pa.decode(q, kc, vc, bt, cl, st.scale, err_flag=err_flag, options=options)
    torch.cuda.synchronize()
    return out, kc, vc


def check_shared(pa, st, fused=False, min_groups=1, **opt):
    g = _groups(pa, st)
    assert g.num_groups >= min_groups
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, kc, vc = _run(pa, st, pa.DecodeOptions(groups=g, **opt), fused, flag)
    assert int(flag.item()) == 0, f"flags {int(flag.item())}"
    okc, ovc = st.pool.k_cache.clone(), st.pool.v_cache.clone()
    oracle.store_kv(st.k_new, st.v_new, okc, ovc, st.slot_mapping)
    assert_bit_equal(kc, okc, "k_cache after the store")
    assert_bit_equal(vc, ovc, "v_cache after the store")
    ref = oracle.decode(st.q, okc, ovc, st.block_tables, st.context_lens, st.scale)
    err = max_err(out, ref)
    assert err <= TOL[st.q.dtype], f"max |err| {err} vs the oracle"
    plain, _, _ = _run(pa, st, None, fused)
    assert max_err(out, plain.cpu().float()) <= TOL[st.q.dtype]
    return err, g


@pytest.mark.parametrize("fused", [False, True])
def test_shared_prefix_workload_full(pa, fused):
    st = inputs.qwen3_8b_shared_decode()
    err, g = check_shared(pa, st, fused=fused, min_groups=32)
    assert g.num_groups == 32 and g.max_group_size == 8 and g.max_prefix_len == 512
    print(f"qwen3_8b_shared_decode, 32 groups of 8 sharing 512 tokens (fused={fused}): max|err| {err:.3e}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (8, 1)])
def test_shared_prefix_group_sizes(pa, dtype, head_dim, hq, hkv):
    # one prefix CTA serves 32 / G sequences: groups of 40 (G = 1: two CTAs), 9, 5 and 2 members
    sizes = [40, 9, 5, 2]
    seqs, grp = [], 0
    for n, share in zip(sizes, [64, 160, 320, 32]):
        for i in range(n):
            seqs.append((share + 1 + (37 * i + 11 * grp) % 300, grp, share))
        grp += 1
    st = inputs.make_decode_shared(seqs, num_q_heads=hq, num_kv_heads=hkv, head_dim=head_dim, block_size=16,
                                   dtype=dtype, seed=101 + hq // hkv + head_dim)
    check_shared(pa, st, min_groups=4)


@pytest.mark.parametrize("bs,share", [(8, 72), (16, 528), (64, 640), (256, 1536)])
@pytest.mark.parametrize("prefix_partition", [0, 64, 192])
def test_shared_prefix_block_sizes_and_partitions(pa, bs, share, prefix_partition):
    # prefixes ending on and off 64-token tiles, split over one or many prefix partitions
    seqs = [(share + 1 + 5 * i, 0, share) for i in range(6)] + [(share + 700 + i, 1, share) for i in range(3)]
    st = inputs.make_decode_shared(seqs, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=bs,
                                   dtype=torch.bfloat16, seed=111 + bs)
    check_shared(pa, st, min_groups=2, prefix_partition=prefix_partition)


@pytest.mark.parametrize("fused", [False, True])
def test_shared_prefix_mixed_batch(pa, fused):
    # groups, unshared sequences, padding rows, members one token past the prefix, and private
    # parts long enough for several partitions (partition 128)
    seqs = [(513, 0, 512), (0, -1, 0), (2000, 0, 512), (700, -1, 0), (1025, 0, 512), (5, -1, 0),
            (33, 1, 32), (3000, 1, 32), (0, -1, 0), (100, 1, 32), (4096, -1, 0), (17, 2, 16), (18, 2, 16)]
    st = inputs.make_decode_shared(seqs, num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                                   dtype=torch.bfloat16, seed=121)
    check_shared(pa, st, fused=fused, min_groups=3, partition=128)


def test_shared_prefix_workspace_holds_the_prefix_partials(pa):
    st = inputs.qwen3_8b_shared_decode()
    g = _groups(pa, st)
    n, bs, hkv, d = st.pool.k_cache.shape
    plain = pa.decode_workspace_bytes(st.batch, st.num_q_heads, hkv, d, st.block_tables.shape[1], bs)
    grouped = pa.decode_workspace_bytes(st.batch, st.num_q_heads, hkv, d, st.block_tables.shape[1], bs,
                                        pa.DecodeOptions(groups=g))
    assert grouped > plain


def test_shared_prefix_bad_descriptors_are_flagged_not_fatal(pa):
    seqs = [(300, 0, 256), (400, 0, 256), (500, 0, 256), (90, -1, 0)]
    st = inputs.make_decode_shared(seqs, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                                   dtype=torch.bfloat16, seed=131)
    g = _groups(pa, st)
    cases = []
    bad = g.prefix_lens.clone()
    bad[1] = 128                                   # a member reading a different prefix
    cases.append(inputs_groups(pa, g, prefix_lens=bad))
    bad = g.prefix_lens.clone()
    bad[0] = bad[1] = bad[2] = 300                 # prefix reaching the newest token of a member
    cases.append(inputs_groups(pa, g, prefix_lens=bad))
    bt = st.block_tables.clone()
    bt[2, 3] = bt[3, 0]                            # a member's table leaves the shared pages
    for opts, tables in ((cases[0], st.block_tables), (cases[1], st.block_tables),
                         (pa.DecodeOptions(groups=g), bt)):
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        kc, vc = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
        pa.decode(st.q.cuda(), kc, vc, tables.cuda(), st.context_lens.cuda(), st.scale, err_flag=flag, options=opts)
        torch.cuda.synchronize()
        assert int(flag.item()) & pa.FLAG_BAD_GROUP
    check_shared(pa, st)   # the device is still healthy


def inputs_groups(pa, g, prefix_lens):
    return pa.DecodeOptions(groups=pa.PrefixGroups(g.group_offsets, g.group_seqs, prefix_lens, g.max_group_size,
                                                   max(g.max_prefix_len, int(prefix_lens.max()))))

