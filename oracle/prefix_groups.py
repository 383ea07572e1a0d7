"""Shared-prefix groups of a decode batch -- TEST INFRASTRUCTURE ONLY (the
oracle of ``pa_prefix_groups`` in
``paged_kv_cache_bs_gb300/csrc/block_manager.cpp``; the two share no code).

Prefix caching makes sequences with a common prompt prefix point at the same
physical pages: "nano-vLLM Part 2: Block Tables, KV Cache, and the Path to the
GPU", section 2.5 (prompt B's block table [0, 3, 4, 5] starts with A's page 0,
whose reference count goes to 2), and "How vLLM works" (prefix caching: full
blocks are shared by reference count).  A decode step can then read such a
page once for every sequence that shares it.  The pages define the sharing but
no grouping of a decode batch; the rule here, written plainly:

1. Sequences with an empty context (padding rows), and sequences whose newest
   token sits in their first page (context length L <= block_size: they hold
   no complete page), are never grouped.
2. The other sequences are grouped by the first entry of their block table, in
   the order the first member of each group appears in the batch.
3. A group of two or more members shares its first n pages, n being the
   number of leading table entries equal across all members, but at most
   (L - 1) // block_size for every member of context length L: the page that
   holds a sequence's newest token (the one this decode step writes) and any
   page after it are never shared (the pages never share a partial page,
   section 2.4: only complete pages are hashed).
4. A group with n < min_shared_pages is dissolved; singletons are not groups.

Returns (group_offsets, group_seqs, prefix_lens): the members of group g are
group_seqs[group_offsets[g]:group_offsets[g + 1]] (batch order), and
prefix_lens[b] = n * block_size for a member of a group, 0 otherwise.
"""

from __future__ import annotations


def prefix_groups(block_tables, context_lens, block_size: int, min_shared_pages: int = 1):
    B = len(context_lens)
    by_first: dict[int, list[int]] = {}
    for b in range(B):
        if (context_lens[b] - 1) // block_size < 1:    # padding row, or no complete page
            continue
        by_first.setdefault(block_tables[b][0], []).append(b)   # dict keeps first-appearance order
    offsets, seqs, prefix = [0], [], [0] * B
    for members in by_first.values():
        if len(members) < 2:
            continue
        cap = min((context_lens[b] - 1) // block_size for b in members)
        lead = block_tables[members[0]]
        n = 0
        while n < cap and all(block_tables[b][n] == lead[n] for b in members):
            n += 1
        if n < max(min_shared_pages, 1):
            continue
        seqs.extend(members)
        offsets.append(len(seqs))
        for b in members:
            prefix[b] = n * block_size
    return offsets, seqs, prefix
