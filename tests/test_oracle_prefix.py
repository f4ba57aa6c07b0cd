"""Pins for the oracle's prefix cache, copy-on-write and block copy.

Each test checks the oracle against something other than itself: a trace
worked out by hand, a closed form from the pages' examples, or a brute-force
longest-common-prefix search over the inserted sequences.
"""
import numpy as np
import pytest

import oracle
from oracle.prefix import PrefixCache, copy_blocks, cow


def _serve(pc, alloc, tokens, bs):
    """Admit one request: reuse the cached prefix, allocate the rest, cache its full blocks."""
    shared = pc.match(tokens)
    need = -(-len(tokens) // bs) - len(shared)
    own = [int(x) for x in alloc.alloc(need)] if need > 0 else []
    table = list(shared) + own
    pc.insert(tokens, table)
    return table, len(shared)


def test_shared_system_prompt_is_stored_once():
    # "LLM Inference Optimization", KV Cache Management: 100 requests with the
    # same system prompt compute its KV once and share it.  A 2304-token prompt
    # in 16-token blocks is 144 blocks; each request adds a private suffix.
    bs, P, R = 16, 2304, 100
    rng = np.random.default_rng(5)
    prompt = list(rng.integers(0, 32000, P))
    suffix = [int(x) for x in rng.integers(1, 200, R)]
    alloc = oracle.Allocator(20000)
    pc = PrefixCache(alloc, bs)
    tables, written = [], 0
    for r in range(R):
        toks = prompt + list(rng.integers(32000, 64000, suffix[r]))
        table, nshared = _serve(pc, alloc, toks, bs)
        assert nshared == (0 if r == 0 else P // bs)
        written += len(toks) - nshared * bs          # tokens whose KV this request computes
        tables.append(table)
    # closed forms: blocks in use, prefill work, and one reference per user of a prompt block
    assert alloc.num_blocks - alloc.num_free() == P // bs + sum(-(-s // bs) for s in suffix)
    assert written == P + sum(suffix)
    for j in range(P // bs):
        assert all(t[j] == tables[0][j] for t in tables)
        assert alloc.refcount(tables[0][j]) == R + 1   # every request + the cache


@pytest.mark.parametrize("p", [0, 1, 15, 16, 17, 100, 159])
def test_changed_token_keeps_only_the_blocks_before_it(p):
    # "LLM Serving - ...", KV memory, paging and prefix identity: reuse needs
    # the exact token prefix; "KV cache & continuous batching", Pitfall 3: a
    # date in the system prompt invalidates the cache.  A change at position p
    # leaves floor(p / bs) reusable blocks.
    bs = 16
    alloc = oracle.Allocator(64)
    pc = PrefixCache(alloc, bs)
    toks = list(range(1000, 1160))                    # 10 full blocks
    table, _ = _serve(pc, alloc, toks, bs)
    other = list(toks)
    other[p] = -1
    got = pc.match(other)
    assert got == table[: p // bs]


def test_only_full_blocks_are_cached():
    bs = 16
    alloc = oracle.Allocator(8)
    pc = PrefixCache(alloc, bs)
    blocks = [int(x) for x in alloc.alloc(2)]
    pc.insert(list(range(15)), blocks[:1])            # 15 tokens: no full block
    assert pc.size() == 0 and alloc.refcount(blocks[0]) == 1
    pc.insert(list(range(31)), blocks)                # 31 tokens: one full block
    assert pc.size() == 1 and alloc.refcount(blocks[0]) == 2 and alloc.refcount(blocks[1]) == 1
    assert pc.match(list(range(15))) == []
    assert pc.match(list(range(40))) == blocks[:1]


def test_match_equals_brute_force_longest_common_prefix():
    # tiny alphabet and block size so that prefixes collide often
    rng = np.random.default_rng(11)
    for trial in range(40):
        bs = int(rng.integers(1, 4))
        alloc = oracle.Allocator(4096)
        pc = PrefixCache(alloc, bs)
        seqs, tables = [], []
        for _ in range(int(rng.integers(1, 8))):
            toks = [int(x) for x in rng.integers(0, 2, int(rng.integers(0, 10)))]
            table, _ = _serve(pc, alloc, toks, bs)
            seqs.append(toks)
            tables.append(table)
        for _ in range(20):
            qry = [int(x) for x in rng.integers(0, 2, int(rng.integers(0, 12)))]
            best, src = 0, None
            for s, t in zip(seqs, tables):
                lcp = 0
                while lcp < min(len(s), len(qry)) and s[lcp] == qry[lcp]:
                    lcp += 1
                k = min(lcp // bs, len(s) // bs)
                if k > best:
                    best, src = k, t
            got = pc.match(qry)
            assert len(got) == best
            if best:
                assert got == src[:best]
            alloc.free(got)


def test_lru_eviction_hand_trace():
    bs = 4
    alloc = oracle.Allocator(16)
    pc = PrefixCache(alloc, bs)
    A = list(range(12))                                # 3 blocks
    B = A[:4] + [9] * 8                                # shares A's first block
    ta, _ = _serve(pc, alloc, A, bs)                   # clock 1-2: blocks 0 1 2
    tb, _ = _serve(pc, alloc, B, bs)                   # clock 3-4: blocks 0 3 4
    assert ta == [0, 1, 2] and tb == [0, 3, 4]
    alloc.free(ta)
    alloc.free(tb)                                     # only the cache holds them now
    m = pc.match(A)                                    # clock 5: A's chain is the most recent
    assert m == [0, 1, 2]
    # a block a sequence still holds is never evicted
    assert pc.evict(1) == 1 and pc.size() == 4         # B's end (block 4) goes first
    assert alloc.refcount(4) == 0
    assert pc.evict(10) == 1                           # block 3; A's chain is held by the match
    alloc.free(m)
    # A's chain from its end: 2, then 1, then 0
    order = []
    for _ in range(3):
        before = {b for b in range(5) if alloc.refcount(b)}
        assert pc.evict(1) == 1
        order += sorted(before - {b for b in range(5) if alloc.refcount(b)})
    assert order == [2, 1, 0] and pc.size() == 0 and alloc.num_free() == 16


def test_eviction_skips_blocks_in_use_and_chain_interiors():
    bs = 2
    alloc = oracle.Allocator(8)
    pc = PrefixCache(alloc, bs)
    ta, _ = _serve(pc, alloc, [1, 1, 2, 2, 3, 3], bs)  # blocks 0 1 2
    tc, _ = _serve(pc, alloc, [4, 4], bs)              # block 3
    alloc.free(ta[:2])
    alloc.free(tc)                                     # a sequence still holds block 2
    # block 2 is in use, blocks 0 and 1 are interior: only block 3 can go
    assert pc.evict(10) == 1 and alloc.refcount(3) == 0
    assert [alloc.refcount(b) for b in ta] == [1, 1, 2]
    alloc.free(ta[2:])
    assert pc.evict(10) == 3 and alloc.num_free() == 8


def test_two_chain_ends_never_share_a_last_use():
    # one call stamps one path, and a path has one end: the LRU order of
    # chain ends is total, so the depth / block-id tie-breaks never decide
    rng = np.random.default_rng(3)
    alloc = oracle.Allocator(4096)
    pc = PrefixCache(alloc, 2)
    for _ in range(200):
        toks = [int(x) for x in rng.integers(0, 3, int(rng.integers(0, 12)))]
        table, _ = _serve(pc, alloc, toks, 2)
        alloc.free(table)
        if rng.random() < 0.3:
            pc.evict(int(rng.integers(1, 4)))
        ends = [v[1] for k, v in pc.entries.items() if pc._is_chain_end(k)]
        assert len(ends) == len(set(ends))


def test_copy_on_write_fork():
    # two sequences share a partly filled block after a fork; the first writer
    # takes a private copy, the second then owns the original and writes in place
    alloc = oracle.Allocator(4)
    a = [int(x) for x in alloc.alloc(2)]               # 0 1
    alloc.share(a)                                     # fork: b holds the same blocks
    assert cow(alloc, a[1]) == (2, True)
    assert alloc.refcount(1) == 1 and alloc.refcount(2) == 1
    assert cow(alloc, a[1]) == (1, False)
    assert cow(alloc, 2) == (2, False)
    # out of blocks: nothing changes
    alloc.alloc(1)                                     # 3
    alloc.share([0])
    with pytest.raises(MemoryError):
        cow(alloc, 0)
    assert alloc.refcount(0) == 3 and alloc.num_free() == 0
    with pytest.raises(ValueError):
        cow(alloc, 3 + 1)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_copy_blocks_copies_only_the_named_blocks(kv):
    c = oracle.Cache(6, 2, 8, 4, kv)
    rng = np.random.default_rng(1)
    c.k[:] = rng.integers(0, 255, c.k.shape)
    c.v[:] = rng.integers(0, 255, c.v.shape)
    if kv == "fp8":
        c.k_scale[:] = rng.random(c.k_scale.shape)
        c.v_scale[:] = rng.random(c.v_scale.shape)
    k0, v0 = c.k.copy(), c.v.copy()
    copy_blocks(c, [1, 4], [5, 0])
    assert np.array_equal(c.k[5], k0[1]) and np.array_equal(c.v[0], v0[4])
    assert np.array_equal(c.k[[1, 2, 3, 4]], k0[[1, 2, 3, 4]])
    if kv == "fp8":
        assert c.k_scale[5, 1] == c.k_scale[1, 1] and c.v_scale[0, 0] == c.v_scale[4, 0]
