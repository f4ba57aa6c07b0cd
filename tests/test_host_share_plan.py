"""pa_share_plan (host): the chunks of sequences whose leading blocks are the
same physical blocks, checked against the plan's definition by brute force."""
import numpy as np
import pytest

import oracle.run
import paged_kv_cache_294_gb300 as pa
import workloads

R = pa.PA_SHARE_MAX_ROWS


def _check_plan(tables, lens, bs, group_rows, min_blocks, plan):
    B = len(lens)
    cap = [max(0, min((int(l) - 1) // bs, tables.shape[1])) if l >= 1 else 0 for l in lens]
    members = plan["chunk_members"]
    seen = set()
    for c, (row, L) in enumerate(zip(members, plan["chunk_blocks"])):
        ms = [int(b) for b in row if b >= 0]
        assert 1 <= len(ms) <= group_rows and all(b == -1 for b in row[len(ms):])
        assert L >= max(min_blocks, 1)
        for k, b in enumerate(ms):
            assert b not in seen
            seen.add(b)
            assert plan["chunk_of"][b] == R * c + k
            assert L <= cap[b]
            assert np.array_equal(tables[b, :L], tables[ms[0], :L])
    for b in range(B):
        if b not in seen:
            assert plan["chunk_of"][b] == -1
    # maximality: a group (same first block among eligible sequences) shares as
    # many blocks as all its members have in common, capped by each member
    groups = {}
    for b in range(B):
        if cap[b] >= max(min_blocks, 1):
            groups.setdefault(int(tables[b, 0]), []).append(b)
    for first, bs_ in groups.items():
        if len(bs_) < 2 or group_rows < 2:
            assert all(plan["chunk_of"][b] == -1 for b in bs_)
            continue
        L = min(cap[b] for b in bs_)
        for b in bs_[1:]:
            c = 0
            while c < L and tables[b, c] == tables[bs_[0], c]:
                c += 1
            L = c
        if L >= max(min_blocks, 1):
            assert all(plan["chunk_of"][b] >= 0 for b in bs_)
            assert all(plan["chunk_blocks"][plan["chunk_of"][b] // R] == L for b in bs_)
        else:
            assert all(plan["chunk_of"][b] == -1 for b in bs_)


def test_shared_prefix_workload_plan():
    w = workloads.make("fp8prefix")
    t = oracle.run.tables_of(w)
    p = pa.pa_share_plan(t, w.seq_lens, w.bs, R // (w.Hq // w.Hkv))
    assert len(p["chunk_blocks"]) == 13 and p["max_chunk_blocks"] == 64
    assert list(p["chunk_members"][0]) == list(range(8))
    assert list(p["chunk_members"][12]) == [96, 97, 98, 99, -1, -1, -1, -1]
    assert (p["chunk_of"][:100] >= 0).all() and (p["chunk_of"][100:] == -1).all()
    _check_plan(t, w.seq_lens, w.bs, 8, 1, p)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("group_rows", [1, 2, 4, 8])
def test_random_plans_meet_the_definition(seed, group_rows):
    rng = np.random.default_rng(seed)
    bs, M = 16, 24
    B = int(rng.integers(1, 40))
    tables = np.full((B, M), -1, np.int32)
    lens = np.zeros(B, np.int32)
    nxt = 0
    prefixes = [list(range(1000 + 50 * g, 1000 + 50 * g + int(rng.integers(1, 12)))) for g in range(4)]
    for b in range(B):
        L = int(rng.integers(0, M * bs + 1))
        lens[b] = L
        nb = -(-L // bs)
        g = int(rng.integers(0, 5))      # g == 4: no shared prefix
        pre = prefixes[g][: int(rng.integers(0, len(prefixes[g]) + 1))] if g < 4 else []
        row = (pre + list(range(nxt, nxt + nb)))[:nb]
        nxt += nb
        tables[b, :len(row)] = row
    min_blocks = int(rng.integers(0, 4))
    p = pa.pa_share_plan(tables, lens, bs, group_rows, min_blocks)
    if group_rows < 2:
        assert len(p["chunk_blocks"]) == 0
    _check_plan(tables, lens, bs, group_rows, min_blocks, p)


def test_plan_stops_at_max_chunks_and_rejects_bad_arguments():
    tables = np.tile(np.arange(8, dtype=np.int32), (20, 1))
    lens = np.full(20, 8 * 16, np.int32)
    p = pa.pa_share_plan(tables, lens, 16, 4, max_chunks=2)
    assert len(p["chunk_blocks"]) == 2 and (p["chunk_of"] >= 0).sum() == 8
    assert p["max_chunk_blocks"] == 7            # the last block holds the newest token
    with pytest.raises(pa.PagedAttnError):
        pa.pa_share_plan(tables, lens, 16, 9)    # more rows than a chunk holds
    with pytest.raises(pa.PagedAttnError):
        pa.pa_share_plan(tables, lens, 0, 4)
