"""The library's host side (allocator, accounting, slots, schedulers) against the oracle.

Bit-exact: block ids, tables, slots and iteration counts must equal the
oracle's on the same inputs and operation traces.
"""
import numpy as np
import pytest

import oracle
import oracle.run
import paged_kv_cache_294_gb300 as pa
import workloads
from paged_kv_cache_294_gb300.engine import replay_trace
from tests.golden.load import page_numbers


def test_page_numbers_through_the_library():
    for kind, v in page_numbers():
        if kind == "kv_bytes":
            assert pa.pa_kv_bytes(*v[:6]) == v[6]
        elif kind == "blocks":
            assert pa.pa_blocks_for_tokens(v[0], v[1]) == v[2]
        elif kind == "sched":
            st, co, slots, lens = v[0], v[1], v[2], v[3:]
            assert pa.pa_sched_simulate(lens, slots, 0) == st
            assert pa.pa_sched_simulate(lens, slots, 1) == co


def test_accounting_matches_oracle():
    rng = np.random.default_rng(0)
    for _ in range(200):
        args = [int(x) for x in (rng.integers(0, 100), rng.integers(0, 65), rng.integers(0, 257),
                                 rng.choice([4, 8, 16, 32]), rng.integers(0, 200000), rng.integers(0, 300))]
        assert pa.pa_kv_bytes(*args) == oracle.kv_bytes(*args)
        t, bs = int(rng.integers(-5, 100000)), int(rng.choice([1, 16, 32]))
        assert pa.pa_blocks_for_tokens(t, bs) == oracle.blocks_for_tokens(t, bs)


def test_scheduler_matches_oracle_and_rejects_bad_domain():
    rng = np.random.default_rng(1)
    for _ in range(300):
        n = int(rng.integers(0, 20))
        lens = [int(x) for x in rng.integers(1, 50, size=n)]
        slots = int(rng.integers(1, 8))
        assert pa.pa_sched_simulate(lens, slots, 0) == oracle.sched_static(lens, slots)
        assert pa.pa_sched_simulate(lens, slots, 1) == oracle.sched_continuous(lens, slots)
    for bad in (([5, 3], 0, 1), ([5, 0], 2, 1), ([5], 1, 2)):
        with pytest.raises(pa.PagedAttnError):
            pa.pa_sched_simulate(*bad)


def _random_trace_check(num_blocks, steps, seed):
    rng = np.random.default_rng(seed)
    a, o = pa.pa_allocator(num_blocks, 16), oracle.Allocator(num_blocks)
    held = []
    for _ in range(steps):
        op = int(rng.integers(4))
        if op <= 1:
            n = int(rng.integers(0, 12))
            try:
                got = a.alloc(n)
            except pa.PagedAttnError as e:
                assert e.status == pa.PA_ERR_OOM
                with pytest.raises(MemoryError):
                    o.alloc(n)
                continue
            assert np.array_equal(got, o.alloc(n))
            held.append(list(got))
        elif op == 2 and held:
            ids = held.pop(int(rng.integers(len(held))))
            a.free(ids)
            o.free(ids)
        elif op == 3 and held:
            ids = held[int(rng.integers(len(held)))]
            a.share(ids)
            o.share(ids)
            held.append(list(ids))
        assert a.num_free() == o.num_free()
    for i in range(num_blocks):
        assert a.refcount(i) == o.refcount(i)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_allocator_bit_exact_on_random_traces(seed):
    _random_trace_check(97, 600, seed)


def test_allocator_error_cases():
    a = pa.pa_allocator(8, 16)
    assert list(a.alloc(3)) == [0, 1, 2]
    with pytest.raises(pa.PagedAttnError) as e:
        a.alloc(6)
    assert e.value.status == pa.PA_ERR_OOM and a.num_free() == 5
    with pytest.raises(pa.PagedAttnError):
        a.free([3])                 # never allocated
    with pytest.raises(pa.PagedAttnError):
        a.free([0, 0])              # two drops, one reference
    assert a.refcount(0) == 1
    with pytest.raises(pa.PagedAttnError):
        a.share([7])
    with pytest.raises(pa.PagedAttnError):
        a.free([-1])
    with pytest.raises(ValueError):
        pa.pa_allocator(-1, 16)


@pytest.mark.parametrize("name,kw", [("70b", {}), ("fp8prefix", {}), ("70b", dict(B=16, seq_len=512))])
def test_workload_trace_tables_bit_exact(name, kw):
    w = workloads.make(name, **kw)
    t_lib, alloc = replay_trace(w.trace, w.num_blocks, w.bs, w.target_rids, w.M)
    t_or = oracle.run.replay_trace(w.trace, w.num_blocks, w.target_rids, w.M)
    assert np.array_equal(t_lib, t_or)
    # every sequence's table covers its length; shared prefix blocks appear in many tables
    for b, L in enumerate(w.seq_lens):
        nb = -(-int(L) // w.bs)
        assert np.all(t_lib[b, :nb] >= 0) and np.all(t_lib[b, nb:] == -1)
    if name == "fp8prefix":
        pre = t_lib[0, :64]
        assert all(np.array_equal(t_lib[b, :64], pre) for b in range(100))
        assert all(alloc.refcount(int(i)) == 100 for i in pre)
    used = t_lib[t_lib >= 0]
    if name == "70b":
        assert len(np.unique(used)) == len(used)                # no sharing in this workload
        # the pool is fragmented: tables are not runs of consecutive ids
        steps = np.diff(t_lib[0, : -(-int(w.seq_lens[0]) // w.bs)])
        assert np.any(steps != 1)


def test_slot_mapping_matches_oracle():
    w = workloads.make("8b", B=8)
    rng = np.random.default_rng(3)
    seq = rng.integers(0, w.B, size=500).astype(np.int32)
    pos = np.array([rng.integers(0, w.seq_lens[s]) for s in seq], dtype=np.int32)
    assert np.array_equal(pa.pa_slot_mapping(w.block_tables, seq, pos, w.bs),
                          oracle.slot_mapping(w.block_tables, seq, pos, w.bs))
    with pytest.raises(pa.PagedAttnError):
        pa.pa_slot_mapping(w.block_tables, np.zeros(1, np.int32), np.array([w.M * w.bs], np.int32), w.bs)


def test_continuous_kv_matches_oracle():
    rng = np.random.default_rng(4)
    for trial in range(20):
        n = int(rng.integers(1, 40))
        prompts = rng.integers(0, 200, size=n)
        outs = rng.integers(1, 120, size=n)
        nb = int(rng.integers(30, 120))
        need = -(-(prompts + outs) // 16)
        if need.max() > nb:
            continue
        seqs = int(rng.integers(1, 10))
        stop = int(rng.integers(-1, 200))
        M = int(need.max())
        a, o = pa.pa_allocator(nb, 16), oracle.Allocator(nb)
        r1 = pa.pa_sched_continuous_kv(a, prompts, outs, seqs, stop, M)
        r2 = oracle.sched_continuous_kv(o, 16, prompts, outs, seqs, stop, M)
        for k in ("iters", "admitted_at", "finished_at", "tables", "lens"):
            assert np.array_equal(np.asarray(r1[k]), np.asarray(r2[k])), k
        assert a.num_free() == o.num_free()
    r = pa.pa_sched_continuous_kv(pa.pa_allocator(1000, 16), [0] * 5, [5, 20, 10, 15, 10], 3)
    assert r["iters"] == 20


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("8b", dict(B=16)), ("70b", dict(B=40)),
                                     ("fp8prefix", dict(B=12, seq_len=600))])
def test_step_slots_match_oracle(name, kw):
    """The decode step's slots (the new token at position len - 1) equal the
    oracle's, including -1 for empty sequences."""
    w = workloads.make(name, **kw)
    tables = oracle.run.tables_of(w)
    lens = np.asarray(w.seq_lens, np.int32).copy()
    lens[:: 5] = 0                      # some sequences get no token this step
    w.seq_lens = lens
    st = oracle.run.OracleStep(w, seqs=[0], tables=tables)
    assert np.array_equal(pa.pa_step_slots(tables, lens, w.bs), st.step_slots)


def test_step_slots_reject_positions_beyond_the_table():
    tables = np.arange(6, dtype=np.int32).reshape(2, 3)
    assert list(pa.pa_step_slots(tables, np.array([48, 1], np.int32), 16)) == [2 * 16 + 15, 3 * 16]
    with pytest.raises(pa.PagedAttnError):
        pa.pa_step_slots(tables, np.array([49, 1], np.int32), 16)


def test_seq_admit_and_append_slot_errors_leave_state_unchanged():
    a = pa.pa_allocator(3, 4)
    c = pa.pa_prefix_cache(a)
    buf = np.zeros(8, np.int32)
    assert pa.pa_seq_admit(a, c, np.arange(9), buf) == (3, 0)           # 9 tokens: 3 blocks
    c.insert(np.arange(9), buf[:3])
    with pytest.raises(pa.PagedAttnError) as e:                          # needs 3 fresh: only cached ones
        pa.pa_seq_admit(a, None, np.arange(100, 109), np.zeros(8, np.int32))
    assert e.value.status == pa.PA_ERR_OOM and a.num_free() == 0
    with pytest.raises(pa.PagedAttnError) as e:                          # too small a buffer
        pa.pa_seq_admit(a, c, np.arange(9), np.zeros(2, np.int32))
    assert e.value.status == pa.PA_ERR_INVALID
    # position 12 opens block 3, but none is free and no cache may give one up
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_seq_append_slot(a, None, buf, 3, 12)
    assert e.value.status == pa.PA_ERR_OOM and list(buf[:3]) == [0, 1, 2]
    with pytest.raises(pa.PagedAttnError) as e:                          # a hole in the block list
        pa.pa_seq_append_slot(a, c, buf, 3, 16)
    assert e.value.status == pa.PA_ERR_INVALID
    # position 5 lands in block 1, which the cache shares (only full blocks are
    # cached: blocks 0 and 1): copy-on-write needs a block, none is free and the
    # cache can give up none (the sequence still holds both) -> OOM, unchanged
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_seq_append_slot(a, c, buf, 3, 5)
    assert e.value.status == pa.PA_ERR_OOM
    assert [a.refcount(i) for i in range(3)] == [2, 2, 1] and list(buf[:3]) == [0, 1, 2]
    # position 9 lands in block 2, held by the sequence alone: written in place
    assert pa.pa_seq_append_slot(a, c, buf, 3, 9) == (2 * 4 + 1, 3, None)
    # free the sequence and re-admit the same tokens: the two cached blocks match
    a.free(buf[:3])
    assert pa.pa_seq_admit(a, c, np.arange(9), buf) == (3, 8)
    assert list(buf[:2]) == [0, 1]
