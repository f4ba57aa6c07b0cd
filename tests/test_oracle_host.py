"""Pins for the oracle's host-side definitions: accounting, scheduler, allocator, slots.

Expected values are the numbers the pages print (tests/golden/pages_numbers.txt,
each line citing its page and section) and invariants any correct
implementation satisfies.
"""
import itertools

import numpy as np
import pytest

import oracle
from tests.golden.load import page_numbers


def test_page_numbers():
    n = 0
    for kind, v in page_numbers():
        if kind == "kv_bytes":
            assert oracle.kv_bytes(*v[:6]) == v[6], v
        elif kind == "blocks":
            assert oracle.blocks_for_tokens(v[0], v[1]) == v[2], v
        elif kind == "table":
            seq_len, cap, ids = v[0], v[1], v[2:]
            assert len(ids) * 16 == cap
            assert oracle.blocks_for_tokens(seq_len, 16) == len(ids)
        elif kind == "sched":
            st, co, slots, lens = v[0], v[1], v[2], v[3:]
            assert oracle.sched_static(lens, slots) == st
            assert oracle.sched_continuous(lens, slots) == co
        n += 1
    assert n >= 14


def test_kv_bytes_decimal_vs_binary_reading():
    # 128,000 tokens of Llama-3-70B at 327,680 B/token: the page's "41 GB" (decimal)
    b = oracle.kv_bytes(80, 8, 128, 16, 128000, 1)
    assert 41e9 <= b < 42e9
    # the pitfall's 256 x 4096 x 320KB: exact bytes with 327,680 B/token; the page's
    # "335 GB" is the same product with 1 KB = 1000 B (320,000 B/token)
    assert oracle.kv_bytes(80, 8, 128, 16, 4096, 256) == 256 * 4096 * 327680
    assert 256 * 4096 * 320000 // 10 ** 9 == 335


def test_kv_bytes_dtype_and_gqa_ratios():
    bf16 = oracle.kv_bytes(80, 8, 128, 16, 1000, 3)
    assert oracle.kv_bytes(80, 8, 128, 8, 1000, 3) * 2 == bf16       # fp8 / int8: 1 byte
    assert oracle.kv_bytes(80, 8, 128, 4, 1000, 3) * 4 == bf16       # int4: 0.5 byte
    assert oracle.kv_bytes(80, 64, 128, 16, 1000, 3) == 8 * bf16     # MHA 64 heads vs GQA 8: 8x
    assert oracle.kv_bytes(80, 1, 128, 16, 1000, 3) * 8 == bf16      # MQA: one KV head


def test_blocks_are_ceil():
    for bs in (1, 2, 16, 32):
        for n in range(0, 200):
            k = oracle.blocks_for_tokens(n, bs)
            assert k * bs >= n and (k == 0 or (k - 1) * bs < n)


def _brute_continuous(lens, slots):
    """Event-by-event simulation with explicit slot objects (a different formulation)."""
    slot_left = [0] * slots
    queue = list(lens)
    t = 0
    while queue or any(slot_left):
        for s in range(slots):
            if slot_left[s] == 0 and queue:
                slot_left[s] = queue.pop(0)
        slot_left = [max(0, x - 1) for x in slot_left]
        t += 1
    return t


def test_scheduler_invariants_and_bruteforce():
    rng = np.random.default_rng(11)
    for _ in range(300):
        n = int(rng.integers(0, 12))
        lens = [int(x) for x in rng.integers(1, 30, size=n)]
        slots = int(rng.integers(1, 6))
        st = oracle.sched_static(lens, slots)
        co = oracle.sched_continuous(lens, slots)
        assert co == _brute_continuous(lens, slots)
        assert st == sum(max(lens[i:i + slots]) for i in range(0, n, slots))
        if n:
            assert co <= st
            assert co >= max(lens) and co * slots >= sum(lens)
            if slots >= n:
                assert co == st == max(lens)


@pytest.mark.parametrize("fn", [oracle.sched_static, oracle.sched_continuous])
def test_scheduler_rejects_bad_domain(fn):
    with pytest.raises(ValueError):
        fn([5, 3], 0)
    with pytest.raises(ValueError):
        fn([5, 0], 2)
    assert fn([], 1) == 0


def test_allocator_lowest_id_and_refcounts():
    a = oracle.Allocator(8)
    assert list(a.alloc(3)) == [0, 1, 2]
    a.free([1])
    assert list(a.alloc(2)) == [1, 3]
    assert a.num_free() == 4
    with pytest.raises(MemoryError):
        a.alloc(5)
    assert a.num_free() == 4                       # all or nothing
    a.share([0, 2])
    assert a.refcount(0) == 2
    a.free([0, 2])
    assert a.refcount(0) == 1 and a.num_free() == 4
    a.free([0, 2])
    assert a.num_free() == 6
    with pytest.raises(ValueError):
        a.free([0])                                 # double free
    with pytest.raises(ValueError):
        a.free([1, 1])                              # more drops than references: nothing changes
    assert a.refcount(1) == 1
    with pytest.raises(ValueError):
        a.share([5])                                # cannot share a free block
    with pytest.raises(ValueError):
        a.free([8])
    assert list(a.alloc(0)) == []


def test_allocator_matches_set_model():
    """Against a set-based model: the free set's smallest members are handed out."""
    rng = np.random.default_rng(5)
    a = oracle.Allocator(50)
    ref = {i: 0 for i in range(50)}
    held = []
    for _ in range(400):
        op = rng.integers(3)
        if op == 0:
            n = int(rng.integers(0, 9))
            free = sorted(i for i, c in ref.items() if c == 0)
            if n > len(free):
                with pytest.raises(MemoryError):
                    a.alloc(n)
                continue
            got = list(a.alloc(n))
            assert got == free[:n]
            for i in got:
                ref[i] = 1
            held.append(got)
        elif op == 1 and held:
            ids = held.pop(int(rng.integers(len(held))))
            a.free(ids)
            for i in ids:
                ref[i] -= 1
        elif op == 2 and held:
            ids = held[int(rng.integers(len(held)))]
            a.share(ids)
            for i in ids:
                ref[i] += 1
            held.append(list(ids))
        assert a.num_free() == sum(1 for c in ref.values() if c == 0)


def test_slot_mapping_page_examples():
    # request A of the PagedAttention example: blocks [12, 7, 28, 4]
    t = np.array([[12, 7, 28, 4]], np.int32)
    pos = np.array([0, 15, 16, 33, 49], np.int32)
    s = oracle.slot_mapping(t, np.zeros(5, np.int32), pos, 16)
    assert list(s) == [12 * 16, 12 * 16 + 15, 7 * 16, 28 * 16 + 1, 4 * 16 + 1]
    with pytest.raises(ValueError):
        oracle.slot_mapping(t, np.zeros(1, np.int32), np.array([64], np.int32), 16)


def test_bf16_append_is_an_exact_copy():
    rng = np.random.default_rng(9)
    c = oracle.Cache(6, 3, 8, 4)
    k = rng.integers(0, 1 << 16, size=(5, 3, 8)).astype(np.uint16)
    v = rng.integers(0, 1 << 16, size=(5, 3, 8)).astype(np.uint16)
    slots = np.array([9, -1, 0, 23, 10], np.int64)
    c.append(k, v, slots)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(c.k[s // 4, :, s % 4], k[t]) and np.array_equal(c.v[s // 4, :, s % 4], v[t])
    written = {(s // 4, s % 4) for s in slots if s >= 0}
    for blk, off in itertools.product(range(6), range(4)):
        if (blk, off) not in written:
            assert np.all(c.k[blk, :, off] == 0)
    with pytest.raises(ValueError):
        c.append(k[:1], v[:1], np.array([24], np.int64))


def test_continuous_kv_reduces_to_the_pages_scheduler():
    lens = [5, 20, 10, 15, 10]
    a = oracle.Allocator(1000)
    r = oracle.sched_continuous_kv(a, 16, [0] * 5, lens, 3)
    assert r["iters"] == 20 == oracle.sched_continuous(lens, 3)
    assert a.num_free() == 1000                      # every block returned at the end
    assert list(r["admitted_at"]) == [0, 0, 0, 5, 10]
    assert list(r["finished_at"]) == [4, 19, 9, 19, 19]


def test_continuous_kv_memory_bound_admission_acts_as_slots():
    """Every request reserves 2 blocks of a 4-block pool: at most 2 run at once."""
    rng = np.random.default_rng(3)
    for _ in range(30):
        n = int(rng.integers(1, 9))
        outs = [int(x) for x in rng.integers(1, 17, size=n)]
        prompts = [32 - o for o in outs]            # prompt + out = 32 tokens = 2 blocks of 16
        a = oracle.Allocator(4)
        r = oracle.sched_continuous_kv(a, 16, prompts, outs, 8)
        assert r["iters"] == oracle.sched_continuous(outs, 2)


def test_continuous_kv_snapshot_tables_and_lengths():
    a = oracle.Allocator(10)
    r = oracle.sched_continuous_kv(a, 4, [3, 6, 2], [4, 3, 5], 2, stop_iter=2, M=3)
    # request 0 reserves ceil(7/4)=2 blocks [0,1]; request 1 ceil(9/4)=3 blocks [2,3,4];
    # request 2 waits for a sequence slot
    assert r["iters"] == 2
    assert list(r["lens"]) == [3 + 2, 6 + 2, 0]
    assert r["tables"].tolist() == [[0, 1, -1], [2, 3, 4], [-1, -1, -1]]
    assert list(r["admitted_at"]) == [0, 0, -1]
    with pytest.raises(ValueError):
        oracle.sched_continuous_kv(oracle.Allocator(2), 4, [20], [1], 1)   # can never fit
