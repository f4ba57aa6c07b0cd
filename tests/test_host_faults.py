"""Host-side failure injection: an allocation the pool refuses.

pa_allocator_fail_nth_alloc makes the n-th later allocation fail with
PA_ERR_OOM while blocks are free, so that every path that handles a refused
allocation ("KV cache memory math" and "Static versus continuous scheduling":
a request the pool cannot hold is refused) runs on purpose: nothing is taken,
references taken before the failure are given back, and the caller's state is
what it was.  Also the split-count override from the environment.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import paged_kv_cache_294_gb300 as pa
from paged_kv_cache_294_gb300.engine import BlockManager

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _pool(a, nb):
    return a.num_free(), [a.refcount(i) for i in range(nb)]


def test_nth_alloc_fails_once_and_takes_nothing():
    a = pa.pa_allocator(16, 4)
    a.fail_nth_alloc(3)
    assert list(a.alloc(1)) == [0]
    assert list(a.alloc(0)) == []                     # asks for nothing: not counted
    assert list(a.alloc(2)) == [1, 2]
    before = _pool(a, 16)
    with pytest.raises(pa.PagedAttnError) as e:
        a.alloc(1)
    assert e.value.status == pa.PA_ERR_OOM and _pool(a, 16) == before
    assert list(a.alloc(2)) == [3, 4]                 # one shot
    a.fail_nth_alloc(1)
    a.fail_nth_alloc(0)                               # disarmed
    assert list(a.alloc(1)) == [5]
    a.fail_nth_alloc(-7)
    assert list(a.alloc(1)) == [6]
    assert pa.load().pa_allocator_fail_nth_alloc(None, 1) == pa.PA_ERR_INVALID


def test_refused_admission_returns_the_matched_prefix():
    bs = 4
    a = pa.pa_allocator(12, bs)
    c = pa.pa_prefix_cache(a)
    buf = np.zeros(8, np.int32)
    assert pa.pa_seq_admit(a, c, np.arange(10), buf) == (3, 0)
    c.insert(np.arange(10), buf[:3])                  # caches the two full blocks
    a.free(buf[:3])
    before = _pool(a, 12)
    a.fail_nth_alloc(1)
    out = np.full(8, -5, np.int32)
    with pytest.raises(pa.PagedAttnError) as e:       # matches two blocks, then needs one more
        pa.pa_seq_admit(a, c, np.arange(11), out)
    assert e.value.status == pa.PA_ERR_OOM
    assert _pool(a, 12) == before and c.size() == 2   # the matched references went back
    assert pa.pa_seq_admit(a, c, np.arange(11), out) == (3, 8)
    assert list(out[:2]) == list(buf[:2])


def test_refused_append_and_copy_on_write_leave_the_sequence():
    bs = 4
    a = pa.pa_allocator(8, bs)
    buf = np.zeros(8, np.int32)
    assert pa.pa_seq_admit(a, None, np.arange(8), buf) == (2, 0)
    before = _pool(a, 8)
    a.fail_nth_alloc(1)                               # position 8 opens block 2
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_seq_append_slot(a, None, buf, 2, 8)
    assert e.value.status == pa.PA_ERR_OOM and _pool(a, 8) == before and list(buf[:2]) == [0, 1]
    assert pa.pa_seq_append_slot(a, None, buf, 2, 8) == (2 * bs, 3, None)
    # block 1 shared by a fork: writing into it needs a private copy
    a.share(buf[1:2])
    before = _pool(a, 8)
    a.fail_nth_alloc(1)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_block_cow(a, int(buf[1]))
    assert e.value.status == pa.PA_ERR_OOM and _pool(a, 8) == before
    assert pa.pa_block_cow(a, int(buf[1])) == (3, True)


def test_block_manager_state_survives_a_refusal():
    m = BlockManager(32, 4)
    m.add(0, list(range(9)))
    m.commit(0)
    before = _pool(m.alloc, 32)
    m.alloc.fail_nth_alloc(1)
    with pytest.raises(pa.PagedAttnError):
        m.add(1, list(range(20)))                     # shares two blocks, needs three more
    assert 1 not in m.blocks and _pool(m.alloc, 32) == before
    assert m.add(1, list(range(20))) == 8
    m.alloc.fail_nth_alloc(1)
    with pytest.raises(pa.PagedAttnError):
        m.append(0, 99)                               # position 9 sits in block 2 (private): no alloc
        m.append(0, 99)
        m.append(0, 99)
        m.append(0, 99)                               # position 12 opens a block: refused
    assert len(m.tokens(0)) == 12 and len(m.blocks[0]) == 3
    slot, copy = m.append(0, 99)
    assert len(m.tokens(0)) == 13 and len(m.blocks[0]) == 4 and copy is None


def test_scheduler_requeues_a_refused_admission():
    # three 5-token requests, three slots: all start at iteration 0 and end at 4
    base = pa.pa_sched_continuous_kv(pa.pa_allocator(64, 16), [0, 0, 0], [5, 5, 5], 3, -1, 1)
    assert list(base["admitted_at"]) == [0, 0, 0] and base["iters"] == 5
    a = pa.pa_allocator(64, 16)
    a.fail_nth_alloc(2)                               # request 1's reservation is refused
    r = pa.pa_sched_continuous_kv(a, [0, 0, 0], [5, 5, 5], 3, -1, 1)
    assert list(r["admitted_at"]) == [0, 1, 1]        # it waits, and request 2 behind it
    assert list(r["finished_at"]) == [4, 5, 5] and r["iters"] == 6
    assert a.num_free() == 64


def test_scheduler_refused_with_nothing_running_takes_nothing():
    a = pa.pa_allocator(64, 16)
    a.fail_nth_alloc(1)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_sched_continuous_kv(a, [10, 0], [5, 5], 2, -1, 1)
    assert e.value.status == pa.PA_ERR_OOM and a.num_free() == 64
    # a request that can never fit stays an argument error
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_sched_continuous_kv(pa.pa_allocator(1, 16), [40], [5], 1, -1, 4)
    assert e.value.status == pa.PA_ERR_INVALID


@pytest.mark.parametrize("env,expect", [("3", [3, 3, 5]), ("abc", None), ("0", None), ("600", None)])
def test_force_splits_from_the_environment(env, expect):
    """PA_FORCE_SPLITS stands in for the automatic split count only; an
    explicit count wins, and a value outside 1 .. 512 is ignored."""
    code = ("import paged_kv_cache_294_gb300 as pa; lib = pa.load(); "
            "print(lib.pa_decode_resolve_splits(4, 8, 8192, 0), lib.pa_decode_resolve_splits(64, 8, 256, 0), "
            "lib.pa_decode_resolve_splits(64, 8, 256, 5))")
    run = lambda e: subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                                   env=e, check=True).stdout.split()
    plain = {k: v for k, v in os.environ.items() if k != "PA_FORCE_SPLITS"}
    auto = [int(x) for x in run(plain)]
    got = [int(x) for x in run(dict(plain, PA_FORCE_SPLITS=env))]
    assert got == (expect if expect is not None else auto)
    assert auto[2] == 5


def test_refused_copy_on_write_of_a_forked_block():
    """A fork shares the parent's partial last block; the parent's next token
    needs a private copy of it.  A refused copy leaves both sequences as they
    were; with cache-only blocks to give up, the library evicts one and tries
    again."""
    m = BlockManager(16, 4)
    m.add(0, list(range(6)))                          # blocks: full [0..3], partial [4, 5]
    m.fork(1, 0)
    before = _pool(m.alloc, 16)
    blocks0, blocks1 = list(m.blocks[0]), list(m.blocks[1])
    m.alloc.fail_nth_alloc(1)
    with pytest.raises(pa.PagedAttnError) as e:       # nothing the cache could give up
        m.append(0, 99)
    assert e.value.status == pa.PA_ERR_OOM and _pool(m.alloc, 16) == before
    assert list(m.blocks[0]) == blocks0 and list(m.blocks[1]) == blocks1 and len(m.tokens(0)) == 6
    # a finished, cached sequence leaves blocks only the cache holds
    m.add(2, list(range(100, 108)))
    m.commit(2)
    m.free(2)
    assert m.cache.size() == 2
    m.alloc.fail_nth_alloc(1)
    slot, copy = m.append(0, 99)                      # refused once, one cached block evicted, then copied
    assert copy is not None and copy[0] == blocks0[1] and m.cache.size() == 1
    assert m.blocks[1] == blocks1 and m.alloc.refcount(blocks0[1]) == 1
