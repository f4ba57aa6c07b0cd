"""The library's prefix cache, copy-on-write and BlockManager against the oracle.

Bit-exact: every match, allocation, copy-on-write decision, eviction count
and reference count must equal the oracle's on the same operation trace.
"""
import os
import sys

import numpy as np
import pytest

import oracle
import paged_kv_cache_294_gb300 as pa
from oracle.prefix import PrefixCache, cow
from paged_kv_cache_294_gb300.engine import BlockManager
from tests.prefix_sim import OracleManager

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _same_pool(a_lib, a_or, nb):
    assert a_lib.num_free() == a_or.num_free()
    assert [a_lib.refcount(i) for i in range(nb)] == [a_or.refcount(i) for i in range(nb)]


@pytest.mark.parametrize("seed", range(6))
def test_primitives_bit_exact_on_random_traces(seed):
    rng = np.random.default_rng(100 + seed)
    nb, bs = 48, int(rng.choice([1, 2, 4]))
    la, oa = pa.pa_allocator(nb, bs), oracle.Allocator(nb)
    lc, oc = pa.pa_prefix_cache(la), PrefixCache(oa, bs)
    held = []                                          # block lists a "sequence" holds
    for _ in range(400):
        op = rng.integers(0, 5)
        if op == 0:                                    # match and keep the blocks
            toks = [int(x) for x in rng.integers(0, 2, int(rng.integers(0, 16)))]
            cap = int(rng.integers(-1, 5))
            m_l = list(lc.match(toks, None if cap < 0 else cap))
            m_o = oc.match(toks, cap)
            assert m_l == m_o
            held.append(m_l)
        elif op == 1:                                  # allocate and insert
            toks = [int(x) for x in rng.integers(0, 2, int(rng.integers(0, 16)))]
            n = -(-len(toks) // bs)
            if n > oa.num_free():
                continue
            blocks = [int(x) for x in la.alloc(n)]
            assert blocks == [int(x) for x in oa.alloc(n)]
            lc.insert(toks, blocks)
            oc.insert(toks, blocks)
            held.append(blocks)
        elif op == 2 and held:                         # a sequence ends
            blocks = held.pop(int(rng.integers(0, len(held))))
            la.free(blocks)
            oa.free(blocks)
        elif op == 3:
            want = int(rng.integers(0, 6))
            assert lc.evict(want) == oc.evict(want)
        elif op == 4 and held:                         # copy-on-write of a held block
            blocks = held[int(rng.integers(0, len(held)))]
            if not blocks:
                continue
            j = int(rng.integers(0, len(blocks)))
            try:
                r_o = cow(oa, blocks[j])
            except MemoryError:
                with pytest.raises(pa.PagedAttnError):
                    pa.pa_block_cow(la, blocks[j])
                continue
            assert pa.pa_block_cow(la, blocks[j]) == r_o
            blocks[j] = r_o[0]
        assert lc.size() == oc.size()
        _same_pool(la, oa, nb)


@pytest.mark.parametrize("seed", range(4))
def test_block_manager_bit_exact_on_random_serving_traces(seed):
    rng = np.random.default_rng(200 + seed)
    nb, bs = 96, int(rng.choice([2, 4, 16]))
    lib, ora = BlockManager(nb, bs), OracleManager(nb, bs)
    prompts = [[int(x) for x in rng.integers(0, 50, int(rng.integers(1, 5 * bs)))] for _ in range(3)]
    live, next_sid = [], 0
    for _ in range(300):
        op = rng.integers(0, 4)
        if op == 0:                                    # admit: a shared prompt + own suffix
            toks = prompts[int(rng.integers(0, 3))] + [int(x) for x in rng.integers(0, 50, int(rng.integers(0, 3 * bs)))]
            try:
                s_o = ora.add(next_sid, toks)
            except MemoryError:
                with pytest.raises(pa.PagedAttnError):
                    lib.add(next_sid, toks)
                continue
            assert lib.add(next_sid, toks) == s_o
            lib.commit(next_sid)
            ora.commit(next_sid)
            live.append(next_sid)
            next_sid += 1
        elif op == 1 and live:                         # fork
            p = live[int(rng.integers(0, len(live)))]
            lib.fork(next_sid, p)
            ora.fork(next_sid, p)
            live.append(next_sid)
            next_sid += 1
        elif op == 2 and live:                         # decode one token
            sid = live[int(rng.integers(0, len(live)))]
            tok = int(rng.integers(0, 50))
            try:
                r_o = ora.append(sid, tok)
            except MemoryError:
                with pytest.raises(pa.PagedAttnError):
                    lib.append(sid, tok)
                continue
            assert lib.append(sid, tok) == r_o
            if rng.random() < 0.3:
                lib.commit(sid)
                ora.commit(sid)
        elif op == 3 and live:                         # finish
            sid = live.pop(int(rng.integers(0, len(live))))
            lib.free(sid)
            ora.free(sid)
        for sid in live:
            assert lib.blocks[sid] == ora.blocks[sid]
        assert lib.cache.size() == ora.cache.size()
        _same_pool(lib.alloc, ora.alloc, nb)


def test_shared_system_prompt_through_the_library():
    # "LLM Inference Optimization", KV Cache Management: 100 requests with one
    # system prompt share its KV: 144 prompt blocks stored once
    bs, P, R = 16, 2304, 100
    rng = np.random.default_rng(5)
    prompt = [int(x) for x in rng.integers(0, 32000, P)]
    suffix = [int(x) for x in rng.integers(1, 200, R)]
    m = BlockManager(20000, bs)
    written = 0
    for r in range(R):
        toks = prompt + [int(x) for x in rng.integers(32000, 64000, suffix[r])]
        start = m.add(r, toks)
        assert start == (0 if r == 0 else P)
        written += len(toks) - start
        m.commit(r)
    assert m.alloc.num_blocks - m.alloc.num_free() == P // bs + sum(-(-s // bs) for s in suffix)
    assert written == P + sum(suffix)
    assert m.alloc.refcount(m.blocks[0][0]) == R + 1


def test_errors_leave_state_unchanged():
    a = pa.pa_allocator(4, 4)
    c = pa.pa_prefix_cache(a)
    with pytest.raises(pa.PagedAttnError):
        c.insert(list(range(8)), [0, 1])               # blocks not allocated
    assert c.size() == 0 and a.num_free() == 4
    b = [int(x) for x in a.alloc(4)]
    a.share([b[0]])
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_block_cow(a, b[0])                       # shared, and no block free
    assert e.value.status == pa.PA_ERR_OOM
    assert a.refcount(b[0]) == 2 and a.num_free() == 0
    with pytest.raises(pa.PagedAttnError):
        pa.pa_block_cow(a, 99)
    with pytest.raises(pa.PagedAttnError):
        c.evict(-1)
    lib = pa.load()
    assert lib.pa_prefix_cache_create(None) is None
    assert lib.pa_prefix_cache_size(None) == -1


def test_block_manager_evicts_cached_blocks_when_the_pool_runs_dry():
    bs = 4
    m, o = BlockManager(6, bs), OracleManager(6, bs)
    for mgr in (m, o):
        mgr.add(0, list(range(16)))                    # 4 blocks
        mgr.commit(0)
        mgr.free(0)                                    # the cache still holds them
        assert mgr.add(1, [7] * 12) == 0               # needs 3: one cached block evicted
    assert m.blocks[1] == o.blocks[1]
    assert m.cache.size() == o.cache.size() == 3
    assert m.add(2, list(range(8))) == o.add(2, list(range(8))) == 8   # the first two still match
    assert m.blocks[2] == o.blocks[2]


def test_allocator_and_cache_can_be_destroyed_in_either_order():
    lib = pa.load()
    for cache_first in (True, False):
        a = lib.pa_allocator_create(64, 4)
        c = lib.pa_prefix_cache_create(a)
        ids = np.zeros(3, np.int32)
        assert lib.pa_block_alloc(a, 3, ids.ctypes.data) == pa.PA_OK
        toks = np.arange(12, dtype=np.int32)
        assert lib.pa_prefix_insert(c, toks.ctypes.data, 12, ids.ctypes.data, 3) == pa.PA_OK
        assert lib.pa_block_free(a, ids.ctypes.data, 3) == pa.PA_OK
        if cache_first:
            lib.pa_prefix_cache_destroy(c)
            assert lib.pa_allocator_num_free(a) == 64
            lib.pa_allocator_destroy(a)
        else:
            lib.pa_allocator_destroy(a)      # deferred: the cache still holds references
            lib.pa_prefix_cache_destroy(c)   # releases its blocks, then the allocator


def test_interpreter_exit_with_live_cache_objects_in_a_cycle():
    # objects left in a garbage cycle at exit are finalised in any order
    code = r"""
import sys, cProfile, numpy as np
sys.path.insert(0, %r)
from paged_kv_cache_294_gb300.engine import BlockManager
rng = np.random.default_rng(11)
prompts = [[int(x) for x in rng.integers(0, 32000, 2304)] for _ in range(8)]
reqs = [prompts[int(rng.integers(0, 8))] + [int(x) for x in rng.integers(32000, 64000, int(rng.integers(1, 513)))]
        for _ in range(300)]
mgr = BlockManager(40000, 16)
def run():
    for i, toks in enumerate(reqs):
        mgr.add(i, toks); mgr.commit(i); mgr.free(i)
cProfile.run("run()", None)
print("ok")
""" % ROOT
    import subprocess
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().endswith("ok")
