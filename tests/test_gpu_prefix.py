"""Prefix-cached serving on the GPU against the oracle.

A shared system prompt, requests that reuse its cached blocks, forks that
share a parent's partly filled block, then decode steps in which the first
writer of a shared block takes a copy (pa_copy_blocks) and every sequence
appends and attends in one pa_decode_step launch.  The oracle replays the
same trace with its own allocator, prefix cache, copy-on-write, cache and
attention: tables and cache bytes must be identical, outputs within the
attention tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_294_gb300 as pa
import workloads
from oracle.prefix import copy_blocks
from paged_kv_cache_294_gb300.engine import BlockManager, PagedDecodeLayer
from tests.gpu_util import BF16_TOL, FP8_TOL, INT8_TOL, cache_bytes, excess
from tests.prefix_sim import OracleManager

pytestmark = pytest.mark.gpu


def _prefill_positions(table_row, start, n, bs):
    pos = np.arange(start, n, dtype=np.int32)
    return pos, table_row[pos // bs].astype(np.int64) * bs + pos % bs


def _library(sc, splits):
    layer = PagedDecodeLayer(sc.num_blocks, sc.Hq, sc.Hkv, sc.d, sc.bs, sc.kv, "cuda")
    layer.scale = sc.scale
    mgr = BlockManager(sc.num_blocks, sc.bs)
    starts = []
    for r, toks in enumerate(sc.requests):
        start = mgr.add(r, toks)
        starts.append(start)
        if len(toks) > start:
            tab = mgr.table([r], sc.M)
            pos = np.arange(start, len(toks), dtype=np.int32)
            slots = pa.pa_slot_mapping(tab, np.zeros(len(pos), np.int32), pos, sc.bs)
            pa.pa_kv_append(layer.k_cache, layer.v_cache, layer.k_scale, layer.v_scale,
                            sc.k_pre[r][start:].cuda(), sc.v_pre[r][start:].cuda(),
                            torch.from_numpy(slots).cuda())
        mgr.commit(r)
    for i, parent in enumerate(sc.forks):
        mgr.fork(len(sc.requests) + i, parent)
    sids = list(range(sc.n_seq))
    outs, tables, n_copies = [], [], 0
    for s in range(len(sc.tokens)):
        pairs = []
        for sid in sids:
            _, copy = mgr.append(sid, sc.tokens[s][sid])
            if copy is not None:
                pairs.append(copy)
        n_copies += len(pairs)
        layer.copy_blocks(pairs)
        layer.set_batch(mgr.table(sids, sc.M), mgr.lens(sids))
        out = torch.empty((sc.n_seq, sc.Hq, sc.d), dtype=torch.bfloat16, device="cuda")
        layer.fused_step(q=sc.q[s].cuda(), k_new=sc.k_new[s].cuda(), v_new=sc.v_new[s].cuda(), out=out,
                         num_splits=splits)
        outs.append(out)
        tables.append(layer.tables_host.copy())
    torch.cuda.synchronize()
    return layer, starts, [o.float().cpu().numpy().astype(np.float64) for o in outs], tables, n_copies


def _oracle(sc):
    om = OracleManager(sc.num_blocks, sc.bs)
    cache = oracle.Cache(sc.num_blocks, sc.Hkv, sc.d, sc.bs, sc.kv)
    starts = []
    for r, toks in enumerate(sc.requests):
        start = om.add(r, toks)
        starts.append(start)
        if len(toks) > start:
            row = np.asarray(om.blocks[r], dtype=np.int64)
            _, slots = _prefill_positions(row, start, len(toks), sc.bs)
            cache.append(sc.k_pre[r][start:], sc.v_pre[r][start:], slots)
        om.commit(r)
    for i, parent in enumerate(sc.forks):
        om.fork(len(sc.requests) + i, parent)
    sids = list(range(sc.n_seq))
    outs, tables = [], []
    for s in range(len(sc.tokens)):
        slots, pairs = [], []
        for sid in sids:
            slot, copy = om.append(sid, sc.tokens[s][sid])
            slots.append(slot)
            if copy is not None:
                pairs.append(copy)
        copy_blocks(cache, [p[0] for p in pairs], [p[1] for p in pairs])
        cache.append(sc.k_new[s], sc.v_new[s], np.asarray(slots, dtype=np.int64))
        tab = np.full((sc.n_seq, sc.M), -1, dtype=np.int32)
        for i, sid in enumerate(sids):
            tab[i, : len(om.blocks[sid])] = om.blocks[sid]
        lens = np.asarray([len(om.tokens[sid]) for sid in sids], dtype=np.int32)
        outs.append(oracle.decode_attention(cache, sc.q[s], tab, lens, sc.Hq, sc.scale))
        tables.append(tab)
    return cache, starts, outs, tables


@pytest.mark.parametrize("layer_name", ["8b", "fp8prefix", "tiny", "8b-int8", "8b-int4"])
@pytest.mark.parametrize("splits", [0, 2])
def test_prefix_cached_serving_matches_the_oracle(layer_name, splits):
    sc = workloads.serving_scenario(layer_name, steps=35)     # every sequence crosses a block boundary
    pa.pa_get_device_error(clear=True)
    layer, starts, outs, tables, n_copies = _library(sc, splits)
    assert pa.pa_get_device_error() == 0
    cache, o_starts, o_outs, o_tables = _oracle(sc)
    # every request after the first reuses the prompt's full blocks
    assert starts == o_starts and starts[0] == 0 and all(s == 5 * sc.bs for s in starts[1:])
    assert n_copies >= 1                     # the forks shared a partly filled block
    tol = {"fp8": FP8_TOL, "int8": INT8_TOL, "int4": INT8_TOL}.get(sc.kv, BF16_TOL)
    for s in range(len(outs)):
        assert np.array_equal(tables[s], o_tables[s])
        assert excess(outs[s], o_outs[s], tol) <= 1.0, "step %d" % s
    assert np.array_equal(cache_bytes(layer.k_cache), cache.k)
    assert np.array_equal(cache_bytes(layer.v_cache), cache.v)
    if sc.kv != "bf16":
        assert np.array_equal(layer.k_scale.cpu().numpy().view(np.uint32), cache.k_scale.view(np.uint32))
        assert np.array_equal(layer.v_scale.cpu().numpy().view(np.uint32), cache.v_scale.view(np.uint32))


@pytest.mark.parametrize("kv,d,bs", [("bf16", 128, 16), ("bf16", 64, 32), ("fp8", 128, 32), ("int8", 128, 16),
                                      ("int4", 128, 16), ("int4", 128, 32)])
def test_copy_blocks_is_bit_exact(kv, d, bs):
    nb, hkv = 300, 4
    g = torch.Generator(device="cuda")
    g.manual_seed(17)
    dt = {"bf16": torch.bfloat16, "fp8": torch.uint8, "int8": torch.int8, "int4": torch.uint8}[kv]
    row = d // 2 if kv == "int4" else d
    k = torch.randint(0, 255, (nb, hkv, bs, row), generator=g, device="cuda", dtype=torch.uint8).view(dt) \
        if dt != torch.bfloat16 else None
    v = torch.randint(0, 255, (nb, hkv, bs, row), generator=g, device="cuda", dtype=torch.uint8).view(dt) \
        if dt != torch.bfloat16 else None
    if kv == "bf16":
        k = torch.randn((nb, hkv, bs, d), generator=g, device="cuda").to(dt)
        v = torch.randn((nb, hkv, bs, d), generator=g, device="cuda").to(dt)
    ks = torch.rand((nb, hkv), generator=g, device="cuda") if kv != "bf16" else None
    vs = torch.rand((nb, hkv), generator=g, device="cuda") if kv != "bf16" else None
    rng = np.random.default_rng(2)
    perm = rng.permutation(nb)
    src, dst = perm[:100].astype(np.int32), perm[100:200].astype(np.int32)
    k0, v0 = cache_bytes(k).copy(), cache_bytes(v).copy()
    ks0 = ks.cpu().numpy().copy() if ks is not None else None
    pa.pa_get_device_error(clear=True)
    pa.pa_copy_blocks(k, v, ks, vs, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(),
                      kv_dtype=pa.PA_KV_INT4 if kv == "int4" else None)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    k0[dst], v0[dst] = k0[src], v0[src]
    assert np.array_equal(cache_bytes(k), k0) and np.array_equal(cache_bytes(v), v0)
    if ks is not None:
        ks0[dst] = ks0[src]
        assert np.array_equal(ks.cpu().numpy(), ks0)


def test_copy_blocks_skips_out_of_range_ids():
    nb, hkv, bs, d = 8, 2, 16, 128
    k = torch.randn((nb, hkv, bs, d), device="cuda").to(torch.bfloat16)
    v = torch.randn((nb, hkv, bs, d), device="cuda").to(torch.bfloat16)
    k0 = k.clone()
    src = torch.tensor([1, 2, 9], dtype=torch.int32, device="cuda")
    dst = torch.tensor([5, -1, 6], dtype=torch.int32, device="cuda")
    pa.pa_get_device_error(clear=True)
    pa.pa_copy_blocks(k, v, None, None, src, dst)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() & pa.PA_DEVERR_BLOCK_ID
    assert torch.equal(k[5], k0[1])
    untouched = [0, 1, 2, 3, 4, 6, 7]
    assert torch.equal(k[untouched], k0[untouched])
    # nothing to copy, and argument errors before any launch
    pa.pa_copy_blocks(k, v, None, None, src[:0], dst[:0])
    with pytest.raises(pa.PagedAttnError):
        pa.pa_copy_blocks(k, v, torch.zeros((nb, hkv), device="cuda"), None, src, dst)
