"""pa_decode_step_shared (shared prefixes read once per chunk of sequences)
against the fp64 oracle.

The plan comes from pa_share_plan on the library's tables.  The outputs must
match the oracle within the parity bound (the partial sums are ordered
differently from pa_decode_step's); the cache bytes the fused step writes must
equal the oracle's append bit for bit; the split-K counters must return to
zero after every call, including calls with a corrupted plan, which the
kernel detects, reports and attends without sharing.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle.run
import paged_kv_cache_294_gb300 as pa
import workloads
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer
from tests.gpu_util import cache_bytes, excess, oracle_out, tol, worst

pytestmark = pytest.mark.gpu
R = pa.PA_SHARE_MAX_ROWS


def _counters_zero(layer, num_splits=0):
    need = pa.pa_decode_shared_workspace_bytes(layer.B, layer.Hq, layer.Hkv, layer.d, layer.M, num_splits,
                                               layer.share_plan["max_chunk_blocks"])
    tail = layer.workspace[:need].view(torch.int32)[-((layer.B * layer.Hkv + 63) // 64 * 64):]
    return int(tail.abs().sum()) == 0


def _check(w, layer, S=0, append=True):
    pa.pa_get_device_error(clear=True)
    layer.shared_step(append=append, num_splits=S)
    torch.cuda.synchronize()
    flags = pa.pa_get_device_error()
    st, ref = oracle_out(w, tables=layer.tables_host) if append else (None, None)
    got = layer.out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert excess(got, ref, tol(w)) <= 1.0, worst(got, ref, tol(w))
    assert _counters_zero(layer, S)
    return st, flags


def _shared_synthetic(groups, indep, Hq, Hkv, bs, kv, seed):
    """groups: [(shared_blocks, [member lengths])], indep: [lengths].  Each
    group's shared blocks are allocated once and written once (through its
    first member); every member then has blocks of its own."""
    rng = np.random.default_rng(seed)
    lens, rows, skip = [], [], []
    nxt = 0
    for shb, mlens in groups:
        shared = list(range(nxt, nxt + shb))
        nxt += shb
        for i, L in enumerate(mlens):
            assert L > shb * bs
            own = -(-L // bs) - shb
            rows.append(shared + list(range(nxt, nxt + own)))
            nxt += own
            lens.append(L)
            skip.append(0 if i == 0 else shb * bs)
    for L in indep:
        nb = -(-L // bs)
        rows.append(list(range(nxt, nxt + nb)))
        nxt += nb
        lens.append(L)
        skip.append(0)
    nb_pool = nxt + 9
    perm = rng.permutation(nb_pool).astype(np.int32)
    M = max(len(r) for r in rows)
    tables = np.full((len(rows), M), -1, np.int32)
    for b, r in enumerate(rows):
        tables[b, :len(r)] = perm[np.asarray(r, dtype=np.int64)]
    lens = np.asarray(lens, np.int32)
    fs, fp = workloads._history(lens, np.asarray(skip))
    vals = workloads._values(seed, len(fs), len(lens), Hq, Hkv, 128, "cpu")
    return workloads.Workload(name="shared-synthetic", Hq=Hq, Hkv=Hkv, d=128, bs=bs, kv=kv, B=len(lens),
                              num_blocks=nb_pool, M=M, scale=1.0 / math.sqrt(128), seq_lens=lens,
                              block_tables=tables, trace=None, target_rids=None, fill_seq=fs, fill_pos=fp, **vals)


def test_full_size_shared_prefix_workload_every_output():
    w = workloads.make("fp8prefix", device="cuda")
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    plan = layer.plan_sharing()
    assert len(plan["chunk_blocks"]) == 13
    pa.pa_get_device_error(clear=True)
    layer.shared_step()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    st = oracle.run.OracleStep(w, tables=layer.tables_host)
    st.append()
    ref = st.decode(threads=os.cpu_count() or 1)
    got = layer.out.float().cpu().numpy().astype(np.float64)
    assert excess(got, ref, tol(w)) <= 1.0, worst(got, ref, tol(w))
    assert np.array_equal(cache_bytes(layer.k_cache), st.cache.k)
    assert np.array_equal(cache_bytes(layer.v_cache), st.cache.v)
    assert np.array_equal(layer.k_scale.cpu().numpy().view(np.uint32), st.cache.k_scale.view(np.uint32))
    assert _counters_zero(layer)
    # the same step again (the append rewrites the same bytes): same outputs
    first = layer.out.clone()
    layer.shared_step()
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), layer.out.view(torch.int16))


@pytest.mark.parametrize("S", [0, 1, 3])
def test_shared_prefix_workload_small(S):
    w = workloads.make("fp8prefix", B=40, seq_len=900)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    assert len(layer.plan_sharing()["chunk_blocks"]) > 0
    _, flags = _check(w, layer, S)
    assert flags == 0


@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8", "int4"])
@pytest.mark.parametrize("Hq,Hkv,bs", [(8, 8, 16), (16, 8, 32), (16, 4, 16), (32, 4, 32), (24, 8, 16), (12, 2, 32)])
def test_shared_groups_head_layouts_and_caches(kv, Hq, Hkv, bs):
    """Groups larger and smaller than a chunk, one-block and long own parts,
    a new token opening a fresh block, independent sequences beside them."""
    groups = [(3, [3 * bs + 1, 3 * bs + 7, 5 * bs, 4 * bs + 9, 3 * bs + 2, 9 * bs + 1, 3 * bs + 3, 3 * bs + 5,
                   6 * bs + 1, 3 * bs + 10]),
              (7, [7 * bs + 4, 20 * bs + 3]),
              (1, [bs + 1, bs + 2, 2 * bs])]
    w = _shared_synthetic(groups, [5, 2 * bs + 3, 40 * bs], Hq, Hkv, bs, kv, seed=Hq + Hkv + bs)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    plan = layer.plan_sharing()
    # a chunk holds 8 / G sequences (rounded down): with G > 4 nothing is shared
    assert len(plan["chunk_blocks"]) >= 3 if 8 // (Hq // Hkv) >= 2 else len(plan["chunk_blocks"]) == 0
    for S in (0, 2):
        _, flags = _check(w, layer, S)
        assert flags == 0
        # the step re-appended the same tokens; rebuild so the next check starts from the same cache
        layer = PagedDecodeLayer.from_workload(w, "cuda")
        layer.plan_sharing()


def test_attention_only_matches_pa_decode_attention():
    w = workloads.make("fp8prefix", B=40, seq_len=900)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    layer.append_step()
    ref = layer.decode().clone()
    layer.plan_sharing()
    layer.shared_step(append=False)
    torch.cuda.synchronize()
    a, b = layer.out.float().cpu().numpy(), ref.float().cpu().numpy()
    assert excess(a.astype(np.float64), b.astype(np.float64), 2 * tol(w)) <= 1.0
    assert _counters_zero(layer)


@pytest.mark.parametrize("fault", ["wrong_slot", "duplicate", "too_long", "bad_chunk"])
def test_corrupted_plans_are_reported_and_attended_without_sharing(fault):
    w = workloads.make("fp8prefix", B=40, seq_len=900)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    layer.plan_sharing()
    co, cm, cb = layer.chunk_of.clone(), layer.chunk_members.clone(), layer.chunk_blocks.clone()
    if fault == "wrong_slot":
        co[1] = co[2]                       # sequence 1 claims sequence 2's slot
    elif fault == "duplicate":
        cm[0, 1] = cm[0, 0]                 # a member listed twice
    elif fault == "too_long":
        cb[0] = int((w.seq_lens[0] - 1) // w.bs) + 1   # reaches the block of the members' newest token
        layer.share_plan = dict(layer.share_plan, max_chunk_blocks=int(cb[0]))
    else:
        co[3] = R * 1000                    # a chunk that does not exist
    layer.chunk_of, layer.chunk_members, layer.chunk_blocks = co, cm, cb
    _, flags = _check(w, layer)
    assert flags & pa.PA_DEVERR_BLOCK_ID
    # a correct plan afterwards, on the same workspace and layout: the
    # counters were left at zero
    layer2 = PagedDecodeLayer.from_workload(w, "cuda")
    layer2.plan_sharing()
    layer2.share_plan = dict(layer2.share_plan, max_chunk_blocks=layer.share_plan["max_chunk_blocks"])
    layer2.workspace = layer.workspace
    _, flags = _check(w, layer2)
    assert flags == 0
