"""pa_prefill_attention (chunked prefill / speculative verify) against the oracle,
on the bf16 cache and on the coded caches (e4m3, int8, int4 with per-(block,
head) scales: tolerance 5e-2 for e4m3 against the oracle on the stored codes,
1e-2 otherwise)."""
import numpy as np
import pytest
import torch

import oracle
import oracle.run
import paged_kv_cache_294_gb300 as pa
import workloads
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer
from tests.gpu_util import BF16_TOL, excess, tol, worst

pytestmark = pytest.mark.gpu


def _gpu(w, max_q=None, tables=None, layer=None):
    layer = PagedDecodeLayer.from_workload(w, "cuda") if layer is None else layer
    q = w.q_chunk.cuda()
    out = torch.full_like(q, float("nan"))
    pa.pa_prefill_attention(out, q, layer.k_cache, layer.v_cache, layer.k_scale, layer.v_scale,
                            layer.block_tables if tables is None else tables, layer.seq_lens,
                            torch.from_numpy(w.q_start).cuda(), w.max_q if max_q is None else max_q, w.scale)
    torch.cuda.synchronize()
    return layer, out.float().cpu().numpy().astype(np.float64)


def _oracle(w, tables):
    st = oracle.run.OracleStep(w, tables=tables)
    return oracle.prefill_attention(st.cache, w.q_chunk, st.tables, w.seq_lens, w.q_start, w.Hq, w.scale,
                                    threads=8)


SHAPES = [("8b", None, None, None), ("70b", None, None, None), ("8b", 8, 8, 32), ("8b", 16, 8, 32),
          ("8b", 32, 2, 16)]
MIXES = [([0, 100, 517, 1000, 3, 40], [300, 28, 129, 5, 1, 0]),     # whole prompt, chunks, verify, one token, empty
         ([0, 0], [128, 256]),                                          # tile-aligned
         ([250, 1333, 7, 64], [5, 5, 5, 5])]                            # verify passes (K = 4)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("mix", range(len(MIXES)))
def test_prefill_matches_the_oracle(shape, mix):
    layer_name, Hq, Hkv, bs = shape
    ctx, chunk = MIXES[mix]
    w = workloads.make_prefill(layer_name, ctx, chunk, seed=mix + 3, Hq=Hq, Hkv=Hkv, bs=bs)
    pa.pa_get_device_error(clear=True)
    layer, got = _gpu(w)
    assert pa.pa_get_device_error() == 0
    ref = _oracle(w, layer.tables_host)
    assert excess(got, ref, BF16_TOL) <= 1.0, worst(got, ref, BF16_TOL)


def test_long_chunk_sampled_rows():
    # a 2048-token chunk after 4096 cached tokens, and a whole 6000-token prompt
    w = workloads.make_prefill("8b", [4096, 0], [2048, 6000], seed=21)
    layer, got = _gpu(w)
    rng = np.random.default_rng(0)
    rows = sorted(set(int(x) for x in rng.integers(0, int(w.q_start[-1]), 24)) | {0, 2047, 2048, 8047})
    caches = {}
    for r in rows:
        b = int(np.searchsorted(w.q_start, r, side="right") - 1)
        C = int(w.q_start[b + 1] - w.q_start[b])
        pos = int(w.seq_lens[b]) - C + (r - int(w.q_start[b]))
        # row r alone: a one-token chunk at its position over a cache truncated after it
        if b not in caches:
            caches[b] = oracle.run.OracleStep(w, seqs=[b], tables=layer.tables_host)
        st = caches[b]
        ref = oracle.prefill_attention(st.cache, w.q_chunk[r:r + 1], st.tables[b:b + 1],
                                       np.array([pos + 1]), np.array([0, 1]), w.Hq, w.scale)
        assert excess(got[r:r + 1], ref, BF16_TOL) <= 1.0, "row %d" % r


def test_stale_nan_rows_and_blocks_are_never_read_into_outputs():
    w = workloads.make_prefill("8b", [20, 3, 100], [13, 30, 7], seed=5)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device="cuda")
    used = set()
    for b, n in enumerate(w.seq_lens):
        nb = -(-int(n) // w.bs)
        used.update(int(x) for x in layer.tables_host[b, :nb])
        last, rows = int(layer.tables_host[b, nb - 1]), int(n) - (nb - 1) * w.bs
        layer.k_cache[last, :, rows:] = nan
        layer.v_cache[last, :, rows:] = nan
    for blk in range(w.num_blocks):
        if blk not in used:
            layer.k_cache[blk] = nan
            layer.v_cache[blk] = nan
    _, got = _gpu(w, layer=layer)
    st = oracle.run.OracleStep(w, tables=layer.tables_host)
    ref = oracle.prefill_attention(st.cache, w.q_chunk, st.tables, w.seq_lens, w.q_start, w.Hq, w.scale)
    assert np.isfinite(got).all()
    assert excess(got, ref, BF16_TOL) <= 1.0, worst(got, ref, BF16_TOL)


def test_one_token_chunks_agree_with_decode():
    w = workloads.make_prefill("8b", [17, 200, 999, 0], [1, 1, 1, 1], seed=9)
    layer, got = _gpu(w)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    layer.decode(q=w.q_chunk.cuda(), out=out)
    dec = out.float().cpu().numpy().astype(np.float64)
    ref = _oracle(w, layer.tables_host)
    assert excess(got, ref, BF16_TOL) <= 1.0 and excess(dec, ref, BF16_TOL) <= 1.0


def test_chunk_longer_than_max_q_is_flagged_and_skipped():
    w = workloads.make_prefill("8b", [10, 10], [40, 8], seed=2)
    pa.pa_get_device_error(clear=True)
    layer, got = _gpu(w, max_q=8)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_SEQ_LEN
    ref = _oracle(w, layer.tables_host)
    assert np.isnan(got[:40]).all()                           # sequence 0 untouched
    assert excess(got[40:], ref[40:], BF16_TOL) <= 1.0, worst(got[40:], ref[40:], BF16_TOL)


def test_out_of_range_block_id_is_flagged_and_other_sequences_are_exact():
    w = workloads.make_prefill("8b", [100, 100], [30, 30], seed=4)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    tables = layer.block_tables.clone()
    tables[0, 1] = 10 ** 7
    pa.pa_get_device_error(clear=True)
    _, got = _gpu(w, tables=tables, layer=layer)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_BLOCK_ID
    assert np.isfinite(got[:30]).all()
    ref = _oracle(w, layer.tables_host)
    assert excess(got[30:], ref[30:], BF16_TOL) <= 1.0, worst(got[30:], ref[30:], BF16_TOL)


def test_unsupported_shapes_and_bad_arguments():
    w = workloads.make_prefill("tiny", [4], [4], seed=1)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    q = w.q_chunk.cuda()
    qs = torch.from_numpy(w.q_start).cuda()
    with pytest.raises(pa.PagedAttnError) as e:               # head_dim 64
        pa.pa_prefill_attention(torch.empty_like(q), q, layer.k_cache, layer.v_cache, None, None,
                                layer.block_tables, layer.seq_lens, qs, 4, w.scale)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    w = workloads.make_prefill("8b", [4], [4], seed=1)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    q = w.q_chunk.cuda()
    with pytest.raises(pa.PagedAttnError):
        pa.pa_prefill_attention(torch.empty_like(q), q, layer.k_cache, layer.v_cache, None, None,
                                layer.block_tables, layer.seq_lens, torch.from_numpy(w.q_start).cuda(), -1,
                                w.scale)


def _sampled_rows_match(w, layer, got, rows):
    caches = {}
    for r in rows:
        b = int(np.searchsorted(w.q_start, r, side="right") - 1)
        C = int(w.q_start[b + 1] - w.q_start[b])
        pos = int(w.seq_lens[b]) - C + (r - int(w.q_start[b]))
        if b not in caches:
            caches[b] = oracle.run.OracleStep(w, seqs=[b], tables=layer.tables_host)
        ref = oracle.prefill_attention(caches[b].cache, w.q_chunk[r:r + 1], caches[b].tables[b:b + 1],
                                       np.array([pos + 1]), np.array([0, 1]), w.Hq, w.scale)
        assert excess(got[r:r + 1], ref, BF16_TOL) <= 1.0, "row %d" % r


@pytest.mark.parametrize("layer_name", ["8b", "70b"])
def test_bench_prefill_configuration_sampled(layer_name):
    # the batch bench.py times: 16 sequences of 2048 cached tokens + a 2048-token chunk
    w = workloads.make_prefill(layer_name, [2048] * 16, [2048] * 16, seed=31, device="cuda")
    layer, got = _gpu(w)
    rng = np.random.default_rng(1)
    rows = sorted(set(int(x) for x in rng.integers(0, int(w.q_start[-1]), 20)) | {0, 2047, 16 * 2048 - 1})
    _sampled_rows_match(w, layer, got, rows)


@pytest.mark.parametrize("layer_name", ["8b", "70b"])
def test_bench_verify_configuration_sampled(layer_name):
    # the verify batch bench.py times: 64 sequences, U[128, 4096] cached, 4 proposals + 1
    rng = np.random.default_rng(7)
    ctx = [int(x) for x in rng.integers(128, 4097, 64)]
    w = workloads.make_prefill(layer_name, ctx, [5] * 64, seed=31, device="cuda")
    layer, got = _gpu(w)
    rows = sorted(set(int(x) for x in np.random.default_rng(2).integers(0, int(w.q_start[-1]), 24)) | {0, 319})
    _sampled_rows_match(w, layer, got, rows)


# ------------------------------------------------------------ coded caches
CODED = [("fp8prefix", None, None, None),      # MHA (G = 1), 32-token pages
         ("8b-int8", None, None, None),        # G = 4
         ("8b-int4", None, None, None),
         ("8b-int8", 64, 8, 32),               # G = 8, 32-token pages
         ("8b-int4", 16, 8, 32),               # G = 2
         ("fp8prefix", 32, 4, 16)]             # G = 8 on e4m3, 16-token pages


@pytest.mark.parametrize("shape", CODED)
@pytest.mark.parametrize("mix", range(len(MIXES)))
def test_prefill_coded_caches_match_the_oracle(shape, mix):
    layer_name, Hq, Hkv, bs = shape
    ctx, chunk = MIXES[mix]
    w = workloads.make_prefill(layer_name, ctx, chunk, seed=mix + 13, Hq=Hq, Hkv=Hkv, bs=bs)
    pa.pa_get_device_error(clear=True)
    layer, got = _gpu(w)
    assert pa.pa_get_device_error() == 0
    ref = _oracle(w, layer.tables_host)
    assert np.all(np.isfinite(got))
    assert excess(got, ref, tol(w)) <= 1.0, worst(got, ref, tol(w))


@pytest.mark.parametrize("layer_name", ["8b-int8", "8b-int4", "fp8prefix"])
def test_prefill_coded_two_tile_chunks_and_growing_scales(layer_name):
    """Chunks longer than one query tile (the two-tile kernel), with V values
    growing along the sequence so that the largest V scale seen moves several
    times and O is rescaled each time."""
    w = workloads.make_prefill(layer_name, [700, 0], [600, 1100], seed=5)
    pos = torch.from_numpy(np.asarray(w.fill_pos, dtype=np.float32))
    w.v_fill = (w.v_fill.float() * (1.0 + pos / 200.0).view(-1, 1, 1)).to(torch.bfloat16)
    pa.pa_get_device_error(clear=True)
    layer, got = _gpu(w)
    assert pa.pa_get_device_error() == 0
    ref = _oracle(w, layer.tables_host)
    assert excess(got, ref, tol(w)) <= 1.0, worst(got, ref, tol(w))


@pytest.mark.parametrize("kv", ["fp8", "int8", "int4"])
def test_prefill_coded_stale_codes_and_zero_scales(kv):
    """Codes past each sequence's end and in unused blocks are set to their
    largest values (e4m3: NaN), and one sequence's K and another's V are all
    zero (scale 0): outputs stay finite and match the oracle."""
    w = workloads.make_prefill("8b", [20, 3, 100, 40], [13, 30, 7, 9], seed=7, kv=kv)
    seq = np.asarray(w.fill_seq)
    kf, vf = w.k_fill.clone(), w.v_fill.clone()
    kf[torch.from_numpy(seq == 1)] = 0
    vf[torch.from_numpy(seq == 2)] = 0
    w.k_fill, w.v_fill = kf, vf
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    fill = {"fp8": 0x7F, "int8": 0x7F, "int4": 0x77}[kv]
    used = set()
    for b, n in enumerate(w.seq_lens):
        nb = -(-int(n) // w.bs)
        used.update(int(x) for x in layer.tables_host[b, :nb])
        last, rows = int(layer.tables_host[b, nb - 1]), int(n) - (nb - 1) * w.bs
        layer.k_cache[last, :, rows:] = fill
        layer.v_cache[last, :, rows:] = fill
    for blk in range(w.num_blocks):
        if blk not in used:
            layer.k_cache[blk] = fill
            layer.v_cache[blk] = fill
    pa.pa_get_device_error(clear=True)
    _, got = _gpu(w, layer=layer)
    assert pa.pa_get_device_error() == 0
    ref = _oracle(w, layer.tables_host)
    assert np.isfinite(got).all()
    assert excess(got, ref, tol(w)) <= 1.0, worst(got, ref, tol(w))


@pytest.mark.parametrize("layer_name", ["8b-int8", "8b-int4"])
def test_bench_coded_verify_configuration_sampled(layer_name):
    # the coded-cache verify batch bench.py times: 64 sequences, U[128, 4096] cached, 4 proposals + 1
    rng = np.random.default_rng(7)
    ctx = [int(x) for x in rng.integers(128, 4097, 64)]
    w = workloads.make_prefill(layer_name, ctx, [5] * 64, seed=31, device="cuda")
    layer, got = _gpu(w)
    rows = sorted(set(int(x) for x in np.random.default_rng(2).integers(0, int(w.q_start[-1]), 24)) | {0, 319})
    caches = {}
    for r in rows:
        b = int(np.searchsorted(w.q_start, r, side="right") - 1)
        C = int(w.q_start[b + 1] - w.q_start[b])
        pos = int(w.seq_lens[b]) - C + (r - int(w.q_start[b]))
        if b not in caches:
            caches[b] = oracle.run.OracleStep(w, seqs=[b], tables=layer.tables_host)
        ref = oracle.prefill_attention(caches[b].cache, w.q_chunk[r:r + 1], caches[b].tables[b:b + 1],
                                       np.array([pos + 1]), np.array([0, 1]), w.Hq, w.scale)
        assert excess(got[r:r + 1], ref, tol(w)) <= 1.0, ("row %d" % r, worst(got[r:r + 1], ref, tol(w)))
