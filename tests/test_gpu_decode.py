"""pa_decode_attention through the C ABI against the fp64 oracle.

Tolerance per output: max(atol, half a bf16 spacing of the reference +
2^-10), atol = 1e-2 for the bf16 cache and 5e-2 for the fp8 cache (against
the oracle evaluated on the stored fp8 cache); the half spacing only exceeds
atol where |ref| >= 4 (resp. >= 16), since the outputs are bf16.  Small cases compare
every output; full-size cases (the benchmark's shapes and launch
configuration) compare sampled sequences, each computed by the oracle from
the same seeded inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.run
import paged_kv_cache_294_gb300 as pa
import workloads
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer
from tests.gpu_util import BF16_TOL, FP8_TOL, excess, gpu_out_f64, oracle_out, run_gpu, tol, worst

pytestmark = pytest.mark.gpu


def check(w, num_splits=0, seqs=None):
    layer = run_gpu(w, num_splits)
    st, ref = oracle_out(w, seqs=seqs, tables=layer.tables_host)
    got = gpu_out_f64(layer, seqs)
    assert np.all(np.isfinite(got))
    err = np.max(np.abs(got - ref))
    assert excess(got, ref, tol(w)) <= 1.0, (w.name, num_splits, err)
    assert pa.pa_get_device_error() == 0
    return layer, err


SMALL = [("tiny", {}), ("8b", dict(B=8, seq_len=600)), ("70b", dict(B=12, seq_len=500)),
         ("long", dict(B=2, seq_len=3000)), ("fp8prefix", dict(B=8, seq_len=700)),
         ("8b-int8", dict(B=8, seq_len=600)), ("8b-int4", dict(B=8, seq_len=600))]


@pytest.mark.parametrize("name,kw", SMALL)
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_small_configs_all_outputs(name, kw, splits):
    check(workloads.make(name, **kw), splits)


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16, 32, 64])
def test_long_context_split_sweep(S):
    w = workloads.make("long", B=2, seq_len=9000)
    check(w, S)


def _synthetic(B, Hq, Hkv, d, bs, lens, kv="bf16", seed=0, k_mult=1.0):
    """A workload object with explicit lengths and a random block permutation."""
    rng = np.random.default_rng(seed)
    M = max(1, max(-(-L // bs) for L in lens))
    nb = sum(-(-L // bs) for L in lens) + 7
    perm = rng.permutation(nb).astype(np.int32)
    tables = workloads._tables_from_perm(np.array(lens), bs, M, perm)
    fs, fp = workloads._history(np.array(lens))
    vals = workloads._values(seed, len(fs), B, Hq, Hkv, d, "cpu", k_mult)
    return workloads.Workload(name="synthetic", Hq=Hq, Hkv=Hkv, d=d, bs=bs, kv=kv, B=B, num_blocks=nb,
                              M=M, scale=1.0 / math.sqrt(d), seq_lens=np.array(lens, np.int32),
                              block_tables=tables, trace=None, target_rids=None, fill_seq=fs,
                              fill_pos=fp, **vals)


SHAPES = [
    # B, Hq, Hkv, d, bs, kv
    (5, 8, 8, 128, 16, "bf16"),     # MHA
    (5, 8, 1, 128, 16, "bf16"),     # MQA, G = 8
    (5, 16, 8, 128, 16, "bf16"),    # G = 2
    (5, 12, 3, 64, 16, "bf16"),     # G = 4, head_dim 64
    (5, 8, 2, 64, 32, "bf16"),
    (5, 16, 2, 128, 32, "bf16"),
    (5, 4, 4, 128, 32, "fp8"),
    (5, 8, 1, 128, 16, "fp8"),
    (5, 6, 3, 128, 32, "fp8"),
    (5, 4, 4, 128, 32, "int8"),
    (5, 8, 1, 128, 16, "int8"),
    (5, 16, 2, 128, 16, "int8"),
    (5, 4, 4, 128, 32, "int4"),
    (5, 8, 1, 128, 16, "int4"),
    (5, 16, 2, 128, 16, "int4"),
    (5, 6, 3, 128, 32, "int4"),
    # odd group sizes: a lane's second head column (2c + 1) is padding for some c
    (5, 24, 8, 128, 16, "bf16"),    # G = 3
    (5, 10, 2, 64, 16, "bf16"),     # G = 5, head_dim 64
    (5, 12, 2, 128, 32, "fp8"),     # G = 6
    (5, 14, 2, 128, 16, "int8"),    # G = 7
    (5, 21, 3, 128, 32, "int4"),    # G = 7, an odd kv-head count
]


@pytest.mark.parametrize("shape", SHAPES)
def test_head_layouts_and_ragged_lengths(shape):
    B, Hq, Hkv, d, bs, kv = shape
    lens = [1, bs - 1, bs, bs + 1, 7 * bs + 3][:B]
    w = _synthetic(B, Hq, Hkv, d, bs, lens, kv, seed=B + Hq + d + bs)
    for S in (0, 2):
        check(w, S)


def test_one_token_returns_v_exactly():
    w = _synthetic(3, 8, 2, 128, 16, [1, 1, 1], seed=4)
    layer = run_gpu(w)
    out = layer.out.view(torch.int16).cpu()
    vn = w.v_new.view(torch.int16)
    for b in range(3):
        for i in range(8):
            assert torch.equal(out[b, i], vn[b, i // 4])


def test_zero_length_gives_zero_rows_and_others_unaffected():
    w = _synthetic(3, 4, 2, 128, 16, [0, 20, 0], seed=5)
    layer = run_gpu(w)
    out = layer.out.float().cpu()
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    st, ref = oracle_out(w, tables=layer.tables_host)
    assert excess(out[1].numpy(), ref[1], BF16_TOL) <= 1.0, worst(out[1].numpy(), ref[1], BF16_TOL)


@pytest.mark.parametrize("S", [1, 3])
def test_bit_identical_under_physical_permutation(S):
    """For a fixed split count the accumulation order is logical, so moving blocks changes nothing."""
    outs = []
    for perm_seed in (1, 2):
        w = _synthetic(4, 16, 2, 128, 16, [33, 200, 517, 64], seed=9)
        rng = np.random.default_rng(perm_seed)
        perm = rng.permutation(w.num_blocks).astype(np.int32)
        w.block_tables = workloads._tables_from_perm(w.seq_lens, w.bs, w.M, perm)
        layer = run_gpu(w, S)
        outs.append(layer.out.view(torch.int16).cpu())
    assert torch.equal(outs[0], outs[1])


def test_stale_nan_bytes_past_the_end_do_not_leak():
    """Rows of a partial last block beyond seq_len hold NaN bf16 patterns: output stays exact-ish."""
    w = _synthetic(3, 8, 2, 128, 16, [5, 19, 40], seed=12)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    k = layer.k_cache.view(torch.int16)
    v = layer.v_cache.view(torch.int16)
    for b, L in enumerate(w.seq_lens):
        blk = int(layer.tables_host[b, (L - 1) // 16])
        k[blk, :, L % 16:, :] = 0x7FC0     # bf16 NaN
        v[blk, :, L % 16:, :] = 0x7FC0
    layer.step()
    torch.cuda.synchronize()
    got = layer.out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    st, ref = oracle_out(w, tables=layer.tables_host)
    assert excess(got, ref, BF16_TOL) <= 1.0, worst(got, ref, BF16_TOL)


def test_fp8_stale_nan_codes_past_the_end_do_not_leak():
    w = _synthetic(2, 4, 4, 128, 32, [7, 45], kv="fp8", seed=13)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    for b, L in enumerate(w.seq_lens):
        blk = int(layer.tables_host[b, (L - 1) // 32])
        layer.k_cache[blk, :, L % 32:, :] = 0x7F     # e4m3 NaN
        layer.v_cache[blk, :, L % 32:, :] = 0x7F
    layer.step()
    torch.cuda.synchronize()
    got = layer.out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    st, ref = oracle_out(w, tables=layer.tables_host)
    assert excess(got, ref, FP8_TOL) <= 1.0, worst(got, ref, FP8_TOL)


@pytest.mark.parametrize("kv,fill", [("int8", 0x7F), ("int4", 0x77)])
@pytest.mark.parametrize("bs", [16, 32])
def test_integer_codes_past_the_end_do_not_leak(kv, fill, bs):
    """Integer codes are always finite, so the kernel does not clear the rows
    past a sequence's end: the largest codes there must still weigh nothing."""
    w = _synthetic(2, 8, 2, 128, bs, [7, 3 * bs + 5], kv=kv, seed=17 + bs)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    st = oracle.run.OracleStep(w, tables=layer.tables_host)
    st.append()
    for b, L in enumerate(w.seq_lens):
        blk = int(layer.tables_host[b, (L - 1) // bs])
        # the same codes past the end in both caches (the step's append never
        # touches rows past its own)
        layer.k_cache[blk, :, L % bs:, :] = fill
        layer.v_cache[blk, :, L % bs:, :] = fill
        st.cache.k[blk, :, L % bs:, :] = fill
        st.cache.v[blk, :, L % bs:, :] = fill
    layer.append_step()
    ref = st.decode()
    for S in (0, 2):
        layer.decode(num_splits=S)
        torch.cuda.synchronize()
        got = layer.out.float().cpu().numpy()
        assert excess(got, ref, tol(w)) <= 1.0


# ------------------------------------------------------------ full sizes, sampled


def _sample(B, k=6):
    return sorted({0, B - 1} | set(np.random.default_rng(7).choice(B, size=k, replace=False).tolist()))


@pytest.mark.parametrize("name", ["8b", "70b", "fp8prefix", "8b-int8", "8b-int4"])
def test_full_size_sampled(name):
    w = workloads.make(name, device="cuda")
    seqs = _sample(w.B)
    if name == "fp8prefix":
        seqs = sorted(set(seqs) | {1, 50, 99, 100, 127})
    check(w, 0, seqs)


def test_full_size_long_sampled():
    w = workloads.make("long", device="cuda")
    check(w, 0, [1])
    check(w, 64, [3])


def test_split_counters_return_to_zero_and_calls_repeat_bit_exactly():
    w = workloads.make("8b", B=6, seq_len=900)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    ws = layer.ensure_workspace(5)
    assert layer.num_splits(5) > 1
    outs = []
    for _ in range(3):
        layer.decode(num_splits=5)
        torch.cuda.synchronize()
        outs.append(layer.out.clone())
        # merge counters: the last 256-byte-aligned part of the workspace
        need = pa.pa_decode_workspace_bytes(layer.B, layer.Hq, layer.Hkv, layer.d, layer.M, 5)
        tail = ws[:need].view(torch.int32)[-((layer.B * layer.Hkv + 63) // 64 * 64):]
        assert int(tail.abs().sum()) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


@pytest.mark.parametrize("S", [0, 2])
def test_large_ragged_batch(S):
    """4200 short sequences (zero lengths included): many CTAs, many zero rows."""
    rng = np.random.default_rng(21)
    lens = [int(x) for x in rng.integers(0, 40, size=4200)]
    w = _synthetic(4200, 4, 2, 64, 16, lens, seed=21)
    check(w, S)


@pytest.mark.parametrize("B", [255, 256, 257])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 3)])
@pytest.mark.parametrize("S", [0, 3])
def test_work_item_grid_edges(B, Hq, Hkv, S):
    """Batches at the edge of the one-warp work-item scan (every lane's eight
    sequences in use; one sequence more than it covers, which takes the direct
    grid), with empty, one-block and multi-partition lengths mixed, one or two
    kv heads per CTA; every output compared."""
    rng = np.random.default_rng(B * 7 + Hkv + S)
    lens = [int(x) for x in rng.choice([0, 1, 16, 17, 200, 700], size=B)]
    w = _synthetic(B, Hq, Hkv, 64, 16, lens, seed=B + Hkv)
    check(w, S)


def test_consecutive_calls_with_different_shapes():
    """Consecutive calls with different batch shapes on one workspace stay correct."""
    for B, lens in ((7, [5, 300, 17, 1, 0, 64, 900]), (3, [2000, 3, 40])):
        w = _synthetic(B, 16, 4, 128, 16, lens, seed=B)
        for S in (0, 1, 4):
            check(w, S)


@pytest.mark.parametrize("kv", ["fp8", "int8", "int4"])
def test_coded_blocks_with_zero_scales(kv):
    """Blocks whose K or V values are all zero get scale 0 and codes 0.  The
    kernel keeps O in units of the largest V scale seen so far: a sequence whose
    first page has V scale 0 and whose later pages do not, one whose every V is
    zero, and one whose K is zero (uniform weights) must all match the oracle."""
    w = _synthetic(4, 8, 2, 128, 16, [40, 33, 70, 5], kv=kv, seed=31)
    seq, pos = np.asarray(w.fill_seq), np.asarray(w.fill_pos)
    vf, kf = w.v_fill.clone(), w.k_fill.clone()
    vf[torch.from_numpy((seq == 0) & (pos < 16))] = 0      # sequence 0: first block's V only
    vf[torch.from_numpy(seq == 1)] = 0                      # sequence 1: every V
    kf[torch.from_numpy(seq == 2)] = 0                      # sequence 2: every K
    w.v_fill, w.k_fill = vf, kf
    w.v_new = w.v_new.clone()
    w.k_new = w.k_new.clone()
    w.v_new[1] = 0
    w.k_new[2] = 0
    for S in (0, 2):
        layer, _ = check(w, S)
    assert torch.all(layer.out[1].float() == 0)


def test_split_count_changes_on_one_workspace():
    """One layer, one workspace, the split count going down and up again: the
    merge counters' place moves with the layout, so the engine zero-fills the
    workspace whenever the layout changes (over old partials the counters
    would be garbage and the merges would not run).  Every call must write
    every output (poisoned with NaN first)."""
    w = workloads.make("long", B=2, seq_len=9000)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    st, ref = oracle_out(w, tables=layer.tables_host)
    for S in (16, 1, 2, 3, 64, 5, 0):
        layer.out.fill_(float("nan"))
        pa.pa_get_device_error(clear=True)
        layer.fused_step(num_splits=S)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0, S
        got = layer.out.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), S
        assert excess(got, ref, tol(w)) <= 1.0, (S, worst(got, ref, tol(w)))


@pytest.mark.parametrize("Hq,Hkv,kv", [(64, 8, "bf16"), (32, 8, "bf16"), (8, 8, "fp8")])
def test_max_split_count_merges_512_partials(Hq, Hkv, kv):
    """The largest split count (512): 8192-token sequences of 512 blocks, one
    block per partition, so the merge reads 512 partials per row (the most
    its shared-memory weights hold: 16 rows x 512 at G = 8)."""
    w = _synthetic(2, Hq, Hkv, 128, 16, [8192, 8000], kv, seed=Hq + Hkv)
    assert pa.pa_decode_resolve_splits(2, Hkv, 512, 512) == 512
    check(w, 512)


@pytest.mark.parametrize("S", [0, 3])
def test_all_sequences_empty(S):
    """Every seq_len 0: every output row is zero, nothing is read from the
    cache, and the merge counters stay at zero."""
    w = _synthetic(5, 8, 2, 128, 16, [0, 0, 0, 0, 0], "bf16", seed=1)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    ws = layer.ensure_workspace(S)
    layer.out.fill_(float("nan"))
    pa.pa_get_device_error(clear=True)
    layer.decode(num_splits=S)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert torch.count_nonzero(layer.out).item() == 0
    need = pa.pa_decode_workspace_bytes(layer.B, layer.Hq, layer.Hkv, layer.d, layer.M, S)
    assert int(ws[:need].view(torch.int32)[-((layer.B * layer.Hkv + 63) // 64 * 64):].abs().sum()) == 0
