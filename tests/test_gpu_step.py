"""pa_decode_step (append + attention in one launch) against the two-launch step.

The fused step must leave exactly the cache bytes (and fp8 scales) that
pa_kv_append writes and return exactly the outputs pa_decode_attention
returns on that cache; the two-launch path is itself checked against the
oracle in test_gpu_append.py / test_gpu_decode.py, and one case here is
checked against the oracle directly.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_294_gb300 as pa
import workloads
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer
from tests.gpu_util import cache_bytes, excess, oracle_out, tol
from tests.test_gpu_decode import _synthetic

pytestmark = pytest.mark.gpu


def _pair(w):
    a = PagedDecodeLayer.from_workload(w, "cuda")
    b = PagedDecodeLayer.from_workload(w, "cuda")
    return a, b


def _same_state(a, b):
    torch.cuda.synchronize()
    assert np.array_equal(cache_bytes(a.k_cache), cache_bytes(b.k_cache))
    assert np.array_equal(cache_bytes(a.v_cache), cache_bytes(b.v_cache))
    if a.k_scale is not None:
        assert torch.equal(a.k_scale.view(torch.int32), b.k_scale.view(torch.int32))
        assert torch.equal(a.v_scale.view(torch.int32), b.v_scale.view(torch.int32))


CASES = [("tiny", {}), ("8b", dict(B=8, seq_len=700)), ("70b", dict(B=12, seq_len=500)),
         ("long", dict(B=2, seq_len=3000)), ("fp8prefix", dict(B=8, seq_len=700)),
         ("8b-int8", dict(B=8, seq_len=700)), ("8b-int4", dict(B=8, seq_len=700))]


@pytest.mark.parametrize("name,kw", CASES)
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_fused_step_equals_append_then_decode(name, kw, splits):
    w = workloads.make(name, **kw)
    a, b = _pair(w)
    pa.pa_get_device_error(clear=True)
    out_a = a.step(num_splits=splits).clone()
    out_b = b.fused_step(num_splits=splits).clone()
    _same_state(a, b)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert pa.pa_get_device_error() == 0


SHAPES = [(5, 8, 8, 128, 16, "bf16"), (5, 8, 1, 128, 16, "bf16"), (5, 12, 3, 64, 16, "bf16"),
          (5, 8, 2, 64, 32, "bf16"), (5, 4, 4, 128, 32, "fp8"), (5, 8, 1, 128, 16, "fp8"),
          (5, 4, 4, 128, 32, "int8"), (5, 8, 2, 128, 16, "int8"),
          (5, 4, 4, 128, 32, "int4"), (5, 8, 2, 128, 16, "int4")]


@pytest.mark.parametrize("shape", SHAPES)
def test_fused_step_shapes_offsets_and_zero_lengths(shape):
    B, Hq, Hkv, d, bs, kv = shape
    # new tokens at offset 0 (fresh block), mid-block and last row; one empty sequence
    lens = [1, bs + 1, bs // 2, 0, 3 * bs][:B]
    w = _synthetic(B, Hq, Hkv, d, bs, lens, kv, seed=B + Hq + d + bs)
    if kv != "bf16":
        # larger new values than the history: the block scale grows and older rows re-encode
        w.k_new = (w.k_new.float() * 7).to(torch.bfloat16)
        w.v_new = (w.v_new.float() * 3).to(torch.bfloat16)
    for S in (0, 2):
        a, b = _pair(w)
        out_a = a.step(num_splits=S).clone()
        out_b = b.fused_step(num_splits=S).clone()
        _same_state(a, b)
        assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))


def test_fused_step_against_the_oracle():
    w = workloads.make("fp8prefix", B=8, seq_len=900)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    layer.fused_step()
    torch.cuda.synchronize()
    st, ref = oracle_out(w, tables=layer.tables_host)
    assert np.array_equal(cache_bytes(layer.k_cache), st.cache.k)
    assert np.array_equal(layer.k_scale.cpu().numpy().view(np.uint32), st.cache.k_scale.view(np.uint32))
    got = layer.out.float().cpu().numpy().astype(np.float64)
    assert excess(got, ref, tol(w)) <= 1.0


def test_fused_step_skips_an_invalid_last_block():
    w = _synthetic(3, 8, 2, 128, 16, [20, 40, 9], seed=3)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    before_k = layer.k_cache.clone()
    tables = layer.block_tables.clone()
    tables[1, 2] = 10 ** 6          # the block that would receive sequence 1's new token
    pa.pa_get_device_error(clear=True)
    pa.pa_decode_step(layer.out, layer.q, layer.k_new, layer.v_new, layer.k_cache, layer.v_cache, None, None,
                      tables, layer.seq_lens, layer.scale, 0, layer.ensure_workspace())
    assert pa.pa_get_device_error() & pa.PA_DEVERR_BLOCK_ID
    changed = (layer.k_cache != before_k).reshape(layer.k_cache.shape[0], -1).any(dim=1).nonzero().flatten()
    allowed = {int(layer.tables_host[0, 1]), int(layer.tables_host[2, 0])}   # the other two new tokens
    assert set(int(x) for x in changed) <= allowed


@pytest.mark.parametrize("name,kw", [("8b", dict(B=8, seq_len=700)), ("fp8prefix", dict(B=8, seq_len=700)),
                                     ("8b-int8", dict(B=8, seq_len=700)),
                                     ("8b-int4", dict(B=8, seq_len=700))])
@pytest.mark.parametrize("splits", [0, 3])
def test_fused_step_replayed_from_a_cuda_graph(name, kw, splits):
    """pa_decode_step captured in a CUDA graph (as a serving loop replays its
    step) writes the same cache bytes and outputs as the call made eagerly."""
    w = workloads.make(name, **kw)
    warm = PagedDecodeLayer.from_workload(w, "cuda")
    warm.fused_step(num_splits=splits)   # one-time per-kernel setup happens outside the capture
    torch.cuda.synchronize()
    a, b = _pair(w)
    pa.pa_get_device_error(clear=True)
    out_a = a.fused_step(num_splits=splits).clone()
    b.ensure_workspace(splits)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        b.fused_step(num_splits=splits)
    graph.replay()
    _same_state(a, b)
    assert torch.equal(out_a.view(torch.int16), b.out.view(torch.int16))
    assert pa.pa_get_device_error() == 0
