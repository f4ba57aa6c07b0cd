"""The decode step the benchmark times, at full size, against the fp64 oracle.

bench.py times pa_decode_step (the append of every sequence's new token,
attention and the split-K merge in one launch) with the automatic split
count on each workload's full batch.  These tests run that same launch on
the same seeded inputs and compare every output of every sequence with the
oracle, element by element, and the cache bytes (and scales) the step leaves
with the oracle's append, bit for bit.  The long-context workload is also run
at every split count the benchmark sweeps.

Bound per output (tests/gpu_util.py): max(atol, half a bf16 spacing of the
reference + 2^-10); atol = 1e-2 for bf16, int8 and int4 caches, 5e-2 for the
fp8 cache (against the oracle on the stored fp8 cache).
"""
import os

import numpy as np
import pytest
import torch

import oracle.run
import paged_kv_cache_294_gb300 as pa
import workloads
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer
from tests.gpu_util import cache_bytes, excess, tol, worst

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1


def _oracle(w, tables):
    st = oracle.run.OracleStep(w, tables=tables)
    st.append()
    return st, st.decode(threads=THREADS)


def _compare(w, layer, ref, what):
    got = layer.out.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), what
    assert excess(got, ref, tol(w)) <= 1.0, (what, worst(got, ref, tol(w)))


@pytest.mark.parametrize("name", ["8b", "70b", "long", "fp8prefix", "8b-int8", "8b-int4"])
def test_full_size_fused_step_every_output(name):
    w = workloads.make(name, device="cuda")
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    pa.pa_get_device_error(clear=True)
    layer.fused_step()                     # automatic split count, as timed
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    st, ref = _oracle(w, layer.tables_host)
    _compare(w, layer, ref, name)
    assert np.array_equal(cache_bytes(layer.k_cache), st.cache.k)
    assert np.array_equal(cache_bytes(layer.v_cache), st.cache.v)
    if layer.k_scale is not None:
        assert np.array_equal(layer.k_scale.cpu().numpy().view(np.uint32), st.cache.k_scale.view(np.uint32))
        assert np.array_equal(layer.v_scale.cpu().numpy().view(np.uint32), st.cache.v_scale.view(np.uint32))


def test_full_size_long_context_every_split_count():
    """4 x 131072 tokens at S = 1 .. 64 and the automatic count: the fused
    step re-appends the same token to the same slot, so every call sees the
    same cache and must give the oracle's output."""
    w = workloads.make("long", device="cuda")
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    st, ref = _oracle(w, layer.tables_host)
    for S in (1, 2, 4, 8, 16, 32, 64, 0):
        pa.pa_get_device_error(clear=True)
        layer.fused_step(num_splits=S)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0, S
        _compare(w, layer, ref, "long S=%d" % S)
