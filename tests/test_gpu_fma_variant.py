"""The CUDA-core page step (PA_DECODE_FMA=1) against the fp64 oracle.

The decode kernel's tensor-core contraction has a CUDA-core counterpart
(packed fp32 FMAs) for bf16 caches with head_dim 128, 16-token pages and 4 or
8 query heads per kv head, kept so that the two can be timed against each
other.  It must give the same quantity: these tests hold it to the same
parity bound, on small cases (both kv heads per CTA and one), at full size,
and through the fused step.
"""
import os

import numpy as np
import pytest
import torch

import oracle.run
import paged_kv_cache_294_gb300 as pa
import workloads
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer
from tests.gpu_util import cache_bytes, excess, oracle_out, tol
from tests.test_gpu_decode import _synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture
def fma(monkeypatch):
    monkeypatch.setenv("PA_DECODE_FMA", "1")


def _run(w, splits, fused=False):
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    pa.pa_get_device_error(clear=True)
    if fused:
        layer.fused_step(num_splits=splits)
    else:
        layer.step(num_splits=splits)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    return layer


@pytest.mark.parametrize("name,kw", [("8b", dict(B=8, seq_len=900)), ("70b", dict(B=12, seq_len=700))])
@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("fused", [False, True])
def test_cuda_core_step_matches_the_oracle(fma, name, kw, splits, fused):
    w = workloads.make(name, **kw)
    layer = _run(w, splits, fused)
    _, ref = oracle_out(w, tables=layer.tables_host)
    got = layer.out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert excess(got, ref, tol(w)) <= 1.0


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (12, 3), (16, 2), (32, 4)])
def test_cuda_core_step_head_layouts_and_ragged_lengths(fma, Hq, Hkv):
    lens = [1, 15, 16, 17, 7 * 16 + 3, 0, 600]
    w = _synthetic(len(lens), Hq, Hkv, 128, 16, lens, seed=Hq + Hkv)
    for S in (0, 2):
        layer = _run(w, S)
        _, ref = oracle_out(w, tables=layer.tables_host)
        got = layer.out.float().cpu().numpy().astype(np.float64)
        assert excess(got, ref, tol(w)) <= 1.0
        assert torch.all(layer.out[5].float() == 0)


def test_cuda_core_step_stale_nan_rows_do_not_leak(fma):
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
    _, ref = oracle_out(w, tables=layer.tables_host)
    assert excess(got, ref, tol(w)) <= 1.0


@pytest.mark.parametrize("name", ["8b", "70b"])
def test_cuda_core_fused_step_full_size_every_output(fma, name):
    w = workloads.make(name, device="cuda")
    layer = _run(w, 0, fused=True)
    st = oracle.run.OracleStep(w, tables=layer.tables_host)
    st.append()
    ref = st.decode(threads=os.cpu_count() or 1)
    got = layer.out.float().cpu().numpy().astype(np.float64)
    assert excess(got, ref, tol(w)) <= 1.0
    assert np.array_equal(cache_bytes(layer.k_cache), st.cache.k)
