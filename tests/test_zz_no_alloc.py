"""The decode entry point that needs no workspace from its caller.

Some callers of this library only get their input and output buffers and may
not allocate device memory (runtime plugins whose memory is planned ahead,
code running while another component owns the allocator).  For them
pa_decode_attention_static_ws uses a workspace array owned by the library.
These tests call it through the C ABI and compare it with pa_decode_attention
given a caller workspace, on two calls in a row (the array keeps the previous
call's contents), and check that too large a request is refused.  This file
is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_294_gb300 as pa
import workloads
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer
from tests.gpu_util import excess, tol

pytestmark = pytest.mark.gpu

CASES = [("8b", dict(B=8, seq_len=900), 0), ("8b", dict(B=8, seq_len=900), 5),
         ("long", dict(B=2, seq_len=4000), 16), ("fp8prefix", dict(B=6, seq_len=600), 0)]


@pytest.mark.parametrize("name,kw,splits", CASES)
def test_static_workspace_matches_caller_workspace_twice(name, kw, splits):
    w = workloads.make(name, **kw)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    pa.pa_get_device_error(clear=True)
    layer.append_step()
    ref = layer.decode(num_splits=splits).clone()
    torch.cuda.synchronize()
    ref64 = ref.float().cpu().numpy().astype(np.float64)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        pa.pa_decode_attention_static_ws(out, layer.q, layer.k_cache, layer.v_cache, layer.k_scale,
                                         layer.v_scale, layer.block_tables, layer.seq_lens, layer.scale,
                                         num_splits=splits)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        assert excess(got, ref64, tol(w)) <= 1.0
    assert pa.pa_get_device_error() == 0


def test_static_workspace_refuses_requests_beyond_its_size():
    B, Hq, Hkv, d, bs, M = 4, 32, 8, 128, 16, 8192
    need = pa.pa_decode_workspace_bytes(B, Hq, Hkv, d, M, 512)
    assert need > pa.PA_STATIC_WORKSPACE_BYTES
    dev = "cuda"
    k = torch.zeros((64, Hkv, bs, d), dtype=torch.bfloat16, device=dev)
    q = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    tables = torch.zeros((B, M), dtype=torch.int32, device=dev)
    lens = torch.full((B,), 5, dtype=torch.int32, device=dev)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_decode_attention_static_ws(out, q, k, k, None, None, tables, lens, 0.1, num_splits=512)
    assert e.value.status == pa.PA_ERR_INVALID
    # a request that fits runs
    pa.pa_decode_attention_static_ws(out, q, k, k, None, None, tables, lens, 0.1, num_splits=1)
    torch.cuda.synchronize()
    assert torch.all(torch.isfinite(out.float()))
