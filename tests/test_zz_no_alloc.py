"""The decode entry point that needs no workspace from its caller.

Some callers of this library only receive their input and output buffers and
may not allocate device memory: plugins of inference runtimes that plan every
byte of device memory ahead of time, or code that runs while another
component owns the allocator, where an allocation would fail, break the plan
or synchronise the device.  For them pa_decode_attention_static_ws uses a
workspace array owned by the library.

These tests call it through the C ABI and check that
  * it returns, bit for bit, what pa_decode_attention returns with a caller
    workspace (the same kernel on the same workspace layout), on two calls in
    a row, since the array keeps the previous call's contents;
  * one case also matches the fp64 oracle;
  * a large call followed by a smaller one of another layout stays exact:
    the first call's partial sums then lie where the second call's merge
    counters sit, and only the per-call clearing of those counters makes the
    shared array reusable;
  * too large a request is refused.
Every call in the process shares the one array.  The file's name sorts last
so that pytest collects it last: if it fails, a run that stops at the first
failure has already run every other test.  It also passes alone in a fresh
process.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_294_gb300 as pa
import workloads
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer
from tests.gpu_util import excess, oracle_out, tol

pytestmark = pytest.mark.gpu

CASES = [("8b", dict(B=8, seq_len=900), 0), ("8b", dict(B=8, seq_len=900), 5),
         ("long", dict(B=2, seq_len=4000), 16), ("fp8prefix", dict(B=6, seq_len=600), 0),
         ("8b-int8", dict(B=4, seq_len=700), 3), ("8b-int4", dict(B=4, seq_len=700), 0)]


def _static(layer, splits):
    out = torch.full_like(layer.out, float("nan"))
    pa.pa_decode_attention_static_ws(out, layer.q, layer.k_cache, layer.v_cache, layer.k_scale, layer.v_scale,
                                     layer.block_tables, layer.seq_lens, layer.scale, num_splits=splits)
    torch.cuda.synchronize()
    return out


def _caller_ws(layer, splits):
    out = layer.decode(num_splits=splits).clone()
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name,kw,splits", CASES)
def test_static_workspace_equals_caller_workspace_twice(name, kw, splits):
    w = workloads.make(name, **kw)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    pa.pa_get_device_error(clear=True)
    layer.append_step()
    ref = _caller_ws(layer, splits)
    for _ in range(2):
        got = _static(layer, splits)
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert pa.pa_get_device_error() == 0


def test_static_workspace_against_the_oracle():
    w = workloads.make("8b", B=8, seq_len=900)
    layer = PagedDecodeLayer.from_workload(w, "cuda")
    layer.append_step()
    got = _static(layer, 5).float().cpu().numpy().astype(np.float64)
    _, ref = oracle_out(w, tables=layer.tables_host)
    assert excess(got, ref, tol(w)) <= 1.0


def test_large_call_then_small_call_with_counters_over_old_partials():
    big = PagedDecodeLayer.from_workload(workloads.make("long", B=4, seq_len=16384), "cuda")
    small = PagedDecodeLayer.from_workload(workloads.make("tiny"), "cuda")
    for layer in (big, small):
        layer.append_step()
    S_big, S_small = 64, 3
    assert big.num_splits(S_big) == S_big and small.num_splits(S_small) == S_small
    # the small call's counters (the last 256-byte-rounded part of its layout)
    # start inside the big call's o_part region [0, B * Hq * S * d * 4)
    need_small = pa.pa_decode_workspace_bytes(small.B, small.Hq, small.Hkv, small.d, small.M, S_small)
    counters_at = need_small - (small.B * small.Hkv * 4 + 255) // 256 * 256
    assert counters_at < big.B * big.Hq * S_big * big.d * 4
    ref_big, ref_small = _caller_ws(big, S_big), _caller_ws(small, S_small)
    for _ in range(2):
        assert torch.equal(_static(big, S_big).view(torch.int16), ref_big.view(torch.int16))
        assert torch.equal(_static(small, S_small).view(torch.int16), ref_small.view(torch.int16))


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
