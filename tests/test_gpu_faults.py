"""Bad inputs return a status or set a device error bit; nothing faults or hangs."""
import numpy as np
import pytest
import torch

import paged_kv_cache_294_gb300 as pa
import workloads
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer

pytestmark = pytest.mark.gpu


def _layer(name="tiny", **kw):
    w = workloads.make(name, **kw)
    return PagedDecodeLayer.from_workload(w, "cuda")


def test_out_of_range_block_id_is_flagged_and_clamped():
    layer = _layer()
    pa.pa_get_device_error(clear=True)
    bad = layer.block_tables.clone()
    bad[3, 2] = 10 ** 6
    bad[2, 0] = -5
    pa.pa_decode_attention(layer.out, layer.q, layer.k_cache, layer.v_cache, None, None, bad,
                           layer.seq_lens, layer.scale, 0, layer.ensure_workspace())
    flags = pa.pa_get_device_error()
    assert flags & pa.PA_DEVERR_BLOCK_ID
    assert torch.all(torch.isfinite(layer.out.float()))


def test_seq_len_beyond_table_is_flagged():
    layer = _layer()
    pa.pa_get_device_error(clear=True)
    lens = layer.seq_lens.clone()
    lens[0] = 10 ** 6
    pa.pa_decode_attention(layer.out, layer.q, layer.k_cache, layer.v_cache, None, None,
                           layer.block_tables, lens, layer.scale, 0, layer.ensure_workspace())
    assert pa.pa_get_device_error() & pa.PA_DEVERR_SEQ_LEN


def test_slot_beyond_pool_is_skipped_and_flagged():
    layer = _layer()
    pa.pa_get_device_error(clear=True)
    before = layer.k_cache.clone()
    slots = torch.tensor([64 * 16, 64 * 16 + 5, -1, 10 ** 9], dtype=torch.int64, device="cuda")
    pa.pa_kv_append(layer.k_cache, layer.v_cache, None, None, layer.k_new, layer.v_new, slots)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_SLOT
    assert torch.equal(before, layer.k_cache)


def test_host_side_argument_errors():
    layer = _layer("8b", B=4, seq_len=300)
    lib = pa.load()
    ws = layer.ensure_workspace(4)
    need = pa.pa_decode_workspace_bytes(layer.B, layer.Hq, layer.Hkv, layer.d, layer.M, 4)
    assert need > 0
    args = dict(out=layer.out.data_ptr(), q=layer.q.data_ptr(), k=layer.k_cache.data_ptr(),
                v=layer.v_cache.data_ptr(), t=layer.block_tables.data_ptr(), l=layer.seq_lens.data_ptr())

    def call(ws_ptr, ws_bytes, splits=4, q=None, dtype=0):
        return lib.pa_decode_attention(args["out"], args["q"] if q is None else q, args["k"], args["v"],
                                       None, None, args["t"], args["l"], layer.B, layer.Hq, layer.Hkv,
                                       layer.d, layer.bs, layer.M, layer.num_blocks, layer.scale, splits,
                                       ws_ptr, ws_bytes, dtype, None)

    assert call(ws.data_ptr(), need - 1) == pa.PA_ERR_INVALID          # workspace too small
    assert call(None, 0) == pa.PA_ERR_INVALID                           # workspace missing
    assert call(ws.data_ptr(), need, q=args["q"] + 2) == pa.PA_ERR_INVALID   # misaligned q
    assert call(ws.data_ptr(), need, dtype=1) == pa.PA_ERR_INVALID      # fp8 without scales
    assert call(ws.data_ptr(), need, dtype=5) == pa.PA_ERR_INVALID      # unknown cache dtype
    assert call(ws.data_ptr(), need) == pa.PA_OK
    torch.cuda.synchronize()
    with pytest.raises(TypeError):
        pa.pa_decode_attention(layer.out.float(), layer.q, layer.k_cache, layer.v_cache, None, None,
                               layer.block_tables, layer.seq_lens, layer.scale)


def test_bounded_wait_gives_up_and_reports():
    """A barrier phase nobody completes: the wait ends by itself and reports a timeout."""
    pa.pa_get_device_error(clear=True)
    pa.pa_selftest_bounded_wait()
    assert pa.pa_get_device_error() == pa.PA_DEVERR_TIMEOUT
    # the context is still usable afterwards
    layer = _layer()
    layer.step()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0


def test_every_tensor_argument_must_be_on_the_calls_device():
    """A host tensor among CUDA ones (a cache, a scale, a workspace, a table)
    is refused before any launch: the kernel or its TMA map would otherwise
    be handed a host pointer."""
    layer = _layer("fp8prefix", B=2, seq_len=100)
    ws = layer.ensure_workspace(0)
    before = layer.out.clone()
    host = {"k_cache": layer.k_cache.cpu(), "k_scale": layer.k_scale.cpu(), "workspace": ws.cpu(),
            "block_tables": layer.block_tables.cpu()}
    for name, t in host.items():
        kw = dict(k_cache=layer.k_cache, k_scale=layer.k_scale, workspace=ws, block_tables=layer.block_tables)
        kw[name] = t
        with pytest.raises(ValueError, match=name):
            pa.pa_decode_attention(layer.out, layer.q, kw["k_cache"], layer.v_cache, kw["k_scale"], layer.v_scale,
                                   kw["block_tables"], layer.seq_lens, layer.scale, 0, kw["workspace"])
        with pytest.raises(ValueError, match=name):
            pa.pa_decode_step(layer.out, layer.q, layer.k_new, layer.v_new, kw["k_cache"], layer.v_cache,
                              kw["k_scale"], layer.v_scale, kw["block_tables"], layer.seq_lens, layer.scale, 0,
                              kw["workspace"])
        if name != "workspace":
            with pytest.raises(ValueError, match=name):
                pa.pa_decode_attention_static_ws(layer.out, layer.q, kw["k_cache"], layer.v_cache, kw["k_scale"],
                                                 layer.v_scale, kw["block_tables"], layer.seq_lens, layer.scale)
    with pytest.raises(ValueError, match="k_cache"):
        pa.pa_kv_append(layer.k_cache.cpu(), layer.v_cache, layer.k_scale, layer.v_scale, layer.k_new,
                        layer.v_new, layer.step_slots)
    with pytest.raises(ValueError, match="v_scale"):
        pa.pa_copy_blocks(layer.k_cache, layer.v_cache, layer.k_scale, layer.v_scale.cpu(),
                          torch.zeros(1, dtype=torch.int32, device="cuda"),
                          torch.ones(1, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), layer.out.view(torch.int16))
