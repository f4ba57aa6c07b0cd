"""PagedDecodeLayer's workspace rules, host side (a CPU layer; no launch).

The decode calls leave the workspace's merge counters at zero, but where the
counters sit follows from the layout (batch, heads, split count): a workspace
that served another layout must be zero-filled again before its next call.
"""
import numpy as np
import torch

import paged_kv_cache_294_gb300 as pa
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer


def _layer(B, M):
    layer = PagedDecodeLayer(num_blocks=256, Hq=8, Hkv=2, d=128, bs=16, device="cpu")
    tables = np.arange(B * M, dtype=np.int32).reshape(B, M) % 256
    lens = np.full(B, M * 16, np.int32)
    layer.set_batch(tables, lens)
    return layer


def test_workspace_size_and_zero_fill_follow_the_layout():
    layer = _layer(4, 8)
    for S in (0, 1, 3, 8, 0):
        ws = layer.ensure_workspace(S)
        assert ws.numel() >= pa.pa_decode_workspace_bytes(4, 8, 2, 128, 8, S)
        assert layer.num_splits(S) == pa.pa_decode_resolve_splits(4, 2, 8, S)
    ws = layer.ensure_workspace(3)
    assert torch.all(ws == 0)
    ws.fill_(7)                                    # stands in for counters a call left behind
    assert layer.ensure_workspace(3) is ws and torch.all(ws == 7)   # same layout: kept as it is
    layer.ensure_workspace(1)                      # another split count: zero-filled
    assert torch.all(layer.workspace == 0)
    layer.ensure_workspace(3)
    layer.workspace.fill_(7)
    # a new batch of another size with the same split request is another
    # layout too (its counters sit past its larger partials)
    layer.set_batch(np.zeros((6, 8), np.int32), np.full(6, 100, np.int32))
    ws = layer.ensure_workspace(3)
    assert ws.numel() >= pa.pa_decode_workspace_bytes(6, 8, 2, 128, 8, 3)
    assert torch.all(ws == 0)


def test_split_request_resolution_is_the_librarys():
    layer = _layer(2, 64)
    for S in (0, 2, 5, 64, 600):
        assert layer.num_splits(S) == pa.pa_decode_resolve_splits(2, 2, 64, S)
        assert layer.ensure_workspace(S).numel() >= pa.pa_decode_workspace_bytes(2, 8, 2, 128, 64, S)
