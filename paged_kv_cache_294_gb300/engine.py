"""A decode-step driver over the C ABI: device state for one paged-KV layer.

`PagedDecodeLayer` owns the device buffers of one attention layer's paged
cache (caches, fp8 scales, block tables, lengths, split-K workspace) and runs
a decode step as the C ABI defines it: pa_kv_append of each sequence's new
token, then pa_decode_attention.  Block tables come either from the caller
or from replaying an allocator trace on the library's pa_allocator; slots
come from pa_slot_mapping.  All arithmetic runs in libpagedattn.so.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import (PA_KV_FP8_E4M3, pa_allocator, pa_decode_attention, pa_decode_resolve_splits,
               pa_decode_step, pa_decode_workspace_bytes, pa_kv_append, pa_slot_mapping)


def replay_trace(trace, num_blocks: int, block_size: int, target_rids: Sequence[int], M: int):
    """Run an admit/finish/share trace on a fresh pa_allocator; return the
    targets' block tables [len(target_rids), M] (-1 padded) and the allocator."""
    alloc = pa_allocator(num_blocks, block_size)
    held: Dict[int, List[int]] = {}
    for op in trace:
        if op.kind == "alloc":
            held.setdefault(op.rid, []).extend(int(x) for x in alloc.alloc(op.n))
        elif op.kind == "free":
            alloc.free(held.pop(op.rid))
        elif op.kind == "share":
            ids = list(held[op.src])[: op.n] if op.n else list(held[op.src])
            alloc.share(ids)
            held.setdefault(op.rid, []).extend(ids)
        else:
            raise ValueError(op.kind)
    tables = np.full((len(target_rids), M), -1, dtype=np.int32)
    for b, rid in enumerate(target_rids):
        ids = held.get(rid, [])
        if len(ids) > M:
            raise ValueError("table wider than M")
        tables[b, : len(ids)] = ids
    return tables, alloc


class PagedDecodeLayer:
    def __init__(self, num_blocks: int, Hq: int, Hkv: int, d: int, bs: int, kv: str = "bf16",
                 device="cuda"):
        self.num_blocks, self.Hq, self.Hkv, self.d, self.bs, self.kv = num_blocks, Hq, Hkv, d, bs, kv
        self.device = torch.device(device)
        dt = torch.uint8 if kv == "fp8" else torch.bfloat16
        self.k_cache = torch.zeros((num_blocks, Hkv, bs, d), dtype=dt, device=self.device)
        self.v_cache = torch.zeros((num_blocks, Hkv, bs, d), dtype=dt, device=self.device)
        if kv == "fp8":
            self.k_scale = torch.zeros((num_blocks, Hkv), dtype=torch.float32, device=self.device)
            self.v_scale = torch.zeros((num_blocks, Hkv), dtype=torch.float32, device=self.device)
        else:
            self.k_scale = self.v_scale = None
        self.workspace: Optional[torch.Tensor] = None

    # ---------------------------------------------------------------- set-up
    def set_batch(self, block_tables: np.ndarray, seq_lens: np.ndarray):
        self.tables_host = np.ascontiguousarray(block_tables, dtype=np.int32)
        self.lens_host = np.ascontiguousarray(seq_lens, dtype=np.int32)
        self.block_tables = torch.from_numpy(self.tables_host).to(self.device)
        self.seq_lens = torch.from_numpy(self.lens_host).to(self.device)
        self.B, self.M = self.tables_host.shape
        # the new token of each sequence sits at position len - 1
        self.step_slots_host = pa_slot_mapping(self.tables_host, np.arange(self.B, dtype=np.int32),
                                               np.maximum(self.lens_host - 1, 0).astype(np.int32), self.bs)
        self.step_slots_host[self.lens_host <= 0] = -1
        self.step_slots = torch.from_numpy(self.step_slots_host).to(self.device)

    def ensure_workspace(self, num_splits: int = 0) -> torch.Tensor:
        need = pa_decode_workspace_bytes(self.B, self.Hq, self.Hkv, self.d, self.M, num_splits)
        if self.workspace is None or self.workspace.numel() < need:
            # zero-filled: the split-K counters must start at zero (calls keep them there)
            self.workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=self.device)
        return self.workspace

    def num_splits(self, num_splits: int = 0) -> int:
        return pa_decode_resolve_splits(self.B, self.Hkv, self.M, num_splits)

    def fill(self, fill_seq: np.ndarray, fill_pos: np.ndarray, k_fill: torch.Tensor, v_fill: torch.Tensor,
             chunk: int = 1 << 20):
        """Write the cached history through pa_kv_append (one call per chunk of tokens,
        cut only at sequence boundaries so fp8 runs stay whole)."""
        if len(fill_seq) == 0:
            return
        slots = pa_slot_mapping(self.tables_host, fill_seq, fill_pos, self.bs)
        n = len(slots)
        start = 0
        while start < n:
            end = min(n, start + chunk)
            while end < n and fill_seq[end] == fill_seq[end - 1]:
                end += 1
            s = torch.from_numpy(slots[start:end]).to(self.device)
            pa_kv_append(self.k_cache, self.v_cache, self.k_scale, self.v_scale,
                         k_fill[start:end].to(self.device), v_fill[start:end].to(self.device), s)
            start = end

    @classmethod
    def from_workload(cls, w, device="cuda") -> "PagedDecodeLayer":
        layer = cls(w.num_blocks, w.Hq, w.Hkv, w.d, w.bs, w.kv, device)
        if w.block_tables is not None:
            tables = w.block_tables
        else:
            tables, layer.allocator = replay_trace(w.trace, w.num_blocks, w.bs, w.target_rids, w.M)
        layer.set_batch(tables, w.seq_lens)
        layer.fill(w.fill_seq, w.fill_pos, w.k_fill, w.v_fill)
        layer.q = w.q.to(device)
        layer.k_new = w.k_new.to(device)
        layer.v_new = w.v_new.to(device)
        layer.scale = w.scale
        layer.out = torch.empty_like(layer.q)
        return layer

    # ---------------------------------------------------------------- step
    def append_step(self, k_new=None, v_new=None, slots=None, stream=None):
        pa_kv_append(self.k_cache, self.v_cache, self.k_scale, self.v_scale,
                     self.k_new if k_new is None else k_new, self.v_new if v_new is None else v_new,
                     self.step_slots if slots is None else slots, stream=stream)

    def decode(self, q=None, out=None, num_splits: int = 0, tables=None, lens=None, stream=None):
        ws = self.ensure_workspace(num_splits)
        out = self.out if out is None else out
        pa_decode_attention(out, self.q if q is None else q, self.k_cache, self.v_cache, self.k_scale,
                            self.v_scale, self.block_tables if tables is None else tables,
                            self.seq_lens if lens is None else lens, self.scale, num_splits,
                            ws, stream=stream)
        return out

    def step(self, num_splits: int = 0, stream=None):
        """pa_kv_append of the new tokens, then pa_decode_attention (two launches)."""
        self.append_step(stream=stream)
        return self.decode(num_splits=num_splits, stream=stream)

    def fused_step(self, q=None, k_new=None, v_new=None, out=None, num_splits: int = 0, tables=None,
                   lens=None, stream=None):
        """The same step through pa_decode_step (one launch)."""
        ws = self.ensure_workspace(num_splits)
        out = self.out if out is None else out
        pa_decode_step(out, self.q if q is None else q, self.k_new if k_new is None else k_new,
                       self.v_new if v_new is None else v_new, self.k_cache, self.v_cache, self.k_scale,
                       self.v_scale, self.block_tables if tables is None else tables,
                       self.seq_lens if lens is None else lens, self.scale, num_splits, ws, stream=stream)
        return out
