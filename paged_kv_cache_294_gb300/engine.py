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

from . import (PA_ERR_OOM, PA_KV_INT4, PagedAttnError, pa_allocator, pa_block_cow, pa_copy_blocks,
               pa_decode_attention, pa_decode_resolve_splits, pa_decode_step, pa_decode_workspace_bytes,
               pa_kv_append, pa_prefix_cache, pa_slot_mapping)


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


class BlockManager:
    """Block tables of live sequences over a pa_allocator, with prefix caching
    and copy-on-write ("KV cache & continuous batching", sections
    "2. PagedAttention" and "4. Prefix caching").

    add(sid, tokens)     reuses the longest cached prefix, allocates blocks for
                         the rest and returns the first position whose KV the
                         caller must still write;
    commit(sid)          caches the sequence's full blocks (after their KV is
                         written);
    fork(child, parent)  the child shares every block of the parent;
    append(sid, token)   reserves the next token's slot: a fresh block at a
                         block boundary, else the block it lands in after
                         pa_block_cow; returns (slot, (src, dst) or None), the
                         pair naming a block copy the caller must run (with
                         pa_copy_blocks) before writing;
    free(sid)            drops the sequence's references.
    When the pool runs dry, blocks only the prefix cache holds are evicted.
    """

    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = True):
        self.bs = int(block_size)
        self.alloc = pa_allocator(num_blocks, block_size)
        self.cache = pa_prefix_cache(self.alloc) if prefix_caching else None
        # each sequence's tokens: an int32 buffer (grown by doubling) and its length,
        # handed to the prefix cache without conversion
        self._tok: Dict[int, list] = {}
        self.blocks: Dict[int, List[int]] = {}

    def tokens(self, sid: int) -> np.ndarray:
        buf, n = self._tok[sid]
        return buf[:n]

    def _alloc(self, n: int) -> List[int]:
        if n <= 0:
            return []
        short = n - self.alloc.num_free()
        if short > 0 and self.cache is not None:
            self.cache.evict(short)
        return [int(x) for x in self.alloc.alloc(n)]

    def add(self, sid: int, tokens: Sequence[int]) -> int:
        if sid in self.blocks:
            raise ValueError("sequence %d exists" % sid)
        toks = np.array(tokens, dtype=np.int32)
        shared = self.cache.match(toks).tolist() if self.cache is not None else []
        try:
            own = self._alloc(-(-len(toks) // self.bs) - len(shared))
        except PagedAttnError:
            self.alloc.free(shared)
            raise
        self._tok[sid], self.blocks[sid] = [toks, len(toks)], shared + own
        return len(shared) * self.bs

    def commit(self, sid: int) -> None:
        if self.cache is not None:
            self.cache.insert(self.tokens(sid), self.blocks[sid])

    def fork(self, child: int, parent: int) -> None:
        if child in self.blocks:
            raise ValueError("sequence %d exists" % child)
        self.alloc.share(self.blocks[parent])
        self._tok[child] = [self.tokens(parent).copy(), len(self.tokens(parent))]
        self.blocks[child] = list(self.blocks[parent])

    def append(self, sid: int, token: int):
        entry, blocks = self._tok[sid], self.blocks[sid]
        n = entry[1]
        j = n // self.bs
        copy = None
        if j == len(blocks):
            blocks.append(self._alloc(1)[0])
        else:
            try:
                dst, needs_copy = pa_block_cow(self.alloc, blocks[j])
            except PagedAttnError as e:
                if e.status != PA_ERR_OOM or self.cache is None or self.cache.evict(1) == 0:
                    raise
                dst, needs_copy = pa_block_cow(self.alloc, blocks[j])
            if needs_copy:
                copy = (blocks[j], dst)
            blocks[j] = dst
        if n == len(entry[0]):
            grown = np.empty(max(16, 2 * n), dtype=np.int32)
            grown[:n] = entry[0][:n]
            entry[0] = grown
        entry[0][n] = int(token)
        entry[1] = n + 1
        return blocks[j] * self.bs + n % self.bs, copy

    def free(self, sid: int) -> None:
        self.alloc.free(self.blocks.pop(sid))
        del self._tok[sid]

    def table(self, sids: Sequence[int], M: int) -> np.ndarray:
        t = np.full((len(sids), M), -1, dtype=np.int32)
        for i, sid in enumerate(sids):
            b = self.blocks[sid]
            if len(b) > M:
                raise ValueError("table wider than M")
            t[i, : len(b)] = b
        return t

    def lens(self, sids: Sequence[int]) -> np.ndarray:
        return np.asarray([self._tok[s][1] for s in sids], dtype=np.int32)


class PagedDecodeLayer:
    def __init__(self, num_blocks: int, Hq: int, Hkv: int, d: int, bs: int, kv: str = "bf16",
                 device="cuda"):
        self.num_blocks, self.Hq, self.Hkv, self.d, self.bs, self.kv = num_blocks, Hq, Hkv, d, bs, kv
        self.device = torch.device(device)
        dt = {"bf16": torch.bfloat16, "fp8": torch.uint8, "int8": torch.int8, "int4": torch.uint8}[kv]
        row = d // 2 if kv == "int4" else d          # int4: two codes per byte
        self.k_cache = torch.zeros((num_blocks, Hkv, bs, row), dtype=dt, device=self.device)
        self.v_cache = torch.zeros((num_blocks, Hkv, bs, row), dtype=dt, device=self.device)
        if kv != "bf16":
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

    def copy_blocks(self, pairs, stream=None):
        """Run the block copies BlockManager.append asked for (copy-on-write)."""
        if not pairs:
            return
        src = torch.tensor([p[0] for p in pairs], dtype=torch.int32).to(self.device)
        dst = torch.tensor([p[1] for p in pairs], dtype=torch.int32).to(self.device)
        pa_copy_blocks(self.k_cache, self.v_cache, self.k_scale, self.v_scale, src, dst, stream=stream,
                       kv_dtype=PA_KV_INT4 if self.kv == "int4" else None)

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
