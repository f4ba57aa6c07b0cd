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

from . import (PA_KV_INT4, PA_SHARE_MAX_ROWS, pa_allocator, pa_blocks_for_tokens, pa_copy_blocks,
               pa_decode_attention, pa_decode_resolve_splits, pa_decode_shared_workspace_bytes, pa_decode_step,
               pa_decode_step_shared, pa_decode_workspace_bytes, pa_kv_append, pa_prefix_cache, pa_seq_admit,
               pa_seq_append_slot, pa_share_plan, pa_slot_mapping, pa_step_slots)


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


class _BlockLists:
    """Read-only view of BlockManager's per-sequence block buffers as lists."""

    def __init__(self, bufs):
        self._bufs = bufs

    def __contains__(self, sid) -> bool:
        return sid in self._bufs

    def __getitem__(self, sid) -> List[int]:
        buf, n = self._bufs[sid]
        return [int(x) for x in buf[:n]]

    def __len__(self) -> int:
        return len(self._bufs)


class BlockManager:
    """Block tables of live sequences over a pa_allocator, with prefix caching
    and copy-on-write ("KV cache & continuous batching", sections
    "2. PagedAttention" and "4. Prefix caching").  Every block decision is
    the library's (pa_seq_admit, pa_seq_append_slot, pa_prefix_insert); this
    class keeps each sequence's tokens and blocks in int32 buffers.

    add(sid, tokens)     reuses the longest cached prefix, allocates blocks for
                         the rest and returns the first position whose KV the
                         caller must still write;
    commit(sid)          caches the sequence's full blocks (after their KV is
                         written);
    fork(child, parent)  the child shares every block of the parent;
    append(sid, token)   reserves the next token's slot: a fresh block when the
                         token opens one, else the block it lands in after
                         copy-on-write; returns (slot, (src, dst) or None), the
                         pair naming a block copy the caller must run (with
                         pa_copy_blocks) before writing;
    free(sid)            drops the sequence's references.
    When the pool runs dry, blocks only the prefix cache holds are evicted.
    """

    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = True):
        self.bs = int(block_size)
        self.alloc = pa_allocator(num_blocks, block_size)
        self.cache = pa_prefix_cache(self.alloc) if prefix_caching else None
        # each sequence's tokens and blocks: an int32 buffer (grown by doubling)
        # and its used length, handed to the library without conversion
        self._tok: Dict[int, list] = {}
        self._blk: Dict[int, list] = {}
        self.blocks = _BlockLists(self._blk)

    def tokens(self, sid: int) -> np.ndarray:
        buf, n = self._tok[sid]
        return buf[:n]

    @staticmethod
    def _room(entry, extra: int = 1):
        """Grow a [buffer, used] pair so that `extra` more entries fit."""
        buf, n = entry
        if n + extra > len(buf):
            grown = np.empty(max(16, 2 * len(buf), n + extra), dtype=np.int32)
            grown[:n] = buf[:n]
            entry[0] = grown

    def add(self, sid: int, tokens: Sequence[int]) -> int:
        if sid in self._blk:
            raise ValueError("sequence %d exists" % sid)
        toks = np.array(tokens, dtype=np.int32)
        buf = np.empty(max(4, pa_blocks_for_tokens(len(toks), self.bs)), dtype=np.int32)
        n, first = pa_seq_admit(self.alloc, self.cache, toks, buf)
        self._tok[sid], self._blk[sid] = [toks, len(toks)], [buf, n]
        return first

    def commit(self, sid: int) -> None:
        if self.cache is not None:
            buf, n = self._blk[sid]
            self.cache.insert(self.tokens(sid), buf[:n])

    def fork(self, child: int, parent: int) -> None:
        if child in self._blk:
            raise ValueError("sequence %d exists" % child)
        buf, n = self._blk[parent]
        self.alloc.share(buf[:n])
        self._tok[child] = [self.tokens(parent).copy(), len(self.tokens(parent))]
        self._blk[child] = [buf[:max(n, 4)].copy(), n]

    def append(self, sid: int, token: int):
        tok, blk = self._tok[sid], self._blk[sid]
        self._room(blk)
        slot, blk[1], copy = pa_seq_append_slot(self.alloc, self.cache, blk[0], blk[1], tok[1])
        self._room(tok)
        tok[0][tok[1]] = int(token)
        tok[1] += 1
        return slot, copy

    def free(self, sid: int) -> None:
        buf, n = self._blk.pop(sid)
        self.alloc.free(buf[:n])
        del self._tok[sid]

    def table(self, sids: Sequence[int], M: int) -> np.ndarray:
        t = np.full((len(sids), M), -1, dtype=np.int32)
        for i, sid in enumerate(sids):
            buf, n = self._blk[sid]
            if n > M:
                raise ValueError("table wider than M")
            t[i, :n] = buf[:n]
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
        self._ws_key = None   # layout the workspace last served (its counters are zero for it)
        self._layouts = {}    # (B, Hq, Hkv, d, M, num_splits) -> (workspace bytes, resolved split count)

    # ---------------------------------------------------------------- set-up
    def set_batch(self, block_tables: np.ndarray, seq_lens: np.ndarray):
        self.tables_host = np.ascontiguousarray(block_tables, dtype=np.int32)
        self.lens_host = np.ascontiguousarray(seq_lens, dtype=np.int32)
        self.block_tables = torch.from_numpy(self.tables_host).to(self.device)
        self.seq_lens = torch.from_numpy(self.lens_host).to(self.device)
        self.B, self.M = self.tables_host.shape
        # the slot of each sequence's new token (its last position; -1 for empty sequences)
        self.step_slots_host = pa_step_slots(self.tables_host, self.lens_host, self.bs)
        self.step_slots = torch.from_numpy(self.step_slots_host).to(self.device)

    def _workspace_for(self, key, need: int) -> torch.Tensor:
        """A zero-filled workspace of at least `need` bytes for the layout `key`.
        Calls leave the counters at zero, but their place follows from the
        layout: a workspace that served another layout is zero-filled again."""
        filled = False
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=self.device)
            filled = True
        elif key != self._ws_key:
            self.workspace.zero_()
            filled = True
        if filled and self.workspace.is_cuda:
            # the fill ran on torch's current stream; a call may come on another
            torch.cuda.current_stream(self.workspace.device).synchronize()
        self._ws_key = key
        return self.workspace

    def ensure_workspace(self, num_splits: int = 0) -> torch.Tensor:
        # the library's answers depend only on these arguments (the split
        # override and the SM count are fixed per process): asked once per
        # layout instead of on every step
        key = (self.B, self.Hq, self.Hkv, self.d, self.M, int(num_splits))
        lay = self._layouts.get(key)
        if lay is None:
            lay = self._layouts[key] = (pa_decode_workspace_bytes(*key), self.num_splits(num_splits))
        need, S = lay
        return self._workspace_for(("plain", S, need), need)

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

    # ---------------------------------------------------------------- shared prefixes
    def plan_sharing(self, min_blocks: int = 1):
        """Plan the shared prefixes of the current batch (pa_share_plan on the
        host tables) and place the plan on the device; returns the plan."""
        plan = pa_share_plan(self.tables_host, self.lens_host, self.bs, PA_SHARE_MAX_ROWS // (self.Hq // self.Hkv),
                             min_blocks)
        self.share_plan = plan
        self.chunk_of = torch.from_numpy(plan["chunk_of"]).to(self.device)
        self.chunk_members = torch.from_numpy(plan["chunk_members"].reshape(-1, PA_SHARE_MAX_ROWS)).to(self.device)
        self.chunk_blocks = torch.from_numpy(plan["chunk_blocks"]).to(self.device)
        return plan

    def ensure_shared_workspace(self, num_splits: int = 0) -> torch.Tensor:
        mcb = self.share_plan["max_chunk_blocks"]
        need = pa_decode_shared_workspace_bytes(self.B, self.Hq, self.Hkv, self.d, self.M, num_splits, mcb)
        return self._workspace_for(("shared", self.num_splits(num_splits), mcb, need), need)

    def shared_step(self, append: bool = True, out=None, num_splits: int = 0, stream=None):
        """The decode step (or attention alone) through pa_decode_step_shared with
        the plan of plan_sharing."""
        ws = self.ensure_shared_workspace(num_splits)
        out = self.out if out is None else out
        pa_decode_step_shared(out, self.q, self.k_new if append else None, self.v_new if append else None,
                              self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.block_tables,
                              self.seq_lens, self.chunk_of, self.chunk_members, self.chunk_blocks,
                              self.share_plan["max_chunk_blocks"], self.scale, num_splits, ws, stream=stream)
        return out

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
