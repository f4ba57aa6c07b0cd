"""Oracle-side evaluation of a seeded workload (test infrastructure).

Builds the oracle's own cache from the workload's inputs with the oracle's
own allocator, slot mapping and append, then evaluates decode attention.
Nothing here reads a value produced by the CUDA library.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import Allocator, Cache, decode_attention, slot_mapping


def replay_trace(trace, num_blocks: int, target_rids: Sequence[int], M: int) -> np.ndarray:
    alloc = Allocator(num_blocks)
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
        tables[b, : len(ids)] = ids
    return tables


def tables_of(w) -> np.ndarray:
    if w.block_tables is not None:
        return np.ascontiguousarray(w.block_tables, dtype=np.int32)
    return replay_trace(w.trace, w.num_blocks, w.target_rids, w.M)


class OracleStep:
    """The oracle's view of one decode step of workload `w`.

    seqs: evaluate only these batch rows (their blocks are written from every
    history token that lands in them, so each block's contents, and for fp8
    its scale, are exactly those of the full workload).
    tables: block tables another implementation used for this workload.  The
    oracle always builds its own (its allocator replaying the workload's
    trace) and only checks that they are the same.
    """

    def __init__(self, w, seqs: Optional[Sequence[int]] = None, tables: Optional[np.ndarray] = None):
        self.w = w
        self.tables = tables_of(w)
        if tables is not None and not np.array_equal(np.asarray(tables), self.tables):
            raise AssertionError("the given block tables differ from the oracle's own for this workload")
        self.seqs = np.arange(w.B) if seqs is None else np.asarray(sorted(set(int(s) for s in seqs)))
        lens = np.asarray(w.seq_lens, dtype=np.int32)
        used = set()
        for b in self.seqs:
            nb = -(-int(lens[b]) // w.bs)
            used.update(int(x) for x in self.tables[b, :nb])
        self.cache = Cache(w.num_blocks, w.Hkv, w.d, w.bs, w.kv)
        if len(w.fill_seq):
            slots = slot_mapping(self.tables, w.fill_seq, w.fill_pos, w.bs)
            if seqs is None:
                idx = np.arange(len(slots))
            else:
                idx = np.flatnonzero(np.isin(slots // w.bs, np.fromiter(used, dtype=np.int64)))
            if len(idx):
                sel = torch.from_numpy(idx).to(w.k_fill.device)
                self.cache.append(w.k_fill[sel].cpu(), w.v_fill[sel].cpu(), slots[idx])
        # the step's append: each evaluated sequence's new token at position len-1
        pos = np.maximum(lens - 1, 0).astype(np.int32)
        self.step_slots = slot_mapping(self.tables, np.arange(w.B, dtype=np.int32), pos, w.bs)
        self.step_slots[lens <= 0] = -1

    def append(self):
        w = self.w
        sl = np.full(w.B, -1, dtype=np.int64)
        sl[self.seqs] = self.step_slots[self.seqs]
        self.cache.append(w.k_new.cpu(), w.v_new.cpu(), sl)

    def decode(self, threads: int = 1, part_blocks: int = 0) -> np.ndarray:
        """Outputs [len(seqs), Hq, d] fp64 for the evaluated rows."""
        w = self.w
        q = w.q.cpu()[self.seqs]
        return decode_attention(self.cache, q, self.tables[self.seqs], np.asarray(w.seq_lens)[self.seqs],
                                w.Hq, w.scale, part_blocks=part_blocks, threads=threads)
