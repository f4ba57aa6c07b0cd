"""Oracle prefix cache, copy-on-write and block copy (test infrastructure).

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests, the smoke
check and the benchmark's CPU legs are its only callers.

"KV cache & continuous batching", section "4. Prefix caching": the KV of a
shared prefix is computed once and reused; vLLM hashes prefix blocks and a
radix tree shares any prefix two requests have in common.  "LLM Serving - KV
Cache, Batching, Speculative Decoding", section "KV memory, paging and prefix
identity": reuse needs the exact token prefix.  "LLM Inference
Optimization", section "KV Cache Management": many requests with one system
prompt share its KV.

The plain definition used here: block j of a sequence holds the KV of tokens
[j*bs, (j+1)*bs), which depend on the tokens [0, (j+1)*bs) only, so the cache
is a dictionary from that whole token prefix (a tuple) to a physical block.
A lookup walks j = 0, 1, ... while the prefix is present.  No hashing, no
tree: the dictionary's own key comparison is the exact-prefix rule.

Readings the pages leave open (each stated where the product states it too):
  * only full blocks are cached;
  * a prefix already cached keeps its block when another sequence inserts the
    same prefix with a different block;
  * eviction frees, one block at a time, the least recently used chain end
    (no cached key extends it by one block) that only the cache references;
    every match or insert call advances a clock by one and stamps the entries
    it touches.  One call stamps one path, and a path has one end, so two
    chain ends never tie; the depth / block-id tie-breaks are only there to
    make the order total by construction;
  * copy-on-write: a writer that is the block's only user writes in place;
    otherwise it takes a fresh block (lowest free id) and drops its reference
    on the shared one.

Parity status: pinned in tests/test_oracle_prefix.py by hand-worked traces,
closed forms (the shared system prompt, a changed token at position p keeps
floor(p/bs) blocks) and a brute-force longest-common-prefix search.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np

from . import Allocator


class PrefixCache:
    def __init__(self, alloc: Allocator, block_size: int):
        self.alloc = alloc
        self.bs = int(block_size)
        self.clock = 0
        # token prefix (tuple, length a multiple of bs) -> [block, last_use]
        self.entries: Dict[Tuple[int, ...], List[int]] = {}

    def size(self) -> int:
        return len(self.entries)

    def match(self, tokens: Sequence[int], max_out: int = -1) -> List[int]:
        """Blocks of the longest cached prefix; the caller gets one reference each."""
        toks = tuple(int(t) for t in tokens)
        self.clock += 1
        out: List[int] = []
        j = 0
        while (j + 1) * self.bs <= len(toks) and (max_out < 0 or len(out) < max_out):
            key = toks[: (j + 1) * self.bs]
            if key not in self.entries:
                break
            out.append(self.entries[key][0])
            j += 1
        if out:
            self.alloc.share(out)
        for i in range(len(out)):
            self.entries[toks[: (i + 1) * self.bs]][1] = self.clock
        return out

    def insert(self, tokens: Sequence[int], blocks: Sequence[int]) -> None:
        toks = tuple(int(t) for t in tokens)
        full = min(len(toks) // self.bs, len(blocks))
        for j in range(full):
            if self.alloc.refcount(int(blocks[j])) <= 0:
                raise ValueError("block %d is not allocated" % int(blocks[j]))
        self.clock += 1
        for j in range(full):
            key = toks[: (j + 1) * self.bs]
            if key in self.entries:
                self.entries[key][1] = self.clock
            else:
                self.alloc.share([int(blocks[j])])
                self.entries[key] = [int(blocks[j]), self.clock]

    def _is_chain_end(self, key) -> bool:
        n = len(key) + self.bs
        return not any(len(k) == n and k[: len(key)] == key for k in self.entries)

    def evict(self, want: int) -> int:
        freed = 0
        while freed < want:
            cands = [k for k, (blk, _) in self.entries.items()
                     if self.alloc.refcount(blk) == 1 and self._is_chain_end(k)]
            if not cands:
                break
            # least recently used, then deepest (longest key), then lowest block id
            k = min(cands, key=lambda k: (self.entries[k][1], -len(k), self.entries[k][0]))
            self.alloc.free([self.entries.pop(k)[0]])
            freed += 1
        return freed

    def release(self) -> None:
        """Drop every reference the cache holds."""
        for blk, _ in self.entries.values():
            self.alloc.free([blk])
        self.entries.clear()


def cow(alloc: Allocator, block: int) -> Tuple[int, bool]:
    """(block to write into, whether the caller must copy the old contents)."""
    rc = alloc.refcount(int(block))
    if rc <= 0:
        raise ValueError("block %d is not allocated" % int(block))
    if rc == 1:
        return int(block), False
    fresh = int(alloc.alloc(1)[0])
    alloc.free([int(block)])
    return fresh, True


def copy_blocks(cache, src: Sequence[int], dst: Sequence[int]) -> None:
    """Block dst[i] of the oracle cache becomes a copy of block src[i]."""
    for s, d in zip(src, dst):
        cache.k[int(d)] = cache.k[int(s)]
        cache.v[int(d)] = cache.v[int(s)]
        if cache.k_scale is not None:
            cache.k_scale[int(d)] = cache.k_scale[int(s)]
            cache.v_scale[int(d)] = cache.v_scale[int(s)]
