"""The oracle side of prefix-cached serving: the same host rules as the
library's BlockManager, restated over the oracle's allocator, prefix cache
and copy-on-write, so that a test can replay one request trace on both and
compare tables, reference counts and (on the GPU) cache bytes and outputs.
"""
from typing import Dict, List

import oracle
from oracle.prefix import PrefixCache, cow


class OracleManager:
    def __init__(self, num_blocks: int, bs: int, prefix_caching: bool = True):
        self.bs = bs
        self.alloc = oracle.Allocator(num_blocks)
        self.cache = PrefixCache(self.alloc, bs) if prefix_caching else None
        self.tokens: Dict[int, List[int]] = {}
        self.blocks: Dict[int, List[int]] = {}

    def _take(self, n):
        if n <= 0:
            return []
        if n > self.alloc.num_free() and self.cache is not None:
            self.cache.evict(n - self.alloc.num_free())
        return [int(x) for x in self.alloc.alloc(n)]

    def add(self, sid, tokens):
        toks = [int(t) for t in tokens]
        shared = self.cache.match(toks) if self.cache is not None else []
        need = -(-len(toks) // self.bs) - len(shared)
        try:
            own = self._take(need)
        except MemoryError:
            self.alloc.free(shared)
            raise
        self.tokens[sid], self.blocks[sid] = toks, list(shared) + own
        return len(shared) * self.bs

    def commit(self, sid):
        if self.cache is not None:
            self.cache.insert(self.tokens[sid], self.blocks[sid])

    def fork(self, child, parent):
        self.alloc.share(self.blocks[parent])
        self.tokens[child] = list(self.tokens[parent])
        self.blocks[child] = list(self.blocks[parent])

    def append(self, sid, token):
        toks, blocks = self.tokens[sid], self.blocks[sid]
        pos = len(toks)
        j = pos // self.bs
        copy = None
        if j == len(blocks):
            blocks.append(self._take(1)[0])
        else:
            try:
                dst, must_copy = cow(self.alloc, blocks[j])
            except MemoryError:
                if self.cache is None or self.cache.evict(1) == 0:
                    raise
                dst, must_copy = cow(self.alloc, blocks[j])
            if must_copy:
                copy = (blocks[j], dst)
            blocks[j] = dst
        toks.append(int(token))
        return blocks[j] * self.bs + pos % self.bs, copy

    def free(self, sid):
        self.alloc.free(self.blocks.pop(sid))
        del self.tokens[sid]
