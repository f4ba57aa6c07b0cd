"""Seeded synthetic inputs for paged decode attention.

This module is shared by the oracle tests, the CUDA parity tests and the
benchmark.  It holds random-number draws and data shaping only: no attention
arithmetic, no slot arithmetic, no block allocation.  Where a workload needs
block tables produced by a block allocator, this module emits the *operation
trace* (allocate n blocks for request r / free request r / share request r's
blocks with request s) and the caller replays it on whichever allocator it
tests.

Workload shapes follow the pages' description of decode over a paged cache:
  * "KV cache & continuous batching" (docs.masst.dev), section "KV cache
    memory math": Llama-3-8B has 8 KV heads of width 128 (GQA), Llama-3-70B
    64 query / 8 KV heads.
  * same page, section "2. PagedAttention": 16-token blocks, per-request block
    tables naming non-contiguous physical blocks.
  * "LLM Inference Optimization" (adaptiverecall.com), section "KV Cache
    Management": 100 requests sharing one system prompt share its KV.

Randomness: integer draws (lengths, permutations, traces) use numpy PCG64
seeded per sub-stream; tensor values are N(0,1) fp32 drawn with a torch
generator and rounded to bf16 (round-to-nearest-even, torch's conversion).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

BASE_SEED = 294

# name -> static shape parameters
CONFIGS: Dict[str, dict] = {
    "tiny": dict(index=0, Hq=4, Hkv=2, d=64, bs=16, kv="bf16", B=4, num_blocks=64),
    "8b": dict(index=1, Hq=32, Hkv=8, d=128, bs=16, kv="bf16", B=64, num_blocks=40000),
    "70b": dict(index=2, Hq=64, Hkv=8, d=128, bs=16, kv="bf16", B=256, num_blocks=65536),
    "long": dict(index=3, Hq=32, Hkv=8, d=128, bs=16, kv="bf16", B=4, num_blocks=32768),
    "fp8prefix": dict(index=4, Hq=32, Hkv=32, d=128, bs=32, kv="fp8", B=128, num_blocks=8192),
    # the 8b workload (same seed, same inputs) on an int8 cache
    "8b-int8": dict(index=1, Hq=32, Hkv=8, d=128, bs=16, kv="int8", B=64, num_blocks=40000),
    # and on an int4 cache (two codes per byte)
    "8b-int4": dict(index=1, Hq=32, Hkv=8, d=128, bs=16, kv="int4", B=64, num_blocks=40000),
}

DESCRIPTIONS = {
    "tiny": "4 seqs, lens {1,17,50,100}, Hq 4 / Hkv 2, d 64, bs 16, bf16, 64-block pool",
    "8b": "Llama-3-8B-shaped layer: Hq 32 / Hkv 8, d 128, bs 16, bf16, B 64, lens U[128,4096], 40000-block pool",
    "70b": "Llama-3-70B-shaped continuous-batching step: Hq 64 / Hkv 8, d 128, bs 16, bf16, B 256, "
           "len = lognormal(median 512, sigma 1, clip [16,6144]) + U[1,2048], tables from an admit/finish trace",
    "long": "long context: Hq 32 / Hkv 8, d 128, bs 16, bf16, B 4 x 131072 tokens, K scaled 0.5",
    "8b-int8": "the 8b workload on an int8 cache (per-(block, head) scales): Hq 32 / Hkv 8, d 128, bs 16, "
               "B 64, lens U[128,4096]",
    "8b-int4": "the 8b workload on an int4 cache (4-bit codes, two per byte, per-(block, head) scales): "
               "Hq 32 / Hkv 8, d 128, bs 16, B 64, lens U[128,4096]",
    "fp8prefix": "shared-prefix MHA, fp8 e4m3 cache: Hq=Hkv=32, d 128, bs 32, B 128 "
                 "(100 x [2048 shared + 256 own], 28 x U[256,8192])",
}

# Sub-stream ids (fixed so that each component's draws are independent of the others).
_S_LENS, _S_TABLES, _S_Q, _S_K, _S_V, _S_TRACE, _S_KNEW, _S_VNEW = range(8)


def _np_rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def _torch_gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + stream)
    return g


def randn_bf16(shape, seed: int, stream: int, device="cpu", mult: float = 1.0,
               chunk: int = 1 << 26) -> torch.Tensor:
    """N(0,1) fp32 draws rounded to bf16, drawn in chunks to bound fp32 temporaries."""
    g = _torch_gen(seed, stream, device)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        if mult != 1.0:
            x.mul_(mult)
        flat[s:e] = x.to(torch.bfloat16)
    return out


@dataclasses.dataclass
class TraceOp:
    """One allocator operation of a seeded admit/finish trace.

    kind: "alloc" (n blocks appended to request rid's table), "free" (release
    every block of rid), "share" (the first n blocks of request `src`'s table
    are appended to rid's table, taking a reference on each).
    """
    kind: str
    rid: int
    n: int = 0
    src: int = -1


@dataclasses.dataclass
class Workload:
    name: str
    Hq: int
    Hkv: int
    d: int
    bs: int
    kv: str                     # "bf16", "fp8", "int8" or "int4"
    B: int
    num_blocks: int
    M: int                      # columns of block_tables
    scale: float                # softmax scale 1/sqrt(d)
    seq_lens: np.ndarray        # int32 [B], includes the token appended this step
    # Either explicit tables (int32 [B, M], -1 padded) or a trace to replay.
    block_tables: Optional[np.ndarray]
    trace: Optional[List[TraceOp]]
    target_rids: Optional[List[int]]   # request id of each batch row in the trace
    # KV history to write before the step: token i is position fill_pos[i] of
    # sequence fill_seq[i]; runs of one sequence are in increasing position order.
    fill_seq: np.ndarray        # int32 [T_fill]
    fill_pos: np.ndarray        # int32 [T_fill]
    k_fill: torch.Tensor        # bf16 [T_fill, Hkv, d]
    v_fill: torch.Tensor
    # The step's new token per sequence (position seq_lens[b]-1).
    k_new: torch.Tensor         # bf16 [B, Hkv, d]
    v_new: torch.Tensor
    q: torch.Tensor             # bf16 [B, Hq, d]
    desc: str = ""

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


def _tables_from_perm(lens: np.ndarray, bs: int, M: int, perm: np.ndarray) -> np.ndarray:
    """Each sequence takes the next ceil(len/bs) ids of a seeded permutation."""
    B = len(lens)
    tables = np.full((B, M), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        nb = -(-int(lens[b]) // bs)
        tables[b, :nb] = perm[pos:pos + nb]
        pos += nb
    assert pos <= len(perm)
    return tables


def _history(lens: np.ndarray, skip_before: Optional[np.ndarray] = None):
    """(seq, pos) pairs of the cached history: positions 0..len-2 of every sequence."""
    seqs, poss = [], []
    for b, L in enumerate(lens):
        lo = 0 if skip_before is None else int(skip_before[b])
        n = int(L) - 1 - lo
        if n > 0:
            seqs.append(np.full(n, b, dtype=np.int32))
            poss.append(np.arange(lo, L - 1, dtype=np.int32))
    if not seqs:
        return np.zeros(0, np.int32), np.zeros(0, np.int32)
    return np.concatenate(seqs), np.concatenate(poss)


def _values(seed, T_fill, B, Hq, Hkv, d, device, k_mult=1.0):
    return dict(
        q=randn_bf16((B, Hq, d), seed, _S_Q, device),
        k_fill=randn_bf16((T_fill, Hkv, d), seed, _S_K, device, mult=k_mult),
        v_fill=randn_bf16((T_fill, Hkv, d), seed, _S_V, device),
        k_new=randn_bf16((B, Hkv, d), seed, _S_KNEW, device, mult=k_mult),
        v_new=randn_bf16((B, Hkv, d), seed, _S_VNEW, device),
    )


def _trace_70b(rng: np.random.Generator, prompt_law, prompt: np.ndarray, lens: np.ndarray,
               bs: int, num_blocks: int) -> Tuple[List[TraceOp], List[int]]:
    """Seeded admit/finish trace that fragments the pool before the targets run.

    Counting only (no block ids): the trace records how many blocks each op
    takes, so any allocator with the same capacity can replay it.
      1. four warm-up rounds: admit fillers (prompt-law lengths) until at least
         60% of the pool is taken, then finish a random half of them;
      2. admit the B targets with their prompt blocks;
      3. iterate: every unfinished target gains one token (one more block at a
         block boundary) and every live filler finishes with probability 0.01,
         until each target holds ceil(len/bs) blocks.
    When an allocation would not fit, a random live filler finishes first.
    """
    ops: List[TraceOp] = []
    free = num_blocks
    live: Dict[int, int] = {}   # filler rid -> blocks held
    next_rid = 0

    def finish(rid):
        nonlocal free
        free += live.pop(rid)
        ops.append(TraceOp("free", rid))

    def make_room(n):
        while free < n:
            assert live, "trace cannot fit"
            rid = sorted(live)[int(rng.integers(len(live)))]
            finish(rid)

    for _ in range(4):
        while num_blocks - free < 0.6 * num_blocks:
            n = -(-int(prompt_law(rng)) // bs)
            if n > free:
                break
            ops.append(TraceOp("alloc", next_rid, n))
            live[next_rid] = n
            free -= n
            next_rid += 1
        rids = sorted(live)
        kill = rng.permutation(len(rids))[: len(rids) // 2]
        for i in sorted(kill):
            finish(rids[i])

    B = len(lens)
    targets = []
    have = np.zeros(B, dtype=np.int64)
    cur = np.minimum(prompt, lens)
    for b in range(B):
        rid = next_rid
        next_rid += 1
        targets.append(rid)
        n = -(-int(cur[b]) // bs)
        make_room(n)
        ops.append(TraceOp("alloc", rid, n))
        free -= n
        have[b] = n
    need = -(-lens.astype(np.int64) // bs)
    while (have < need).any():
        for b in range(B):
            if cur[b] < lens[b]:
                cur[b] += 1
                nb = -(-int(cur[b]) // bs)
                if nb > have[b]:
                    make_room(nb - have[b])
                    ops.append(TraceOp("alloc", targets[b], int(nb - have[b])))
                    free -= int(nb - have[b])
                    have[b] = nb
        for rid in sorted(live):
            if rng.random() < 0.01:
                finish(rid)
    return ops, targets


def _trace_prefix(rng: np.random.Generator, n_shared: int, prefix_blocks: int,
                  own_blocks: int, indep_blocks: np.ndarray, num_blocks: int):
    """Scramble the pool, then build 100 sequences over one shared prefix.

    Warm-up: allocate random-sized filler requests until ~70% full, finish a
    random half, twice.  Then the first shared sequence allocates the prefix
    blocks and its own, each later shared sequence takes a reference on the
    first one's blocks (so the prefix blocks end with n_shared references) and
    allocates its own, and the independent sequences allocate theirs.
    """
    ops: List[TraceOp] = []
    free = num_blocks
    live: Dict[int, int] = {}
    rid = 0
    for _ in range(2):
        while num_blocks - free < 0.7 * num_blocks:
            n = int(rng.integers(1, 65))
            ops.append(TraceOp("alloc", rid, n))
            live[rid] = n
            free -= n
            rid += 1
        rids = sorted(live)
        for i in sorted(rng.permutation(len(rids))[: len(rids) // 2]):
            r = rids[i]
            free += live.pop(r)
            ops.append(TraceOp("free", r))
    # release all fillers except a scattered third, so the targets fit
    rids = sorted(live)
    for i in sorted(rng.permutation(len(rids))[: (2 * len(rids)) // 3]):
        r = rids[i]
        free += live.pop(r)
        ops.append(TraceOp("free", r))
    # the first sequence computes the prefix; the others take references on its blocks
    prefix_rid = rid
    targets = []
    for i in range(n_shared):
        if i == 0:
            ops.append(TraceOp("alloc", rid, prefix_blocks))
        else:
            ops.append(TraceOp("share", rid, n=prefix_blocks, src=prefix_rid))
        ops.append(TraceOp("alloc", rid, own_blocks))
        targets.append(rid)
        rid += 1
    for nb in indep_blocks:
        ops.append(TraceOp("alloc", rid, int(nb)))
        targets.append(rid)
        rid += 1
    return ops, targets


def make(name: str, device="cpu", B: Optional[int] = None, seq_len: Optional[int] = None,
         seed: Optional[int] = None) -> Workload:
    """Build a seeded workload.

    B / seq_len shrink a configuration for parity tests (same recipe, fewer
    or shorter sequences); the defaults give the full configuration.
    """
    cfg = dict(CONFIGS[name])
    idx = cfg.pop("index")
    seed = BASE_SEED * 100 + idx if seed is None else seed
    Hq, Hkv, d, bs, kv = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["bs"], cfg["kv"]
    num_blocks = cfg["num_blocks"]
    Bfull = cfg["B"]
    scale = 1.0 / math.sqrt(d)
    rl = _np_rng(seed, _S_LENS)
    rt = _np_rng(seed, _S_TABLES)
    trace = targets = tables = None
    k_mult = 1.0

    if name == "tiny":
        lens = np.array([1, 17, 50, 100], dtype=np.int32)
        if B is not None:
            lens = lens[:B]
        M = 7
        perm = rt.permutation(num_blocks).astype(np.int32)
        tables = _tables_from_perm(lens, bs, M, perm)
        fs, fp = _history(lens)
    elif name in ("8b", "8b-int8", "8b-int4"):
        Bn = Bfull if B is None else B
        hi = 4096 if seq_len is None else seq_len
        lens = rl.integers(128 if seq_len is None else 1, hi + 1, size=Bn).astype(np.int32)
        M = 256 if seq_len is None else -(-hi // bs)
        if B is not None and B < Bfull:
            num_blocks = max(-(-num_blocks * Bn // Bfull), int(np.sum(-(-lens // bs))))   # same pool density
        perm = rt.permutation(num_blocks).astype(np.int32)
        tables = _tables_from_perm(lens, bs, M, perm)
        fs, fp = _history(lens)
    elif name == "70b":
        Bn = Bfull if B is None else B
        cap = 6144 if seq_len is None else seq_len

        def prompt_law(r):
            x = int(round(math.exp(math.log(512.0) + r.standard_normal())))
            return min(max(x, 16), cap)

        prompt = np.array([prompt_law(rl) for _ in range(Bn)], dtype=np.int64)
        gen = rl.integers(1, (2048 if seq_len is None else max(1, seq_len // 3)) + 1, size=Bn)
        lens = (prompt + gen).astype(np.int32)
        M = -(-int((6144 + 2048) if seq_len is None else (cap + max(1, seq_len // 3))) // bs)
        if B is not None and B < Bfull:
            num_blocks = max(4 * int(np.sum(-(-lens // bs))), 256)
        trace, targets = _trace_70b(_np_rng(seed, _S_TRACE), prompt_law, prompt,
                                    lens.astype(np.int64), bs, num_blocks)
        fs, fp = _history(lens)
    elif name == "long":
        Bn = Bfull if B is None else B
        L = 131072 if seq_len is None else seq_len
        lens = np.full(Bn, L, dtype=np.int32)
        M = -(-L // bs)
        num_blocks = max(num_blocks, Bn * M) if seq_len is None else Bn * M + 16
        perm = rt.permutation(num_blocks).astype(np.int32)
        tables = _tables_from_perm(lens, bs, M, perm)
        fs, fp = _history(lens)
        k_mult = 0.5
    elif name == "fp8prefix":
        n_shared, n_indep = 100, 28
        prefix_tok, own_tok = 2048, 256
        hi = 8192
        if B is not None:
            n_shared = min(n_shared, max(1, (B * 100) // 128))
            n_indep = B - n_shared
        if seq_len is not None:
            prefix_tok = max(bs, (seq_len // 2) // bs * bs)
            own_tok = max(bs, (seq_len // 4) // bs * bs)
            hi = seq_len
        indep = rl.integers(min(256, hi), hi + 1, size=n_indep)
        lens = np.concatenate([np.full(n_shared, prefix_tok + own_tok), indep]).astype(np.int32)
        M = -(-max(int(lens.max()), prefix_tok + own_tok) // bs)
        prefix_blocks = prefix_tok // bs
        own_blocks = own_tok // bs
        indep_blocks = -(-indep // bs)
        if B is not None or seq_len is not None:
            num_blocks = max(2 * int(prefix_blocks + n_shared * own_blocks + indep_blocks.sum()), 256)
        trace, targets = _trace_prefix(_np_rng(seed, _S_TRACE), n_shared, prefix_blocks, own_blocks,
                                       indep_blocks, num_blocks)
        # history: the prefix once (through sequence 0), then each sequence's own tokens
        skip = np.zeros(len(lens), dtype=np.int64)
        skip[1:n_shared] = prefix_tok
        fs, fp = _history(lens, skip)
    else:
        raise KeyError(name)

    Bn = len(lens)
    vals = _values(seed, len(fs), Bn, Hq, Hkv, d, device, k_mult)
    return Workload(name=name, Hq=Hq, Hkv=Hkv, d=d, bs=bs, kv=kv, B=Bn, num_blocks=num_blocks,
                    M=M, scale=scale, seq_lens=lens, block_tables=tables, trace=trace,
                    target_rids=targets, fill_seq=fs, fill_pos=fp, desc=DESCRIPTIONS[name],
                    **vals)


@dataclasses.dataclass
class ServingScenario:
    """Requests with one shared system prompt, forks, then decode steps.

    Request r's tokens are prompt + suffix[r]; its KV for every position is
    k_pre[r] / v_pre[r] (a request that reuses a cached prefix writes only the
    positions after it).  After all requests are admitted, forks[i] =
    (parent) makes sequence R + i a copy of sequence `parent`.  Each step
    appends one token to every live sequence (ids 0 .. R + len(forks) - 1, in
    order): tokens[s][i], with new K/V k_new[s][i] / v_new[s][i] and query
    q[s][i].
    """
    Hq: int
    Hkv: int
    d: int
    bs: int
    kv: str
    num_blocks: int
    M: int
    scale: float
    prompt: List[int]
    requests: List[List[int]]
    k_pre: List[torch.Tensor]           # bf16 [len_r, Hkv, d]
    v_pre: List[torch.Tensor]
    forks: List[int]
    tokens: List[List[int]]             # [steps][n_seq]
    q: List[torch.Tensor]               # [steps] bf16 [n_seq, Hq, d]
    k_new: List[torch.Tensor]           # [steps] bf16 [n_seq, Hkv, d]
    v_new: List[torch.Tensor]

    @property
    def n_seq(self) -> int:
        return len(self.requests) + len(self.forks)


def serving_scenario(layer: str = "8b", R: int = 6, n_forks: int = 2, steps: int = 20, seed: int = 7,
                     device="cpu") -> ServingScenario:
    """A small prefix-sharing trace on one layer's shape (the system prompt ends
    mid-block, so its last block is recomputed per request; suffixes span 0 to
    2 blocks; forks share a parent's partly filled last block)."""
    cfg = CONFIGS[layer]
    Hq, Hkv, d, bs, kv = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["bs"], cfg["kv"]
    rng = _np_rng(seed, 50)
    P = 5 * bs + 7
    prompt = [int(x) for x in rng.integers(0, 32000, P)]
    requests = [prompt + [int(x) for x in rng.integers(32000, 64000, int(rng.integers(0, 2 * bs + 1)))]
                for _ in range(R)]
    forks = [int(x) for x in rng.integers(0, R, n_forks)]
    n_seq = R + n_forks
    k_pre = [randn_bf16((len(t), Hkv, d), seed, 100 + r, device) for r, t in enumerate(requests)]
    v_pre = [randn_bf16((len(t), Hkv, d), seed, 200 + r, device) for r, t in enumerate(requests)]
    tokens = [[int(x) for x in rng.integers(0, 64000, n_seq)] for _ in range(steps)]
    q = [randn_bf16((n_seq, Hq, d), seed, 300 + s, device) for s in range(steps)]
    # unit-variance values like the history: a block filled one token at a time
    # still grows its fp8 scale whenever a new row sets a new absmax
    k_new = [randn_bf16((n_seq, Hkv, d), seed, 400 + s, device) for s in range(steps)]
    v_new = [randn_bf16((n_seq, Hkv, d), seed, 500 + s, device) for s in range(steps)]
    longest = max(len(t) for t in requests) + steps
    M = -(-longest // bs) + 1
    num_blocks = 4 * n_seq * M
    return ServingScenario(Hq=Hq, Hkv=Hkv, d=d, bs=bs, kv=kv, num_blocks=num_blocks, M=M,
                           scale=1.0 / math.sqrt(d), prompt=prompt, requests=requests, k_pre=k_pre,
                           v_pre=v_pre, forks=forks, tokens=tokens, q=q, k_new=k_new, v_new=v_new)


@dataclasses.dataclass
class PrefillWorkload(Workload):
    """A decode-shaped workload whose last C_b tokens per sequence are a query
    chunk: q_chunk [q_start[-1], Hq, d], sequence b's rows from q_start[b].
    The history (fill_*) covers every position, the chunk's included."""
    q_chunk: Optional[torch.Tensor] = None
    q_start: Optional[np.ndarray] = None
    max_q: int = 0


def make_prefill(layer: str, ctx: List[int], chunk: List[int], seed: int = 11, device="cpu",
                 Hq: Optional[int] = None, Hkv: Optional[int] = None, bs: Optional[int] = None,
                 kv: Optional[str] = None) -> PrefillWorkload:
    """Sequences with ctx[b] earlier tokens and a chunk of chunk[b] query tokens
    (seq_len = ctx + chunk) on one layer's shape and cache type (or `kv`),
    tables from a seeded permutation of the pool."""
    cfg = dict(CONFIGS[layer])
    kv = cfg["kv"] if kv is None else kv
    Hq = cfg["Hq"] if Hq is None else Hq
    Hkv = cfg["Hkv"] if Hkv is None else Hkv
    bs = cfg["bs"] if bs is None else bs
    d = cfg["d"]
    lens = (np.asarray(ctx, dtype=np.int64) + np.asarray(chunk, dtype=np.int64)).astype(np.int32)
    B = len(lens)
    M = max(1, int(max(-(-int(n) // bs) for n in lens)))
    blocks = int(sum(-(-int(n) // bs) for n in lens))
    num_blocks = max(blocks + 8, 64)
    rng = _np_rng(seed, _S_TABLES)
    tables = _tables_from_perm(lens, bs, M, rng.permutation(num_blocks).astype(np.int32))
    fs, fp = _history(lens + 1)          # every position 0 .. len-1, the chunk's too
    vals = _values(seed, len(fs), B, Hq, Hkv, d, device)
    q_start = np.concatenate([[0], np.cumsum(np.asarray(chunk, dtype=np.int64))]).astype(np.int32)
    q_chunk = randn_bf16((int(q_start[-1]), Hq, d), seed, 40, device)
    return PrefillWorkload(name="prefill-" + layer, Hq=Hq, Hkv=Hkv, d=d, bs=bs, kv=kv, B=B,
                           num_blocks=num_blocks, M=M, scale=1.0 / math.sqrt(d), seq_lens=lens,
                           block_tables=tables, trace=None, target_rids=None, fill_seq=fs, fill_pos=fp,
                           desc="prefill chunks %s over contexts %s" % (list(chunk)[:4], list(ctx)[:4]),
                           q_chunk=q_chunk, q_start=q_start, max_q=int(max(chunk) if len(chunk) else 0),
                           **vals)


def roofline_bytes(w: Workload) -> dict:
    """Bytes the step must move at minimum: K/V history read once, q read, out written.

    Counts each logical token of each sequence (a shared prefix counts once per
    sequence: "logical"), and separately each distinct physical block once
    ("unique").  Element size 2 (bf16), 1 (fp8, int8) or 1/2 (int4) plus, for
    the coded caches, one fp32 scale per (block, kv_head) for K and for V.
    """
    tok_bytes = 2 * w.Hkv * {"bf16": 2 * w.d, "int4": w.d // 2}.get(w.kv, w.d)
    logical_tokens = int(np.sum(w.seq_lens.astype(np.int64)))
    qo = 2 * w.B * w.Hq * w.d * 2
    out = dict(logical_kv=logical_tokens * tok_bytes, q_out=qo)
    out["logical"] = out["logical_kv"] + qo
    return out
