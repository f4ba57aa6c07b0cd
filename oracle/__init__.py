"""CPU oracle for paged decode attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline / reference arm are the only callers.  The product library never
imports, links or executes anything in this directory, and this directory
imports nothing from the product.

The arithmetic lives in ``pa_oracle.c`` (plain C, fp64), compiled by
``build()`` with gcc.  This module only marshals numpy arrays into it.
Each wrapper names the page section its definition follows; see the C file.

Parity status of each function (what pins it, in tests/test_oracle_*.py):
  decode_attention        brute-force dense attention, cached == causal, closed forms
  decode_attention_split  equals decode_attention for every partition size
  prefill_attention       whole-sequence chunks equal a library causal attention
                          (torch, fp64); one-token chunks equal decode_attention;
                          a verify chunk equals the sequential decode steps
  kv_append (bf16)        exact copy: checked against direct indexing
  kv_append (fp8)         scale == absmax/448, round-trip bounds, brute-force encode
  int8 codec / append     numpy rint + clip on fp32 quotients, the growth / restart /
                          zero cases; attention on the int8 cache against torch
  int4 codec / append     the same pins with 7 in place of 127, plus the nibble order
                          (element 2j low, 2j+1 high) read back by hand; attention on
                          the int4 cache against torch on the unpacked values
  e4m3_encode/value       nearest-value brute force over the 256-code table, format facts
  kv_bytes/blocks_for     the pages' printed per-token sizes and block counts
  sched_*                 the pages' printed iteration counts
  sched_continuous_kv     equals sched_continuous when memory never binds; equal-size
                          requests under a pool of k reservations behave as k slots
  Allocator               lowest-id / refcount invariants on hand-checked traces
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libpa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c to _build/libpa_oracle.so (gcc, no contraction of fp32 ops)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-Wall",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, u64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        sig = {
            "or_bf16_value": (dbl, [ctypes.c_uint16]),
            "or_e4m3_value": (dbl, [ctypes.c_uint8]),
            "or_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "or_kv_bytes": (u64, [i64, i64, i64, i64, i64, i64]),
            "or_blocks_for_tokens": (i64, [i64, i64]),
            "or_sched_static": (i32, [P, i32, i32, P]),
            "or_sched_continuous": (i32, [P, i32, i32, P]),
            "or_alloc_create": (P, [i32]),
            "or_alloc_destroy": (None, [P]),
            "or_alloc_num_free": (i32, [P]),
            "or_alloc_alloc": (i32, [P, i32, P]),
            "or_alloc_free": (i32, [P, P, i32]),
            "or_alloc_share": (i32, [P, P, i32]),
            "or_alloc_refcount": (i32, [P, i32]),
            "or_slot_mapping": (i32, [P, i32, P, P, i32, i32, P]),
            "or_sched_continuous_kv": (i32, [P, i32, P, P, i32, i32, i64, i32, P, P, P, P, P]),
            "or_kv_append_bf16": (i32, [P, P, P, P, P, i32, i64, i32, i32, i32]),
            "or_kv_append_fp8": (i32, [P, P, P, P, P, P, P, i32, i64, i32, i32, i32]),
            "or_kv_append_int8": (i32, [P, P, P, P, P, P, P, i32, i64, i32, i32, i32]),
            "or_int8_value": (dbl, [ctypes.c_uint8]),
            "or_int8_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "or_kv_append_int4": (i32, [P, P, P, P, P, P, P, i32, i64, i32, i32, i32]),
            "or_int4_value": (dbl, [ctypes.c_uint8]),
            "or_int4_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "or_decode_attention": (i32, [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                          i64, dbl, i32]),
            "or_decode_attention_split": (i32, [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                                i32, i64, dbl, i32, i32]),
            "or_prefill_attention": (i32, [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                           i64, dbl, i32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    """bf16 tensor/array -> uint16 bit patterns (numpy, C-contiguous)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy()
                                        .view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint16))


# ---------------------------------------------------------------- formats
def bf16_value(bits: int) -> float:
    return _load().or_bf16_value(int(bits))


def e4m3_value(code: int) -> float:
    return _load().or_e4m3_value(int(code))


def e4m3_encode(x: float) -> int:
    return int(_load().or_e4m3_encode(float(x)))


def int8_value(code: int) -> float:
    return float(_load().or_int8_value(int(code) & 0xFF))


def int8_encode(x: float) -> int:
    """Code byte (two's complement) of clamp(rint(x), -127, 127)."""
    return int(_load().or_int8_encode(float(x)))


def int4_value(nibble: int) -> float:
    return float(_load().or_int4_value(int(nibble) & 0xF))


def int4_encode(x: float) -> int:
    """Nibble (0..15, two's complement) of clamp(rint(x), -7, 7)."""
    return int(_load().or_int4_encode(float(x)))


_KV_CODE = {"bf16": 0, "fp8": 1, "int8": 2, "int4": 3}


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    f = _load().or_e4m3_encode
    flat = np.asarray(x, dtype=np.float32).ravel()
    return np.array([f(float(v)) for v in flat], dtype=np.uint8).reshape(np.shape(x))


# ---------------------------------------------------------------- accounting
def kv_bytes(layers, kv_heads, head_dim, dtype_bits, tokens, batch) -> int:
    return int(_load().or_kv_bytes(layers, kv_heads, head_dim, dtype_bits, tokens, batch))


def blocks_for_tokens(tokens, block_size) -> int:
    return int(_load().or_blocks_for_tokens(tokens, block_size))


# ---------------------------------------------------------------- scheduler
def _sched(fn, lens, slots):
    arr = np.ascontiguousarray(np.asarray(lens, dtype=np.int64))
    out = np.zeros(1, dtype=np.int64)
    rc = fn(_p(arr) if arr.size else None, int(arr.size), int(slots), _p(out))
    if rc != 0:
        raise ValueError("invalid scheduler arguments")
    return int(out[0])


def sched_static(lens, slots) -> int:
    return _sched(_load().or_sched_static, lens, slots)


def sched_continuous(lens, slots) -> int:
    return _sched(_load().or_sched_continuous, lens, slots)


# ---------------------------------------------------------------- allocator
class Allocator:
    """Reference-counted block pool; allocations take the lowest free ids."""

    def __init__(self, num_blocks: int):
        self._lib = _load()
        self._h = self._lib.or_alloc_create(int(num_blocks))
        if not self._h:
            raise MemoryError
        self.num_blocks = num_blocks

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.or_alloc_destroy(h)

    def alloc(self, n: int) -> np.ndarray:
        out = np.zeros(max(n, 1), dtype=np.int32)
        rc = self._lib.or_alloc_alloc(self._h, int(n), _p(out))
        if rc == -2:
            raise MemoryError("out of blocks")
        if rc != 0:
            raise ValueError("invalid allocation")
        return out[:n]

    def free(self, ids) -> None:
        a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        if self._lib.or_alloc_free(self._h, _p(a) if a.size else None, int(a.size)) != 0:
            raise ValueError("invalid free")

    def share(self, ids) -> None:
        a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        if self._lib.or_alloc_share(self._h, _p(a) if a.size else None, int(a.size)) != 0:
            raise ValueError("invalid share")

    def num_free(self) -> int:
        return int(self._lib.or_alloc_num_free(self._h))

    def refcount(self, i: int) -> int:
        return int(self._lib.or_alloc_refcount(self._h, int(i)))


def sched_continuous_kv(alloc: Allocator, block_size: int, prompt_lens, out_lens, max_num_seqs: int,
                        stop_iter: int = -1, M: int = 0) -> dict:
    """Iteration-level scheduling with KV admission on `alloc` (see the C file)."""
    p = np.ascontiguousarray(np.asarray(prompt_lens, dtype=np.int64))
    o = np.ascontiguousarray(np.asarray(out_lens, dtype=np.int64))
    n = len(p)
    it = np.zeros(1, np.int64)
    adm = np.zeros(max(n, 1), np.int64)
    fin = np.zeros(max(n, 1), np.int64)
    tables = np.zeros((max(n, 1), max(M, 1)), np.int32)
    lens = np.zeros(max(n, 1), np.int32)
    rc = _load().or_sched_continuous_kv(alloc._h, int(block_size), _p(p) if n else None,
                                        _p(o) if n else None, n, int(max_num_seqs), int(stop_iter),
                                        int(M), _p(it), _p(adm), _p(fin), _p(tables) if M > 0 else None,
                                        _p(lens))
    if rc != 0:
        raise ValueError("invalid scheduler arguments")
    return dict(iters=int(it[0]), admitted_at=adm[:n], finished_at=fin[:n], tables=tables[:n, :M],
                lens=lens[:n])


# ---------------------------------------------------------------- slots
def slot_mapping(tables: np.ndarray, seq: np.ndarray, pos: np.ndarray, block_size: int) -> np.ndarray:
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    seq = np.ascontiguousarray(seq, dtype=np.int32)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    out = np.zeros(max(len(seq), 1), dtype=np.int64)
    rc = _load().or_slot_mapping(_p(tables), int(tables.shape[1]), _p(seq), _p(pos), int(len(seq)),
                                 int(block_size), _p(out))
    if rc != 0:
        raise ValueError("position beyond the block table")
    return out[: len(seq)]


# ---------------------------------------------------------------- cache
class Cache:
    """Host-side paged cache in the shared layout [num_blocks][Hkv][bs][d]
    (int4: [num_blocks][Hkv][bs][d / 2] bytes, two codes per byte)."""

    def __init__(self, num_blocks, Hkv, d, bs, kv="bf16"):
        self.num_blocks, self.Hkv, self.d, self.bs, self.kv = num_blocks, Hkv, d, bs, kv
        if kv not in _KV_CODE:
            raise ValueError("kv must be bf16, fp8, int8 or int4")
        dt = np.uint8 if kv != "bf16" else np.uint16
        row = d // 2 if kv == "int4" else d
        # np.zeros maps lazily: only pages the appends touch take memory
        self.k = np.zeros((num_blocks, Hkv, bs, row), dtype=dt)
        self.v = np.zeros((num_blocks, Hkv, bs, row), dtype=dt)
        if kv != "bf16":
            self.k_scale = np.zeros((num_blocks, Hkv), dtype=np.float32)
            self.v_scale = np.zeros((num_blocks, Hkv), dtype=np.float32)
        else:
            self.k_scale = self.v_scale = None

    def append(self, k_new, v_new, slots: np.ndarray) -> None:
        kn, vn = _u16(k_new), _u16(v_new)
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        T = len(slots)
        lib = _load()
        if self.kv != "bf16":
            fn = {"fp8": lib.or_kv_append_fp8, "int8": lib.or_kv_append_int8,
                  "int4": lib.or_kv_append_int4}[self.kv]
            rc = fn(_p(self.k), _p(self.v), _p(self.k_scale), _p(self.v_scale), _p(kn), _p(vn), _p(slots), T,
                    self.num_blocks, self.Hkv, self.d, self.bs)
        else:
            rc = lib.or_kv_append_bf16(_p(self.k), _p(self.v), _p(kn), _p(vn), _p(slots), T,
                                       self.num_blocks, self.Hkv, self.d, self.bs)
        if rc != 0:
            raise ValueError("slot beyond the pool")


def decode_attention(cache: Cache, q, block_tables: np.ndarray, seq_lens: np.ndarray, Hq: int,
                     scale: float, part_blocks: int = 0, threads: int = 1) -> np.ndarray:
    """fp64 decode attention; returns out [B, Hq, d] float64.

    part_blocks > 0 evaluates the split-K form (partitions of part_blocks
    blocks merged by log-sum-exp).  threads > 1 runs disjoint ranges of the
    batch on a thread pool (the C code releases the GIL through ctypes).
    """
    qb = _u16(q)
    B = int(len(seq_lens))
    d = cache.d
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    M = int(tables.shape[1]) if tables.ndim == 2 else 0
    out = np.zeros((B, Hq, d), dtype=np.float64)
    lib = _load()
    fp8 = _KV_CODE[cache.kv]

    def run(b0, b1):
        if b1 <= b0:
            return 0
        args = [out[b0:b1].ctypes.data, qb[b0:b1].ctypes.data, _p(cache.k), _p(cache.v),
                _p(cache.k_scale), _p(cache.v_scale), tables[b0:b1].ctypes.data,
                lens[b0:b1].ctypes.data, b1 - b0, Hq, cache.Hkv, d, cache.bs, M, cache.num_blocks,
                float(scale), fp8]
        if part_blocks > 0:
            return lib.or_decode_attention_split(*args, int(part_blocks))
        return lib.or_decode_attention(*args)

    if threads <= 1 or B <= 1:
        rcs = [run(0, B)]
    else:
        # interleave rows over workers so long and short sequences mix
        order = list(range(B))
        with ThreadPoolExecutor(max_workers=threads) as ex:
            rcs = list(ex.map(lambda b: run(b, b + 1), order))
    if any(rc != 0 for rc in rcs):
        raise ValueError("invalid decode arguments (block id or length out of range)")
    return out


def prefill_attention(cache: Cache, q, block_tables: np.ndarray, seq_lens: np.ndarray,
                      q_start: np.ndarray, Hq: int, scale: float, threads: int = 1) -> np.ndarray:
    """fp64 multi-query (chunked-prefill / verify) attention; out [total_q, Hq, d].

    Sequence b's queries are rows q_start[b] .. q_start[b+1]-1 of q: the last
    C_b positions of its seq_lens[b] cached tokens, each attending causally.
    """
    qb = _u16(q)
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qs = np.ascontiguousarray(q_start, dtype=np.int32)
    B = int(len(lens))
    M = int(tables.shape[1]) if tables.ndim == 2 else 0
    d = cache.d
    out = np.zeros((int(qs[-1]) if len(qs) else 0, Hq, d), dtype=np.float64)
    lib = _load()
    fp8 = _KV_CODE[cache.kv]

    def run(b):
        qsb = np.ascontiguousarray(qs[b:b + 2] - qs[b])
        r0 = int(qs[b])
        if int(qs[b + 1]) == r0:
            return 0
        return lib.or_prefill_attention(out[r0:].ctypes.data, qb[r0:].ctypes.data, _p(cache.k), _p(cache.v),
                                        _p(cache.k_scale), _p(cache.v_scale), tables[b:b + 1].ctypes.data,
                                        lens[b:b + 1].ctypes.data, qsb.ctypes.data, 1, Hq, cache.Hkv, d,
                                        cache.bs, M, cache.num_blocks, float(scale), fp8)

    if threads <= 1 or B <= 1:
        rcs = [run(b) for b in range(B)]
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            rcs = list(ex.map(run, range(B)))
    if any(rc != 0 for rc in rcs):
        raise ValueError("invalid prefill arguments (block id, length or query count out of range)")
    return out
