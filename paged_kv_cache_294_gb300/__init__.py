"""Paged-KV decode attention for NVIDIA GB300 (sm_103a): Python binding.

A thin ctypes layer over libpagedattn.so whose functions carry the C ABI's
names (include/pa.h).  It converts torch tensors to device pointers and
checks dtypes and shapes; every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if the library cannot be
loaded, every call raises.

Tensor layouts (row-major):
  k_cache, v_cache  [num_blocks, Hkv, block_size, head_dim] bf16, uint8 (e4m3 codes) or
                    int8 (int8 codes); [num_blocks, Hkv, block_size, head_dim / 2] uint8
                    for int4 codes (two per byte), told apart from e4m3 by the last
                    dimension against head_dim (pa_copy_blocks: kv_dtype=PA_KV_INT4)
  k_scale, v_scale  [num_blocks, Hkv] float32 (coded caches only)
  q, out            [B, Hq, head_dim] bf16
  k_new, v_new      [T, Hkv, head_dim] bf16
  block_tables      [B, M] int32;  seq_lens [B] int32;  slot_mapping [T] int64
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

from . import _build

PA_OK, PA_ERR_INVALID, PA_ERR_OOM, PA_ERR_CUDA, PA_ERR_UNSUPPORTED = range(5)
PA_KV_BF16, PA_KV_FP8_E4M3, PA_KV_INT8, PA_KV_INT4 = 0, 1, 2, 3
PA_DEVERR_BLOCK_ID, PA_DEVERR_SEQ_LEN, PA_DEVERR_SLOT, PA_DEVERR_TIMEOUT = 1, 2, 4, 8

_lib = None


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s" % (what, status_string(status)))


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libpagedattn.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError("libpagedattn.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    P, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    sig = {
        "pa_status_string": (ctypes.c_char_p, [i32]),
        "pa_kv_append": (i32, [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]),
        "pa_decode_resolve_splits": (i32, [i32, i32, i32, i32]),
        "pa_decode_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "pa_decode_attention": (i32, [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                      ctypes.c_float, i32, P, sz, i32, P]),
        "pa_decode_step": (i32, [P, P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                 ctypes.c_float, i32, P, sz, i32, P]),
        "pa_decode_attention_static_ws": (i32, [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                ctypes.c_float, i32, i32, P]),
        "pa_prefill_attention": (i32, [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                       ctypes.c_float, i32, P]),
        "pa_get_device_error": (i32, [P, i32]),
        "pa_selftest_bounded_wait": (i32, [P]),
        "pa_allocator_create": (P, [i32, i32]),
        "pa_allocator_destroy": (None, [P]),
        "pa_block_alloc": (i32, [P, i32, P]),
        "pa_block_free": (i32, [P, P, i32]),
        "pa_block_share": (i32, [P, P, i32]),
        "pa_allocator_fail_nth_alloc": (i32, [P, i64]),
        "pa_allocator_num_free": (i32, [P]),
        "pa_allocator_num_blocks": (i32, [P]),
        "pa_allocator_refcount": (i32, [P, i32]),
        "pa_allocator_block_size": (i32, [P]),
        "pa_prefix_cache_create": (P, [P]),
        "pa_prefix_cache_destroy": (None, [P]),
        "pa_prefix_cache_size": (i32, [P]),
        "pa_prefix_match": (i32, [P, P, i64, P, i32, P]),
        "pa_prefix_insert": (i32, [P, P, i64, P, i32]),
        "pa_prefix_evict": (i32, [P, i32, P]),
        "pa_block_cow": (i32, [P, i32, P, P]),
        "pa_copy_blocks": (i32, [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]),
        "pa_blocks_for_tokens": (i64, [i64, i32]),
        "pa_kv_bytes": (u64, [i32, i32, i32, i32, i64, i64]),
        "pa_slot_mapping": (i32, [P, i32, P, P, i32, i32, P]),
        "pa_step_slots": (i32, [P, i32, P, i32, i32, P]),
        "pa_seq_admit": (i32, [P, P, P, i64, P, i32, P, P]),
        "pa_seq_append_slot": (i32, [P, P, P, P, i32, i64, P, P, P]),
        "pa_share_plan": (i32, [P, i32, P, i32, i32, i32, i32, P, P, P, i32, P, P]),
        "pa_decode_shared_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32, i32]),
        "pa_decode_step_shared": (i32, [P, P, P, P, P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                        i32, i32, ctypes.c_float, i32, P, sz, i32, P]),
        "pa_sched_simulate": (i32, [P, i32, i32, i32, P]),
        "pa_sched_continuous_kv": (i32, [P, P, P, i32, i32, i64, i32, P, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_string(s: int) -> str:
    return load().pa_status_string(int(s)).decode()


def _check(status: int, what: str):
    if status != PA_OK:
        raise PagedAttnError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _np_ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _stream(stream, device=None) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        if device is not None and stream.device != device:
            raise ValueError("stream is on %s, the call's tensors on %s" % (stream.device, device))
        return stream.cuda_stream
    return int(stream)


def _kv_dtype(cache: torch.Tensor, head_dim: Optional[int] = None) -> int:
    """Cache type from the tensor: a uint8 cache whose rows hold head_dim / 2
    bytes holds int4 codes, one with head_dim bytes e4m3 codes."""
    if cache.dtype == torch.bfloat16:
        return PA_KV_BF16
    if cache.dtype == torch.uint8:
        if head_dim is not None and cache.dim() == 4 and 2 * cache.shape[3] == head_dim:
            return PA_KV_INT4
        return PA_KV_FP8_E4M3
    if cache.dtype == torch.int8:
        return PA_KV_INT8
    raise TypeError("cache dtype must be bfloat16, uint8 (e4m3 or int4 codes) or int8")


def _row_len(kvd: int, d: int) -> int:
    """Last dimension of a cache tensor of type kvd for head_dim d."""
    return d // 2 if kvd == PA_KV_INT4 else d


def _need(t: torch.Tensor, dtype, name: str, dim: Optional[int] = None):
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dim is not None and t.dim() != dim:
        raise ValueError("%s must have %d dimensions" % (name, dim))


def _one_device(ref: torch.Tensor, **tensors) -> torch.device:
    """The call's device: ref's.  Every other tensor argument (None skipped)
    must be a CUDA tensor on that same device, checked before anything is
    launched (a host or foreign-device pointer handed to a kernel or a TMA
    map would be read by the GPU)."""
    dev = ref.device
    if dev.type != "cuda":
        raise ValueError("tensor arguments must be CUDA tensors")
    for name, t in tensors.items():
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
        if t.device != dev:
            raise ValueError("%s is on %s, the call's other tensors on %s" % (name, t.device, dev))
    return dev


def _call(dev: torch.device, what: str, fn, *args, stream=None):
    """Run a device entry point with `dev` current, on `stream` (default: the
    current torch stream of dev), and raise on a non-OK status."""
    with torch.cuda.device(dev):
        _check(fn(*args, _stream(stream, dev)), what)


# ------------------------------------------------------------------ device ops
def pa_kv_append(k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: Optional[torch.Tensor],
                 v_scale: Optional[torch.Tensor], k_new: torch.Tensor, v_new: torch.Tensor,
                 slot_mapping: torch.Tensor, stream=None) -> None:
    lib = load()
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    d = k_new.shape[2]
    kvd = _kv_dtype(k_cache, d)
    if kvd != PA_KV_BF16:
        _need(k_scale, torch.float32, "k_scale", 2)
        _need(v_scale, torch.float32, "v_scale", 2)
    nb, hkv, bs, dc = k_cache.shape
    T = slot_mapping.shape[0]
    if (dc != _row_len(kvd, d) or tuple(k_new.shape) != (T, hkv, d) or tuple(v_new.shape) != (T, hkv, d)
            or v_cache.shape != k_cache.shape):
        raise ValueError("shape mismatch between caches, new K/V and slot_mapping")
    dev = _one_device(k_new, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale, v_new=v_new,
                      slot_mapping=slot_mapping)
    _call(dev, "pa_kv_append", lib.pa_kv_append, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
          _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, nb, hkv, d, bs, kvd, stream=stream)


def pa_decode_resolve_splits(batch: int, num_kv_heads: int, max_blocks_per_seq: int,
                             num_splits: int = 0) -> int:
    return int(load().pa_decode_resolve_splits(batch, num_kv_heads, max_blocks_per_seq, num_splits))


def pa_decode_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                              max_blocks_per_seq: int, num_splits: int = 0) -> int:
    return int(load().pa_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                                max_blocks_per_seq, num_splits))


def pa_decode_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                        k_scale: Optional[torch.Tensor], v_scale: Optional[torch.Tensor],
                        block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                        num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                        stream=None) -> None:
    lib = load()
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, hq, d = q.shape
    kvd = _kv_dtype(k_cache, d)
    nb, hkv, bs, dc = k_cache.shape
    M = block_tables.shape[1]
    if (dc != _row_len(kvd, d) or tuple(out.shape) != (B, hq, d) or block_tables.shape[0] != B
            or seq_lens.shape[0] != B):
        raise ValueError("shape mismatch")
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dev = _one_device(q, out=out, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                      block_tables=block_tables, seq_lens=seq_lens, workspace=workspace)
    _call(dev, "pa_decode_attention", lib.pa_decode_attention, _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
          _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens), B, hq, hkv, d, bs, M, nb,
          float(scale), int(num_splits), _ptr(workspace), ws, kvd, stream=stream)


def pa_decode_step(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: Optional[torch.Tensor],
                   v_scale: Optional[torch.Tensor], block_tables: torch.Tensor, seq_lens: torch.Tensor,
                   scale: float, num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    """Append each sequence's new token (position seq_len-1) and attend, in one launch."""
    lib = load()
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, hq, d = q.shape
    kvd = _kv_dtype(k_cache, d)
    nb, hkv, bs, dc = k_cache.shape
    M = block_tables.shape[1]
    if (dc != _row_len(kvd, d) or tuple(out.shape) != (B, hq, d) or tuple(k_new.shape) != (B, hkv, d)
            or tuple(v_new.shape) != (B, hkv, d) or block_tables.shape[0] != B or seq_lens.shape[0] != B):
        raise ValueError("shape mismatch")
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dev = _one_device(q, out=out, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale,
                      v_scale=v_scale, block_tables=block_tables, seq_lens=seq_lens, workspace=workspace)
    _call(dev, "pa_decode_step", lib.pa_decode_step, _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
          _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens), B, hq, hkv, d, bs, M,
          nb, float(scale), int(num_splits), _ptr(workspace), ws, kvd, stream=stream)


PA_SHARE_MAX_ROWS = 8


def pa_share_plan(block_tables: np.ndarray, seq_lens: np.ndarray, block_size: int, group_rows: int,
                  min_blocks: int = 1, max_chunks: Optional[int] = None) -> dict:
    """Shared-prefix plan (host): dict(chunk_of [B], chunk_members [n, PA_SHARE_MAX_ROWS],
    chunk_blocks [n], max_chunk_blocks); chunk_of[b] = PA_SHARE_MAX_ROWS * chunk + slot or -1."""
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    n = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = len(n)
    if t.ndim != 2 or t.shape[0] != B:
        raise ValueError("block_tables must be [B, M] and seq_lens [B]")
    cap = B if max_chunks is None else int(max_chunks)
    chunk_of = np.full(max(B, 1), -1, np.int32)
    members = np.full((max(cap, 1), PA_SHARE_MAX_ROWS), -1, np.int32)
    blocks = np.zeros(max(cap, 1), np.int32)
    nc, mx = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().pa_share_plan(_np_ptr(t) if B else None, int(t.shape[1]), _np_ptr(n) if B else None, B,
                                int(block_size), int(group_rows), int(min_blocks), _np_ptr(chunk_of),
                                _np_ptr(members), _np_ptr(blocks), cap, ctypes.byref(nc), ctypes.byref(mx)),
           "pa_share_plan")
    return dict(chunk_of=chunk_of[:B], chunk_members=members[: nc.value], chunk_blocks=blocks[: nc.value],
                max_chunk_blocks=int(mx.value))


def pa_decode_shared_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                     max_blocks_per_seq: int, num_splits: int, max_chunk_blocks: int) -> int:
    return int(load().pa_decode_shared_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                                       max_blocks_per_seq, num_splits, max_chunk_blocks))


def pa_decode_step_shared(out: torch.Tensor, q: torch.Tensor, k_new: Optional[torch.Tensor],
                          v_new: Optional[torch.Tensor], k_cache: torch.Tensor, v_cache: torch.Tensor,
                          k_scale: Optional[torch.Tensor], v_scale: Optional[torch.Tensor], block_tables: torch.Tensor,
                          seq_lens: torch.Tensor, chunk_of: torch.Tensor, chunk_members: torch.Tensor,
                          chunk_blocks: torch.Tensor, max_chunk_blocks: int, scale: float, num_splits: int = 0,
                          workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """The decode step (k_new / v_new given) or attention alone (both None) with
    shared prefixes read once per chunk of sequences (plan from pa_share_plan,
    its arrays on the device)."""
    lib = load()
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(chunk_of, torch.int32, "chunk_of", 1)
    _need(chunk_members, torch.int32, "chunk_members", 2)
    _need(chunk_blocks, torch.int32, "chunk_blocks", 1)
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new are given together")
    B, hq, d = q.shape
    kvd = _kv_dtype(k_cache, d)
    nb, hkv, bs, dc = k_cache.shape
    M = block_tables.shape[1]
    n_chunks = int(chunk_blocks.shape[0])
    if (dc != _row_len(kvd, d) or tuple(out.shape) != (B, hq, d) or block_tables.shape[0] != B
            or seq_lens.shape[0] != B or chunk_of.shape[0] != B
            or tuple(chunk_members.shape) != (n_chunks, PA_SHARE_MAX_ROWS)):
        raise ValueError("shape mismatch")
    if k_new is not None:
        _need(k_new, torch.bfloat16, "k_new", 3)
        _need(v_new, torch.bfloat16, "v_new", 3)
        if tuple(k_new.shape) != (B, hkv, d) or tuple(v_new.shape) != (B, hkv, d):
            raise ValueError("shape mismatch")
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dev = _one_device(q, out=out, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale,
                      v_scale=v_scale, block_tables=block_tables, seq_lens=seq_lens, chunk_of=chunk_of,
                      chunk_members=chunk_members, chunk_blocks=chunk_blocks, workspace=workspace)
    _call(dev, "pa_decode_step_shared", lib.pa_decode_step_shared, _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new),
          _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens),
          _ptr(chunk_of), _ptr(chunk_members) if n_chunks else None, _ptr(chunk_blocks) if n_chunks else None,
          n_chunks, int(max_chunk_blocks), B, hq, hkv, d, bs, M, nb, float(scale), int(num_splits), _ptr(workspace),
          ws, kvd, stream=stream)


PA_STATIC_WORKSPACE_BYTES = 16 << 20


def pa_decode_attention_static_ws(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                  v_cache: torch.Tensor, k_scale: Optional[torch.Tensor],
                                  v_scale: Optional[torch.Tensor], block_tables: torch.Tensor,
                                  seq_lens: torch.Tensor, scale: float, num_splits: int = 0,
                                  stream=None) -> None:
    """pa_decode_attention without a caller workspace, for callers that may not
    allocate device memory (the library's own PA_STATIC_WORKSPACE_BYTES array
    is used; calls sharing it must not overlap on the GPU)."""
    lib = load()
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, hq, d = q.shape
    kvd = _kv_dtype(k_cache, d)
    nb, hkv, bs, dc = k_cache.shape
    M = block_tables.shape[1]
    if dc != _row_len(kvd, d) or tuple(out.shape) != (B, hq, d) or block_tables.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("shape mismatch")
    dev = _one_device(q, out=out, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                      block_tables=block_tables, seq_lens=seq_lens)
    _call(dev, "pa_decode_attention_static_ws", lib.pa_decode_attention_static_ws, _ptr(out), _ptr(q),
          _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens), B, hq,
          hkv, d, bs, M, nb, float(scale), int(num_splits), kvd, stream=stream)


def pa_prefill_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         k_scale: Optional[torch.Tensor], v_scale: Optional[torch.Tensor],
                         block_tables: torch.Tensor, seq_lens: torch.Tensor, q_start: torch.Tensor,
                         max_q_len: int, scale: float, stream=None) -> None:
    """Chunked-prefill / verify attention: sequence b's queries (rows q_start[b] ..
    q_start[b+1]-1 of q) are the last positions of its seq_lens[b] cached tokens."""
    lib = load()
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(q_start, torch.int32, "q_start", 1)
    d = q.shape[2]
    kvd = _kv_dtype(k_cache, d)
    nb, hkv, bs, dc = k_cache.shape
    B, M = block_tables.shape
    if out.shape != q.shape or dc != _row_len(kvd, d) or q_start.shape[0] != B + 1 or seq_lens.shape[0] != B:
        raise ValueError("shape mismatch between q, out, caches, tables, lengths and q_start")
    dev = _one_device(q, out=out, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                      block_tables=block_tables, seq_lens=seq_lens, q_start=q_start)
    _call(dev, "pa_prefill_attention", lib.pa_prefill_attention, _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
          _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens), _ptr(q_start), B, q.shape[1], hkv, d,
          bs, M, nb, int(max_q_len), float(scale), kvd, stream=stream)


def pa_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: Optional[torch.Tensor],
                   v_scale: Optional[torch.Tensor], src: torch.Tensor, dst: torch.Tensor, stream=None,
                   kv_dtype: Optional[int] = None) -> None:
    """Block dst[i] becomes a copy of block src[i] (K and V pages, scales of a
    coded cache).  A uint8 cache is taken as e4m3 codes unless kv_dtype is
    PA_KV_INT4."""
    lib = load()
    kvd = _kv_dtype(k_cache)
    if kv_dtype is not None:
        if kv_dtype == PA_KV_INT4 and kvd != PA_KV_FP8_E4M3:
            raise TypeError("an int4 cache is a uint8 tensor")
        if kv_dtype != PA_KV_INT4 and kv_dtype != kvd:
            raise TypeError("kv_dtype does not match the cache tensor")
        kvd = kv_dtype
    _need(src, torch.int32, "src", 1)
    _need(dst, torch.int32, "dst", 1)
    if src.shape != dst.shape or v_cache.shape != k_cache.shape:
        raise ValueError("src/dst or cache shapes differ")
    nb, hkv, bs, dc = k_cache.shape
    d = 2 * dc if kvd == PA_KV_INT4 else dc
    dev = _one_device(src, dst=dst, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale)
    _call(dev, "pa_copy_blocks", lib.pa_copy_blocks, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
          _ptr(src), _ptr(dst), int(src.shape[0]), nb, hkv, d, bs, kvd, stream=stream)


def pa_get_device_error(clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _check(load().pa_get_device_error(ctypes.byref(v), 1 if clear else 0), "pa_get_device_error")
    return int(v.value)


def pa_selftest_bounded_wait(stream=None) -> None:
    _check(load().pa_selftest_bounded_wait(_stream(stream)), "pa_selftest_bounded_wait")


# ------------------------------------------------------------------ host side
class pa_allocator:
    """Reference-counted KV block pool (lowest free ids first)."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = load()
        self._h = self._lib.pa_allocator_create(int(num_blocks), int(block_size))
        if not self._h:
            raise ValueError("invalid allocator arguments")
        self.num_blocks, self.block_size = num_blocks, block_size

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.pa_allocator_destroy(h)

    @property
    def handle(self):
        return self._h

    def alloc(self, n: int) -> np.ndarray:
        return pa_block_alloc(self, n)

    def free(self, ids) -> None:
        pa_block_free(self, ids)

    def share(self, ids) -> None:
        pa_block_share(self, ids)

    def num_free(self) -> int:
        return int(self._lib.pa_allocator_num_free(self._h))

    def fail_nth_alloc(self, n: int) -> None:
        """Fault injection: the n-th later allocation of at least one block fails with OOM (n <= 0 disarms)."""
        _check(self._lib.pa_allocator_fail_nth_alloc(self._h, int(n)), "pa_allocator_fail_nth_alloc")

    def refcount(self, i: int) -> int:
        return int(self._lib.pa_allocator_refcount(self._h, int(i)))


class pa_prefix_cache:
    """Cache of full KV blocks keyed by their whole token prefix."""

    def __init__(self, a: pa_allocator):
        self._lib = load()
        self._alloc = a            # the cache holds references on a's blocks: keep a alive
        self._h = self._lib.pa_prefix_cache_create(a.handle)
        if not self._h:
            raise ValueError("invalid allocator")

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.pa_prefix_cache_destroy(h)

    @property
    def handle(self):
        return self._h

    def size(self) -> int:
        return int(self._lib.pa_prefix_cache_size(self._h))

    def match(self, tokens, max_out: Optional[int] = None) -> np.ndarray:
        return pa_prefix_match(self, tokens, max_out)

    def insert(self, tokens, blocks) -> None:
        pa_prefix_insert(self, tokens, blocks)

    def evict(self, want: int) -> int:
        return pa_prefix_evict(self, want)


def pa_prefix_match(c: pa_prefix_cache, tokens, max_out: Optional[int] = None) -> np.ndarray:
    """Blocks of the longest cached prefix of tokens; the caller gets a reference on each."""
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    bs = c._alloc.block_size
    cap = len(t) // bs if max_out is None else int(max_out)
    out = np.zeros(max(cap, 1), np.int32)
    n = ctypes.c_int(0)
    _check(load().pa_prefix_match(c.handle, _np_ptr(t) if t.size else None, int(t.size), _np_ptr(out), cap,
                                  ctypes.byref(n)), "pa_prefix_match")
    return out[: n.value]


def pa_prefix_insert(c: pa_prefix_cache, tokens, blocks) -> None:
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    b = np.ascontiguousarray(np.asarray(blocks, dtype=np.int32))
    _check(load().pa_prefix_insert(c.handle, _np_ptr(t) if t.size else None, int(t.size),
                                   _np_ptr(b) if b.size else None, int(b.size)), "pa_prefix_insert")


def pa_prefix_evict(c: pa_prefix_cache, want: int) -> int:
    n = ctypes.c_int(0)
    _check(load().pa_prefix_evict(c.handle, int(want), ctypes.byref(n)), "pa_prefix_evict")
    return int(n.value)


def pa_block_cow(a: pa_allocator, block: int):
    """(block to write, needs_copy) for a block the caller holds a reference on."""
    out = ctypes.c_int32(0)
    nc = ctypes.c_int(0)
    _check(load().pa_block_cow(a.handle, int(block), ctypes.byref(out), ctypes.byref(nc)), "pa_block_cow")
    return int(out.value), bool(nc.value)


def pa_block_alloc(a: pa_allocator, n: int) -> np.ndarray:
    out = np.zeros(max(int(n), 1), dtype=np.int32)
    _check(load().pa_block_alloc(a.handle, int(n), _np_ptr(out)), "pa_block_alloc")
    return out[:n]


def pa_block_free(a: pa_allocator, ids: Sequence[int]) -> None:
    arr = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    _check(load().pa_block_free(a.handle, _np_ptr(arr) if arr.size else None, int(arr.size)),
           "pa_block_free")


def pa_block_share(a: pa_allocator, ids: Sequence[int]) -> None:
    arr = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    _check(load().pa_block_share(a.handle, _np_ptr(arr) if arr.size else None, int(arr.size)),
           "pa_block_share")


def pa_blocks_for_tokens(tokens: int, block_size: int) -> int:
    return int(load().pa_blocks_for_tokens(int(tokens), int(block_size)))


def pa_kv_bytes(layers: int, kv_heads: int, head_dim: int, dtype_bits: int, tokens: int, batch: int) -> int:
    return int(load().pa_kv_bytes(layers, kv_heads, head_dim, dtype_bits, tokens, batch))


def pa_slot_mapping(block_tables: np.ndarray, seq_ids: np.ndarray, positions: np.ndarray,
                    block_size: int) -> np.ndarray:
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    s = np.ascontiguousarray(seq_ids, dtype=np.int32)
    p = np.ascontiguousarray(positions, dtype=np.int32)
    out = np.zeros(max(len(s), 1), dtype=np.int64)
    _check(load().pa_slot_mapping(_np_ptr(t), int(t.shape[1]), _np_ptr(s), _np_ptr(p), int(len(s)),
                                  int(block_size), _np_ptr(out)), "pa_slot_mapping")
    return out[: len(s)]


def pa_step_slots(block_tables: np.ndarray, seq_lens: np.ndarray, block_size: int) -> np.ndarray:
    """Slot of each sequence's new token (position seq_len - 1); -1 where seq_len <= 0."""
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    n = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if t.ndim != 2 or n.shape != (t.shape[0],):
        raise ValueError("block_tables must be [B, M] and seq_lens [B]")
    out = np.zeros(max(len(n), 1), dtype=np.int64)
    _check(load().pa_step_slots(_np_ptr(t), int(t.shape[1]), _np_ptr(n), int(len(n)), int(block_size),
                                _np_ptr(out)), "pa_step_slots")
    return out[: len(n)]


def pa_seq_admit(a: pa_allocator, c: Optional[pa_prefix_cache], tokens: np.ndarray, blocks: np.ndarray):
    """Blocks for a new sequence (cached prefix first, then fresh ones) written
    into the int32 buffer `blocks`; returns (number of blocks, first position
    whose KV the caller must write)."""
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    if blocks.dtype != np.int32 or not blocks.flags["C_CONTIGUOUS"]:
        raise TypeError("blocks must be a contiguous int32 buffer")
    n = ctypes.c_int(0)
    first = ctypes.c_int64(0)
    _check(load().pa_seq_admit(a.handle, c.handle if c is not None else None, _np_ptr(t) if t.size else None,
                               int(t.size), _np_ptr(blocks) if blocks.size else None, int(blocks.size),
                               ctypes.byref(n), ctypes.byref(first)), "pa_seq_admit")
    return int(n.value), int(first.value)


def pa_seq_append_slot(a: pa_allocator, c: Optional[pa_prefix_cache], blocks: np.ndarray, n_blocks: int, pos: int):
    """Reserve position pos of a sequence holding blocks[:n_blocks] (int32 buffer,
    updated in place); returns (slot, new n_blocks, (src, dst) page copy or None)."""
    if blocks.dtype != np.int32 or not blocks.flags["C_CONTIGUOUS"]:
        raise TypeError("blocks must be a contiguous int32 buffer")
    n = ctypes.c_int(int(n_blocks))
    slot = ctypes.c_int64(0)
    src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
    _check(load().pa_seq_append_slot(a.handle, c.handle if c is not None else None,
                                     _np_ptr(blocks) if blocks.size else None, ctypes.byref(n), int(blocks.size),
                                     int(pos), ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst)),
           "pa_seq_append_slot")
    copy = (int(src.value), int(dst.value)) if src.value >= 0 else None
    return int(slot.value), int(n.value), copy


def pa_sched_simulate(out_lens: Sequence[int], slots: int, mode: int) -> int:
    arr = np.ascontiguousarray(np.asarray(out_lens, dtype=np.int64))
    it = ctypes.c_int64(0)
    _check(load().pa_sched_simulate(_np_ptr(arr) if arr.size else None, int(arr.size), int(slots),
                                    int(mode), ctypes.byref(it)), "pa_sched_simulate")
    return int(it.value)


def pa_sched_continuous_kv(a: pa_allocator, prompt_lens, out_lens, max_num_seqs: int,
                           stop_iter: int = -1, max_blocks_per_seq: int = 0):
    """Returns dict(iters, admitted_at, finished_at, tables, lens)."""
    p = np.ascontiguousarray(np.asarray(prompt_lens, dtype=np.int64))
    o = np.ascontiguousarray(np.asarray(out_lens, dtype=np.int64))
    n = len(p)
    it = ctypes.c_int64(0)
    adm = np.zeros(max(n, 1), np.int64)
    fin = np.zeros(max(n, 1), np.int64)
    tables = np.zeros((max(n, 1), max(max_blocks_per_seq, 1)), np.int32)
    lens = np.zeros(max(n, 1), np.int32)
    _check(load().pa_sched_continuous_kv(a.handle, _np_ptr(p) if n else None, _np_ptr(o) if n else None,
                                         n, int(max_num_seqs), int(stop_iter), int(max_blocks_per_seq),
                                         ctypes.byref(it), _np_ptr(adm), _np_ptr(fin),
                                         _np_ptr(tables) if max_blocks_per_seq > 0 else None,
                                         _np_ptr(lens)),
           "pa_sched_continuous_kv")
    return dict(iters=int(it.value), admitted_at=adm[:n], finished_at=fin[:n],
                tables=tables[:n, :max_blocks_per_seq], lens=lens[:n])
