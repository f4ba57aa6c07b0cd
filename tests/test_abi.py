"""The C-ABI library builds, loads without a GPU and exports every declared symbol."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_cache_294_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ("pa_kv_append", "pa_decode_attention", "pa_block_alloc", "pa_block_free",
                 "pa_decode_workspace_bytes", "pa_sched_simulate"):
        assert must in names
    assert len(names) >= 19


def test_library_loads_and_exports_every_declared_symbol():
    lib = pa.load()
    path = pa.library_path()
    assert os.path.exists(path)
    raw = ctypes.CDLL(path)
    for name in declared_symbols():
        assert hasattr(raw, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pa_[a-z0-9_]+)\b", nm))
    assert set(declared_symbols()) <= exported
    assert lib.pa_status_string(0) == b"PA_OK"


def test_library_is_built_for_sm_103a():
    out = subprocess.run(["cuobjdump", "--list-elf", pa.library_path()], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


def test_argument_errors_return_status_without_a_gpu():
    lib = pa.load()
    # Hq not a multiple of Hkv, bad dtype, bad block size: rejected on the host before any launch
    assert lib.pa_decode_attention(None, None, None, None, None, None, None, None, 1, 6, 4, 128, 16,
                                   4, 64, 1.0, 0, None, 0, 0, None) == pa.PA_ERR_INVALID
    assert lib.pa_decode_attention(None, None, None, None, None, None, None, None, 1, 8, 4, 128, 16,
                                   4, 64, 1.0, 0, None, 0, 7, None) == pa.PA_ERR_INVALID
    assert lib.pa_decode_attention(None, None, None, None, None, None, None, None, 1, 8, 4, 128, 8,
                                   4, 64, 1.0, 0, None, 0, 0, None) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_decode_attention(None, None, None, None, None, None, None, None, 1, 8, 4, 64, 16,
                                   4, 64, 1.0, 0, None, 0, 1, None) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_decode_attention(None, None, None, None, None, None, None, None, 1, 64, 4, 128, 16,
                                   4, 64, 1.0, 0, None, 0, 0, None) == pa.PA_ERR_UNSUPPORTED
    # int8 (kv_dtype 2) and int4 (3) caches: head_dim 64 unsupported; kv_dtype 4 rejected
    for kvd in (2, 3):
        assert lib.pa_decode_attention(None, None, None, None, None, None, None, None, 1, 8, 4, 64, 16,
                                       4, 64, 1.0, 0, None, 0, kvd, None) == pa.PA_ERR_UNSUPPORTED
        assert lib.pa_kv_append(None, None, None, None, None, None, None, 1, 64, 4, 64, 16, kvd,
                                None) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_decode_attention(None, None, None, None, None, None, None, None, 1, 8, 4, 128, 16,
                                   4, 64, 1.0, 0, None, 0, 4, None) == pa.PA_ERR_INVALID
    # the multi-query entry point: every cache type at head_dim 128 (coded ones
    # need their scales), head_dim 64 unsupported
    for kvd in (0, 1, 2, 3):
        assert lib.pa_prefill_attention(None, None, None, None, None, None, None, None, None, 1, 8, 4, 64, 16,
                                         4, 64, 8, 1.0, kvd, None) == pa.PA_ERR_UNSUPPORTED
        assert lib.pa_prefill_attention(None, None, None, None, None, None, None, None, None, 1, 8, 4, 128, 16,
                                         4, 64, 8, 1.0, kvd, None) == pa.PA_ERR_INVALID
    # null pointers with a non-empty batch
    assert lib.pa_decode_attention(None, None, None, None, None, None, None, None, 1, 8, 4, 128, 16,
                                   4, 64, 1.0, 0, None, 0, 0, None) == pa.PA_ERR_INVALID
    # pool too large for 32-bit TMA rows
    assert lib.pa_kv_append(None, None, None, None, None, None, None, 1, 1 << 27, 8, 128, 16, 0,
                            None) == pa.PA_ERR_INVALID
    # more than 2^31 - 1 work items (S x kv-head sets x batch): rejected before any pointer is read
    S = pa.pa_decode_resolve_splits(1 << 26, 8, 64, 8)
    assert S == 8 and S * 4 * (1 << 26) > 2 ** 31 - 1
    assert lib.pa_decode_attention(None, None, None, None, None, None, None, None, 1 << 26, 32, 8, 128, 16,
                                   64, 64, 1.0, 8, None, 0, 0, None) == pa.PA_ERR_UNSUPPORTED
    # empty work is a no-op
    assert lib.pa_kv_append(None, None, None, None, None, None, None, 0, 64, 2, 64, 16, 0, None) == pa.PA_OK
    assert lib.pa_decode_attention(None, None, None, None, None, None, None, None, 0, 8, 4, 128, 16,
                                   4, 64, 1.0, 0, None, 0, 0, None) == pa.PA_OK


def test_split_planning():
    # explicit split counts: P = ceil(M/S) blocks per partition, S_eff = ceil(M/P)
    assert pa.pa_decode_resolve_splits(4, 8, 8192, 64) == 64
    assert pa.pa_decode_resolve_splits(4, 8, 7, 5) == 4
    assert pa.pa_decode_resolve_splits(4, 8, 7, 100) == 7
    assert pa.pa_decode_resolve_splits(4, 8, 7, 1) == 1
    up = lambda x: -(-x // 256) * 256
    assert pa.pa_decode_workspace_bytes(4, 32, 8, 128, 8192, 1) == up(4 * 8 * 4)
    ws = pa.pa_decode_workspace_bytes(4, 32, 8, 128, 8192, 64)
    assert ws == up(4 * 32 * 64 * 128 * 4) + up(4 * 32 * 64 * 4) + up(4 * 8 * 4)
    assert pa.pa_decode_resolve_splits(4, 8, 8192, 4096) == 512      # at most 512 partitions
    # automatic choice: a CTA streams 32 .. 256 pages; it covers two kv heads
    # when their count is even, so its partition is half as many blocks
    for B, Hkv, M in [(64, 8, 256), (256, 8, 512), (128, 32, 256), (4, 2, 7), (64, 3, 256), (300, 1, 512)]:
        S = pa.pa_decode_resolve_splits(B, Hkv, M, 0)
        P = -(-M // S)
        hpc = 2 if Hkv % 2 == 0 else 1
        assert 1 <= S <= M
        assert P == M or P * hpc >= 32
        assert P * hpc <= 256 + hpc - 1
    # few (sequence, head set) groups with long tables: one wave of long
    # partitions (the device's SM count decides the exact number; without a
    # device the library plans for a GB300's 152 SMs)
    S = pa.pa_decode_resolve_splits(4, 8, 8192, 0)
    assert 4 * 4 * S <= 3 * 152 and S >= 16 and -(-8192 // S) * 2 >= 256
