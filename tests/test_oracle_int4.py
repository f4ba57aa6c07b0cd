"""Pins for the oracle's int4 cache codec, nibble packing and append.

"KV cache & continuous batching", section "KV cache memory math": int4 holds
half a byte per element.  The rule (a reading; the pages give only the size):
one fp32 scale per (block, kv_head), s = absmax / 7, code =
clamp(round-half-even(x / s), -7, 7), value = code * s, with the growth /
restart rule of the other coded caches; element 2j of a row sits in the low
nibble of the row's byte j, element 2j+1 in the high nibble, as 4-bit two's
complement.  Everything here is checked against numpy's own rint / clip on
float32 quotients, a nibble unpacker written below from that definition,
hand-packed bytes and torch attention on the unpacked values, not against
the oracle's C code.
"""
import numpy as np
import pytest
import torch

import oracle


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def _f32(t):
    return t.to(torch.float32).numpy()


def _codes(q_f32):
    """numpy's rounding of fp32 quotients to int4 code values (int8 array in [-7, 7])."""
    return np.clip(np.rint(q_f32.astype(np.float64)), -7, 7).astype(np.int8)


def _unpack(rows):
    """[..., d/2] packed bytes -> [..., d] signed code values."""
    rows = np.asarray(rows, np.uint8)
    lo = (rows & 0xF).astype(np.int8)
    hi = (rows >> 4).astype(np.int8)
    out = np.empty(rows.shape[:-1] + (2 * rows.shape[-1],), np.int8)
    out[..., 0::2] = np.where(lo >= 8, lo - 16, lo)
    out[..., 1::2] = np.where(hi >= 8, hi - 16, hi)
    return out


def test_codec_rounds_half_to_even_and_clamps():
    for x, c in [(0.5, 0), (1.5, 2), (2.5, 2), (-2.5, -2), (-3.5, -4), (6.5, 6), (7.4, 7), (8.0, 7),
                 (1e9, 7), (-1e9, -7), (-7.6, -7), (0.0, 0), (-0.4, 0)]:
        assert oracle.int4_encode(x) == (c & 0xF), x
    for c in range(-7, 8):
        assert oracle.int4_value(c & 0xF) == c
        assert oracle.int4_encode(float(c)) == (c & 0xF)
    assert oracle.int4_value(8) == -8          # the nibble exists but encoding never makes it
    assert oracle.int4_encode(float("nan")) == 0


def test_nibble_order_against_hand_packed_bytes():
    # absmax 7 gives s = 1 exactly, so each value is its own code
    vals = np.array([7, -3, 0, 1, -7, 2, 5, -1], np.float32)
    cache = oracle.Cache(1, 1, 8, 4, kv="int4")
    x = _bf16(vals.reshape(1, 1, 8))
    cache.append(x, x, np.array([2], np.int64))
    assert cache.k_scale[0, 0] == 1.0
    # byte j = low nibble element 2j | high nibble element 2j+1
    want = [0x07 | (0xD << 4), 0x0 | (0x1 << 4), 0x9 | (0x2 << 4), 0x5 | (0xF << 4)]
    assert list(cache.k[0, 0, 2]) == want
    assert np.all(cache.k[0, 0, [0, 1, 3]] == 0)


def test_fresh_block_scale_and_codes_match_numpy():
    rng = np.random.default_rng(0)
    bs, d, Hkv = 8, 16, 2
    cache = oracle.Cache(4, Hkv, d, bs, kv="int4")
    assert cache.k.shape == (4, Hkv, bs, d // 2)
    k = _bf16(rng.standard_normal((5, Hkv, d)) * 3)
    v = _bf16(rng.standard_normal((5, Hkv, d)))
    cache.append(k, v, np.array([16, 17, 18, 19, 20], np.int64))
    for h in range(Hkv):
        for name, x, c, sc in (("k", k, cache.k, cache.k_scale), ("v", v, cache.v, cache.v_scale)):
            a = np.float32(np.max(np.abs(_f32(x)[:, h])))
            s = np.float32(a / np.float32(7.0))
            assert sc[2, h] == s, name
            assert np.array_equal(_unpack(c[2, h, :5]), _codes(_f32(x)[:, h] / s)), name
            deq = _unpack(c[2, h, :5]).astype(np.float64) * s
            assert np.all(np.abs(deq - _f32(x)[:, h]) <= 0.5 * s * (1 + 1e-6)), name
            assert np.max(np.abs(_unpack(c[2, h, :5]).astype(np.int32))) == 7, name
    assert np.all(cache.k[[0, 1, 3]] == 0) and np.all(cache.k_scale[[0, 1, 3]] == 0)


def test_growth_reencodes_older_codes():
    rng = np.random.default_rng(1)
    cache = oracle.Cache(2, 1, 16, 8, kv="int4")
    first = _bf16(rng.standard_normal((3, 1, 16)))
    cache.append(first, first, np.array([8, 9, 10], np.int64))
    s_old, codes_old = cache.k_scale[1, 0], _unpack(cache.k[1, 0, :3])
    big = _bf16(rng.standard_normal((1, 1, 16)) * 10)
    cache.append(big, big, np.array([11], np.int64))
    s_new = cache.k_scale[1, 0]
    a = max(np.max(np.abs(_f32(first))), np.max(np.abs(_f32(big))))
    assert s_new == np.float32(np.float32(a) / np.float32(7.0)) and s_new > s_old
    prod = (codes_old.astype(np.float32) * np.float32(s_old)).astype(np.float32)
    assert np.array_equal(_unpack(cache.k[1, 0, :3]), _codes((prod / np.float32(s_new)).astype(np.float32)))
    assert np.array_equal(_unpack(cache.k[1, 0, 3]), _codes((_f32(big)[0, 0] / s_new).astype(np.float32)))


def test_no_growth_keeps_neighbour_rows_restart_and_zero_blocks():
    rng = np.random.default_rng(2)
    cache = oracle.Cache(1, 1, 8, 4, kv="int4")
    x = _bf16(rng.standard_normal((2, 1, 8)) * 4)
    cache.append(x, x, np.array([0, 1], np.int64))
    rows, s = cache.k[0, 0, :2].copy(), cache.k_scale[0, 0]
    small = _bf16(rng.standard_normal((1, 1, 8)) * 0.01)
    cache.append(small, small, np.array([2], np.int64))
    assert cache.k_scale[0, 0] == s and np.array_equal(cache.k[0, 0, :2], rows)
    assert np.array_equal(_unpack(cache.k[0, 0, 2]), _codes(_f32(small)[0, 0] / s))
    cache.append(small, small, np.array([0], np.int64))           # offset 0 restarts the block
    assert cache.k_scale[0, 0] == np.float32(np.float32(np.max(np.abs(_f32(small)))) / np.float32(7))
    z = oracle.Cache(1, 1, 8, 4, kv="int4")
    zero = _bf16(np.zeros((2, 1, 8)))
    z.append(zero, zero, np.array([0, 1], np.int64))
    assert z.k_scale[0, 0] == 0 and np.all(z.k == 0)


@pytest.mark.parametrize("G", [1, 4])
def test_int4_attention_matches_torch_on_unpacked_values(G):
    rng = np.random.default_rng(4 + G)
    bs, d, Hkv, L = 8, 32, 2, 29
    Hq = Hkv * G
    cache = oracle.Cache(6, Hkv, d, bs, kv="int4")
    tables = np.array([[4, 1, 5, 0]], np.int32)
    k = _bf16(rng.standard_normal((L, Hkv, d)))
    v = _bf16(rng.standard_normal((L, Hkv, d)))
    slots = tables[0, np.arange(L) // bs].astype(np.int64) * bs + np.arange(L) % bs
    cache.append(k, v, slots)
    q = _bf16(rng.standard_normal((1, Hq, d)))
    out = oracle.decode_attention(cache, q, tables, np.array([L], np.int32), Hq, 0.25)
    blk, off = tables[0, np.arange(L) // bs], np.arange(L) % bs
    Kd = torch.from_numpy(_unpack(cache.k[blk, :, off]).astype(np.float64)
                          * cache.k_scale[blk][:, :, None].astype(np.float64))
    Vd = torch.from_numpy(_unpack(cache.v[blk, :, off]).astype(np.float64)
                          * cache.v_scale[blk][:, :, None].astype(np.float64))
    qd = q.double()[0]                                              # [Hq, d]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qd[:, None, :], Kd.permute(1, 0, 2).repeat_interleave(G, 0), Vd.permute(1, 0, 2).repeat_interleave(G, 0),
        scale=0.25)[:, 0, :]
    assert np.max(np.abs(out[0] - ref.numpy())) <= 1e-12
    # split-K form and the prefill form on the same cache agree too
    split = oracle.decode_attention(cache, q, tables, np.array([L], np.int32), Hq, 0.25, part_blocks=1)
    assert np.max(np.abs(split - out)) <= 1e-12
    q2 = _bf16(rng.standard_normal((3, Hq, d)))
    got = oracle.prefill_attention(cache, q2, tables, np.array([L]), np.array([0, 3]), Hq, 0.25)
    mask = torch.arange(L)[None, :] <= torch.arange(L - 3, L)[:, None]
    ref2 = torch.nn.functional.scaled_dot_product_attention(
        q2.double().permute(1, 0, 2), Kd.permute(1, 0, 2).repeat_interleave(G, 0),
        Vd.permute(1, 0, 2).repeat_interleave(G, 0), attn_mask=mask, scale=0.25).permute(1, 0, 2)
    assert np.max(np.abs(got - ref2.numpy())) <= 1e-12
