"""Pins for the oracle's int8 cache codec and append.

"LLM Inference Optimization", section "Memory Bandwidth Optimization": KV
cache quantization to INT8 halves the cache reads.  The rule (a reading; the
pages give none): one fp32 scale per (block, kv_head), s = absmax / 127, code =
clamp(round-half-even(x / s), -127, 127), value = code * s, with the same
growth / restart rule as the fp8 cache.  Everything here is checked against
numpy's own rint / clip on float32 quotients and torch attention on the
dequantized values, not against the oracle's C code.
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
    """numpy's rounding of fp32 quotients to int8 codes (two's-complement bytes)."""
    return np.clip(np.rint(q_f32.astype(np.float64)), -127, 127).astype(np.int8).view(np.uint8)


def test_codec_rounds_half_to_even_and_clamps():
    for x, c in [(0.5, 0), (1.5, 2), (2.5, 2), (-2.5, -2), (-3.5, -4), (126.5, 126), (127.4, 127),
                 (128.0, 127), (1e9, 127), (-1e9, -127), (-127.6, -127), (0.0, 0), (-0.4, 0)]:
        assert oracle.int8_encode(x) == (c & 0xFF), x
    for c in range(-127, 128):
        assert oracle.int8_value(c & 0xFF) == c
        assert oracle.int8_encode(float(c)) == (c & 0xFF)
    assert oracle.int8_encode(float("nan")) == 0


def test_fresh_block_scale_and_codes_match_numpy():
    rng = np.random.default_rng(0)
    bs, d, Hkv = 8, 16, 2
    cache = oracle.Cache(4, Hkv, d, bs, kv="int8")
    k = _bf16(rng.standard_normal((5, Hkv, d)) * 3)
    v = _bf16(rng.standard_normal((5, Hkv, d)))
    cache.append(k, v, np.array([16, 17, 18, 19, 20], np.int64))
    for h in range(Hkv):
        a = np.float32(np.max(np.abs(_f32(k)[:, h])))
        s = np.float32(a / np.float32(127.0))
        assert cache.k_scale[2, h] == s
        assert np.array_equal(cache.k[2, h, :5], _codes(_f32(k)[:, h] / s))
        # round trip within half a step, and the absmax lands on +-127
        deq = cache.k[2, h, :5].view(np.int8).astype(np.float64) * s
        assert np.all(np.abs(deq - _f32(k)[:, h]) <= 0.5 * s * (1 + 1e-6))
        assert np.max(np.abs(cache.k[2, h, :5].view(np.int8).astype(np.int32))) == 127
    assert np.all(cache.k[[0, 1, 3]] == 0) and np.all(cache.k_scale[[0, 1, 3]] == 0)


def test_growth_reencodes_older_codes():
    rng = np.random.default_rng(1)
    cache = oracle.Cache(2, 1, 16, 8, kv="int8")
    first = _bf16(rng.standard_normal((3, 1, 16)))
    cache.append(first, first, np.array([8, 9, 10], np.int64))
    s_old, codes_old = cache.k_scale[1, 0], cache.k[1, 0, :3].copy()
    big = _bf16(rng.standard_normal((1, 1, 16)) * 10)
    cache.append(big, big, np.array([11], np.int64))
    s_new = cache.k_scale[1, 0]
    a = max(np.max(np.abs(_f32(first))), np.max(np.abs(_f32(big))))
    assert s_new == np.float32(np.float32(a) / np.float32(127.0)) and s_new > s_old
    prod = (codes_old.view(np.int8).astype(np.float32) * np.float32(s_old)).astype(np.float32)
    assert np.array_equal(cache.k[1, 0, :3], _codes((prod / np.float32(s_new)).astype(np.float32)))
    assert np.array_equal(cache.k[1, 0, 3], _codes((_f32(big)[0, 0] / s_new).astype(np.float32)))


def test_no_growth_restart_and_zero_blocks():
    rng = np.random.default_rng(2)
    cache = oracle.Cache(1, 1, 8, 4, kv="int8")
    x = _bf16(rng.standard_normal((2, 1, 8)) * 4)
    cache.append(x, x, np.array([0, 1], np.int64))
    codes, s = cache.k[0, 0, :2].copy(), cache.k_scale[0, 0]
    small = _bf16(rng.standard_normal((1, 1, 8)) * 0.01)
    cache.append(small, small, np.array([2], np.int64))
    assert cache.k_scale[0, 0] == s and np.array_equal(cache.k[0, 0, :2], codes)
    cache.append(small, small, np.array([0], np.int64))           # offset 0 restarts the block
    assert cache.k_scale[0, 0] == np.float32(np.float32(np.max(np.abs(_f32(small)))) / np.float32(127))
    z = oracle.Cache(1, 1, 8, 4, kv="int8")
    zero = _bf16(np.zeros((2, 1, 8)))
    z.append(zero, zero, np.array([0, 1], np.int64))
    assert z.k_scale[0, 0] == 0 and np.all(z.k == 0)


@pytest.mark.parametrize("G", [1, 4])
def test_int8_attention_matches_torch_on_dequantized_values(G):
    rng = np.random.default_rng(4 + G)
    bs, d, Hkv, L = 8, 32, 2, 29
    Hq = Hkv * G
    cache = oracle.Cache(6, Hkv, d, bs, kv="int8")
    tables = np.array([[4, 1, 5, 0]], np.int32)
    k = _bf16(rng.standard_normal((L, Hkv, d)))
    v = _bf16(rng.standard_normal((L, Hkv, d)))
    slots = tables[0, np.arange(L) // bs].astype(np.int64) * bs + np.arange(L) % bs
    cache.append(k, v, slots)
    q = _bf16(rng.standard_normal((1, Hq, d)))
    out = oracle.decode_attention(cache, q, tables, np.array([L], np.int32), Hq, 0.25)
    blk, off = tables[0, np.arange(L) // bs], np.arange(L) % bs
    Kd = torch.from_numpy(cache.k[blk, :, off].view(np.int8).astype(np.float64)
                          * cache.k_scale[blk][:, :, None].astype(np.float64))
    Vd = torch.from_numpy(cache.v[blk, :, off].view(np.int8).astype(np.float64)
                          * cache.v_scale[blk][:, :, None].astype(np.float64))
    qd = q.double()[0]                                              # [Hq, d]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qd[:, None, :], Kd.permute(1, 0, 2).repeat_interleave(G, 0), Vd.permute(1, 0, 2).repeat_interleave(G, 0),
        scale=0.25)[:, 0, :]
    assert np.max(np.abs(out[0] - ref.numpy())) <= 1e-12
    # the prefill form on the same cache agrees with the library too
    q2 = _bf16(rng.standard_normal((3, Hq, d)))
    got = oracle.prefill_attention(cache, q2, tables, np.array([L]), np.array([0, 3]), Hq, 0.25)
    mask = torch.arange(L)[None, :] <= torch.arange(L - 3, L)[:, None]
    ref2 = torch.nn.functional.scaled_dot_product_attention(
        q2.double().permute(1, 0, 2), Kd.permute(1, 0, 2).repeat_interleave(G, 0),
        Vd.permute(1, 0, 2).repeat_interleave(G, 0), attn_mask=mask, scale=0.25).permute(1, 0, 2)
    assert np.max(np.abs(got - ref2.numpy())) <= 1e-12
