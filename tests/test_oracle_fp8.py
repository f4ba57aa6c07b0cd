"""Pins for the oracle's E4M3 codec and fp8 append.

The codec is checked against two things outside the oracle: torch's own
float8_e4m3fn conversion (an independent implementation of the OCP E4M3
format) and a nearest-value brute force over the 256-code table.  The fp8
append's scale rule (per (block, kv_head) absmax / 448, "KV cache & continuous
batching", section "KV cache memory math": 1 byte per fp8 element) is checked
through invariants that hold for any correct implementation: the scale equals
the block's absmax / 448, every value round-trips within the format's
rounding bound, and older entries are rescaled only when the scale grows.
"""
import numpy as np
import pytest
import torch

import oracle


def torch_e4m3_value(code: int) -> float:
    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64))


def torch_e4m3_encode(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_all_256_codes_match_torch():
    for c in range(256):
        a, b = oracle.e4m3_value(c), torch_e4m3_value(c)
        if np.isnan(b):
            assert np.isnan(a), c
        else:
            assert a == b, (c, a, b)


def test_format_facts():
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0xFE) == -448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x38) == 1.0
    assert np.isnan(oracle.e4m3_value(0x7F)) and np.isnan(oracle.e4m3_value(0xFF))
    pos = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))            # strictly increasing
    assert str(oracle.e4m3_value(0x80)) == "-0.0"


def _table():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    vals = np.array([torch_e4m3_value(c) for c in codes])
    return codes, vals


def brute_encode(x: float, codes, vals) -> int:
    """Nearest finite code; ties to the code with even mantissa; saturate at 448."""
    if x >= 448:
        return 0x7E
    if x <= -448:
        return 0xFE
    dist = np.abs(vals - x)
    best = np.flatnonzero(dist == dist.min())
    cands = codes[best]
    if len(cands) > 1:
        cands = [c for c in cands if (c & 1) == 0] or list(cands)
        # +0 / -0 tie: keep the sign of x
        if len(cands) > 1:
            cands = [c for c in cands if (c >> 7) == (1 if np.signbit(x) else 0)]
    return int(cands[0])


def test_encode_roundtrips_every_finite_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c


def test_encode_midpoints_round_to_even_and_match_torch():
    codes, vals = _table()
    pos = sorted(set(v for v in vals if v >= 0))
    mids = [(a + b) / 2 for a, b in zip(pos, pos[1:])]
    xs = np.array(mids + [-m for m in mids], dtype=np.float32)
    # every midpoint is exact in fp32
    assert np.all(xs.astype(np.float64) == np.array(mids + [-m for m in mids]))
    ours = oracle.e4m3_encode_array(xs)
    assert np.array_equal(ours, torch_e4m3_encode(xs))
    for x, c in zip(xs, ours):
        assert c == brute_encode(float(x), codes, vals)
        assert (c & 1) == 0


def test_encode_random_sample_matches_torch_and_bruteforce():
    rng = np.random.default_rng(2024)
    codes, vals = _table()
    # stratified: random fp32 bit patterns over exponents covering subnormal..saturation
    e = rng.integers(127 - 14, 127 + 9, size=6000)
    m = rng.integers(0, 1 << 23, size=6000)
    s = rng.integers(0, 2, size=6000)
    bits = (s.astype(np.uint32) << 31) | (e.astype(np.uint32) << 23) | m.astype(np.uint32)
    xs = bits.view(np.float32)
    xs = xs[np.abs(xs) < 448]
    ours = oracle.e4m3_encode_array(xs)
    assert np.array_equal(ours, torch_e4m3_encode(xs))
    for x, c in list(zip(xs, ours))[:1500]:
        assert c == brute_encode(float(x), codes, vals)


def test_encode_saturates():
    for x, c in [(448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (np.inf, 0x7E),
                 (-500.0, 0xFE), (-np.inf, 0xFE)]:
        assert oracle.e4m3_encode(x) == c
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-30) == 0x80


# ------------------------------------------------------------ fp8 append


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def _f32(t):
    return t.to(torch.float32).numpy()


def _dequant(cache, blk, h):
    vals = np.vectorize(oracle.e4m3_value)
    return vals(cache.k[blk, h]) * np.float64(cache.k_scale[blk, h])


def _bound(x, s):
    """E4M3 rounding bound of x / s, scaled back: half a spacing (2^-4 relative, 2^-10 abs)."""
    return np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6)


def test_fresh_block_scale_is_absmax_over_448():
    rng = np.random.default_rng(0)
    bs, d, Hkv = 8, 16, 2
    cache = oracle.Cache(4, Hkv, d, bs, kv="fp8")
    k = _bf16(rng.standard_normal((5, Hkv, d)) * 3)
    v = _bf16(rng.standard_normal((5, Hkv, d)))
    cache.append(k, v, np.array([16, 17, 18, 19, 20], np.int64))    # block 2, offsets 0..4
    for h in range(Hkv):
        a = np.float32(np.max(np.abs(_f32(k)[:, h])))
        assert cache.k_scale[2, h] == np.float32(a / np.float32(448.0))
        deq = _dequant(cache, 2, h)[:5]
        assert np.all(np.abs(deq - _f32(k)[:, h]) <= _bound(_f32(k)[:, h], cache.k_scale[2, h]))
        # the absmax element lands on (or rounds to) the top code
        assert np.max(np.abs(cache.k[2, h, :5].astype(np.int32) & 0x7F)) >= 0x7D
    assert np.all(cache.k[[0, 1, 3]] == 0) and np.all(cache.k_scale[[0, 1, 3]] == 0)
    # codes are torch's e4m3 rounding of x / s
    s = cache.k_scale[2, 0]
    want = torch_e4m3_encode((_f32(k)[:, 0] / s).astype(np.float32))
    assert np.array_equal(cache.k[2, 0, :5], want)


def test_growth_rescales_older_entries_and_keeps_them_close():
    rng = np.random.default_rng(1)
    bs, d = 8, 16
    cache = oracle.Cache(2, 1, d, bs, kv="fp8")
    first = _bf16(rng.standard_normal((3, 1, d)))
    cache.append(first, first, np.array([8, 9, 10], np.int64))
    s_old = cache.k_scale[1, 0]
    codes_old = cache.k[1, 0, :3].copy()
    big = _bf16(rng.standard_normal((1, 1, d)) * 10)
    cache.append(big, big, np.array([11], np.int64))
    s_new = cache.k_scale[1, 0]
    assert s_new > s_old
    a = max(np.max(np.abs(_f32(first))), np.max(np.abs(_f32(big))))
    assert s_new == np.float32(np.float32(a) / np.float32(448.0))
    # older entries: re-encoded value(e_old) * s_old / s_new (one extra rounding)
    deq = _dequant(cache, 1, 0)
    x_old = _f32(first)[:, 0]
    assert np.all(np.abs(deq[:3] - x_old) <= 2 * _bound(x_old, s_new))
    want = torch_e4m3_encode(
        (np.vectorize(oracle.e4m3_value)(codes_old).astype(np.float32) * np.float32(s_old)).astype(np.float32)
        / np.float32(s_new))
    assert np.array_equal(cache.k[1, 0, :3], want)
    assert np.all(np.abs(deq[3] - _f32(big)[0, 0]) <= _bound(_f32(big)[0, 0], s_new))


def test_no_growth_keeps_codes_and_scale():
    rng = np.random.default_rng(2)
    cache = oracle.Cache(1, 1, 8, 4, kv="fp8")
    x = _bf16(rng.standard_normal((2, 1, 8)) * 4)
    cache.append(x, x, np.array([0, 1], np.int64))
    codes, s = cache.k[0, 0, :2].copy(), cache.k_scale[0, 0]
    small = _bf16(rng.standard_normal((1, 1, 8)) * 0.01)
    cache.append(small, small, np.array([2], np.int64))
    assert cache.k_scale[0, 0] == s
    assert np.array_equal(cache.k[0, 0, :2], codes)


def test_offset_zero_restarts_the_block():
    rng = np.random.default_rng(3)
    cache = oracle.Cache(1, 1, 8, 4, kv="fp8")
    big = _bf16(rng.standard_normal((4, 1, 8)) * 50)
    cache.append(big, big, np.arange(4, dtype=np.int64))
    small = _bf16(rng.standard_normal((1, 1, 8)))
    cache.append(small, small, np.array([0], np.int64))
    assert cache.k_scale[0, 0] == np.float32(np.float32(np.max(np.abs(_f32(small)))) / np.float32(448))


def test_all_zero_block_has_zero_scale_and_zero_codes():
    cache = oracle.Cache(1, 1, 8, 4, kv="fp8")
    z = _bf16(np.zeros((2, 1, 8)))
    cache.append(z, z, np.array([0, 1], np.int64))
    assert cache.k_scale[0, 0] == 0 and np.all(cache.k == 0)


def test_fp8_decode_matches_dense_on_dequantized_values():
    """The fp8 attention definition: element value = value(code) * scale, then plain attention."""
    rng = np.random.default_rng(4)
    bs, d, Hkv, Hq, L = 8, 16, 2, 4, 29
    cache = oracle.Cache(6, Hkv, d, bs, kv="fp8")
    tables = np.array([[4, 1, 5, 0]], np.int32)
    k = _bf16(rng.standard_normal((L, Hkv, d)))
    v = _bf16(rng.standard_normal((L, Hkv, d)))
    slots = oracle.slot_mapping(tables, np.zeros(L, np.int32), np.arange(L, dtype=np.int32), bs)
    cache.append(k, v, slots)
    q = _bf16(rng.standard_normal((1, Hq, d)))
    out = oracle.decode_attention(cache, q, tables, np.array([L], np.int32), Hq, 0.25)
    dv = np.vectorize(oracle.e4m3_value)
    Kd = np.zeros((L, Hkv, d))
    Vd = np.zeros((L, Hkv, d))
    for t in range(L):
        blk, off = tables[0, t // bs], t % bs
        Kd[t] = dv(cache.k[blk, :, off]) * cache.k_scale[blk][:, None].astype(np.float64)
        Vd[t] = dv(cache.v[blk, :, off]) * cache.v_scale[blk][:, None].astype(np.float64)
    qd = q.to(torch.float64).numpy()
    for i in range(Hq):
        s = Kd[:, i // 2] @ qd[0, i] * 0.25
        w = np.exp(s - s.max())
        assert np.max(np.abs(out[0, i] - (w / w.sum()) @ Vd[:, i // 2])) <= 1e-12
