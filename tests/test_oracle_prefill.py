"""Pins for the oracle's multi-query (chunked-prefill / verify) attention.

The general case is checked against a library routine: torch's
scaled_dot_product_attention in float64 on the K/V gathered through the block
table, with the causal chunk mask written out.  fp8 codes are decoded with
torch's float8_e4m3fn type.  One-token chunks must equal the (separately
pinned) decode attention, and a verify chunk of K+1 tokens must equal K+1
sequential decode steps.
"""
import numpy as np
import pytest
import torch

import oracle


def _cache(kv, B, Hkv, d, bs, lens, seed):
    rng = np.random.default_rng(seed)
    M = max(-(-int(n) // bs) for n in lens) + 1
    nb = B * M + 3
    perm = rng.permutation(nb)
    tables = np.full((B, M), -1, dtype=np.int32)
    c = oracle.Cache(nb, Hkv, d, bs, kv)
    pos = 0
    for b, n in enumerate(lens):
        k = -(-int(n) // bs)
        tables[b, :k] = perm[pos:pos + k]
        pos += k
        if n:
            slots = tables[b, np.arange(n) // bs].astype(np.int64) * bs + np.arange(n) % bs
            kk = torch.randn(int(n), Hkv, d, dtype=torch.float64, generator=torch.Generator().manual_seed(seed + b))
            vv = torch.randn(int(n), Hkv, d, dtype=torch.float64, generator=torch.Generator().manual_seed(seed + 99 + b))
            c.append(kk.to(torch.bfloat16), vv.to(torch.bfloat16), slots)
    return c, tables


def _gather(c, table, n, h):
    blk = table[np.arange(n) // c.bs]
    off = np.arange(n) % c.bs
    k, v = c.k[blk, h, off], c.v[blk, h, off]
    if c.kv == "fp8":
        kt = torch.from_numpy(np.ascontiguousarray(k)).view(torch.float8_e4m3fn).double()
        vt = torch.from_numpy(np.ascontiguousarray(v)).view(torch.float8_e4m3fn).double()
        return kt * torch.from_numpy(c.k_scale[blk, h]).double()[:, None], \
            vt * torch.from_numpy(c.v_scale[blk, h]).double()[:, None]
    return (torch.from_numpy(np.ascontiguousarray(k).view(np.int16)).view(torch.bfloat16).double(),
            torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).double())


def _library_reference(c, q, tables, lens, q_start, Hq, scale):
    Hkv = c.Hkv
    G = Hq // Hkv
    out = torch.zeros(q.shape, dtype=torch.float64)
    for b, n in enumerate(lens):
        C = int(q_start[b + 1] - q_start[b])
        if C == 0:
            continue
        rows = slice(int(q_start[b]), int(q_start[b + 1]))
        qpos = torch.arange(n - C, n)
        mask = torch.arange(n)[None, :] <= qpos[:, None]          # [C, n]
        for h in range(Hkv):
            k, v = _gather(c, tables[b], int(n), h)
            qq = q[rows, h * G:(h + 1) * G].double().permute(1, 0, 2)   # [G, C, d]
            o = torch.nn.functional.scaled_dot_product_attention(
                qq, k.expand(G, -1, -1), v.expand(G, -1, -1), attn_mask=mask, scale=scale)
            out[rows, h * G:(h + 1) * G] = o.permute(1, 0, 2)
    return out.numpy()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("G", [1, 4])
def test_chunks_equal_library_causal_attention(kv, G):
    Hkv, d, bs = 2, 64 if kv == "bf16" else 128, 16
    Hq = Hkv * G
    lens = [37, 5, 64, 1, 100]
    C = [37, 5, 20, 1, 3]              # whole sequence, whole, a middle chunk, one token, verify
    c, tables = _cache(kv, len(lens), Hkv, d, bs, lens, seed=3 + G)
    q_start = np.concatenate([[0], np.cumsum(C)]).astype(np.int32)
    q = torch.randn(int(q_start[-1]), Hq, d, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    scale = 1.0 / np.sqrt(d)
    got = oracle.prefill_attention(c, q, tables, np.asarray(lens), q_start, Hq, scale)
    ref = _library_reference(c, q, tables, lens, q_start, Hq, scale)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_one_token_chunks_equal_decode_and_empty_chunks_write_nothing():
    Hkv, G, d, bs = 2, 2, 64, 16
    lens = [1, 17, 50, 0]
    c, tables = _cache("bf16", 4, Hkv, d, bs, lens, seed=8)
    q = torch.randn(4, Hkv * G, d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    q_start = np.array([0, 1, 2, 3, 3], dtype=np.int32)
    got = oracle.prefill_attention(c, q[:3], tables, np.asarray(lens), q_start, Hkv * G, 0.125)
    dec = oracle.decode_attention(c, q[:3], tables[:3], np.asarray(lens[:3]), Hkv * G, 0.125)
    assert np.array_equal(got, dec)


def test_verify_chunk_equals_sequential_decode_steps():
    # "LLM Serving - ...", Speculative decoding: the target scores K proposals in
    # one pass; query i of the chunk sees exactly what decode step i would see
    Hkv, G, d, bs, K = 2, 4, 64, 16, 4
    L = 53
    c, tables = _cache("bf16", 1, Hkv, d, bs, [L], seed=4)
    q = torch.randn(K + 1, Hkv * G, d, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    got = oracle.prefill_attention(c, q, tables, np.array([L]), np.array([0, K + 1]), Hkv * G, 0.125)
    for i in range(K + 1):
        step = oracle.decode_attention(c, q[i:i + 1], tables, np.array([L - K + i]), Hkv * G, 0.125)
        assert np.array_equal(got[i:i + 1], step)


def test_more_queries_than_cached_tokens_is_rejected():
    c, tables = _cache("bf16", 1, 1, 64, 16, [4], seed=1)
    q = torch.zeros(5, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.prefill_attention(c, q, tables, np.array([4]), np.array([0, 5]), 1, 0.125)
