"""Pins for the oracle's decode attention, independent of the oracle's own code.

What pins it:
  * brute-force dense attention written here with numpy (softmax(q K^T s) V
    over logically ordered, contiguous K/V), for random shapes, ragged
    lengths and random physical-block permutations ("KV cache & continuous
    batching", section "2. PagedAttention": the paged kernel gathers the same
    K/V through the block table);
  * the hands-on identity of "LLM Serving - KV Cache, Batching, Speculative
    Decoding" (section "Hands-on: cache equivalence and scheduling oracles"):
    cached attention at position t equals the last row of full causal
    attention at 1e-12 in fp64, and wrong cached values break it;
  * closed forms: one token returns its V row exactly, equal scores return
    the mean of V, a dominant score returns its V row, GQA head grouping;
  * split-K partitions merged by log-sum-exp equal the unsplit result.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def bf16_round(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def bf16_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def build_case(rng, B, Hq, Hkv, d, bs, lens, num_blocks, perm=None):
    """Random bf16 K/V per sequence (logical order) and a paged oracle cache."""
    M = max(1, max(-(-L // bs) for L in lens))
    need = sum(-(-L // bs) for L in lens)
    if perm is None:
        perm = rng.permutation(num_blocks)
    assert need <= num_blocks
    tables = np.full((B, M), -1, np.int32)
    p = 0
    for b, L in enumerate(lens):
        nb = -(-L // bs)
        tables[b, :nb] = perm[p:p + nb]
        p += nb
    k_log = [bf16_round(rng.standard_normal((L, Hkv, d))) for L in lens]
    v_log = [bf16_round(rng.standard_normal((L, Hkv, d))) for L in lens]
    q = bf16_round(rng.standard_normal((B, Hq, d)))
    return tables, k_log, v_log, q, M


def fill_cache(cache, tables, k_log, v_log, bs):
    for b, (k, v) in enumerate(zip(k_log, v_log)):
        L = k.shape[0]
        if L == 0:
            continue
        pos = np.arange(L, dtype=np.int32)
        slots = oracle.slot_mapping(tables, np.full(L, b, np.int32), pos, bs)
        cache.append(k, v, slots)


def dense_reference(q, k_log, v_log, Hq, Hkv, scale):
    """softmax(q K^T * scale) V over contiguous K/V; query head i reads KV head i // (Hq/Hkv)."""
    G = Hq // Hkv
    qd = bf16_f64(q)
    out = np.zeros(qd.shape, dtype=np.float64)
    for b in range(qd.shape[0]):
        K = bf16_f64(k_log[b])
        V = bf16_f64(v_log[b])
        if K.shape[0] == 0:
            continue
        for i in range(Hq):
            s = K[:, i // G, :] @ qd[b, i] * scale
            w = np.exp(s - s.max())
            out[b, i] = (w / w.sum()) @ V[:, i // G, :]
    return out


SHAPES = [
    # B, Hq, Hkv, d, bs, lens
    (4, 4, 2, 64, 16, [1, 17, 50, 100]),
    (3, 8, 8, 32, 16, [16, 33, 5]),          # MHA
    (3, 8, 1, 16, 8, [9, 1, 24]),            # MQA
    (2, 16, 2, 32, 32, [31, 65]),            # G = 8
    (5, 6, 3, 8, 4, [4, 5, 3, 12, 1]),       # odd head count
]


@pytest.mark.parametrize("shape", SHAPES)
def test_paged_equals_dense_bruteforce(shape):
    B, Hq, Hkv, d, bs, lens = shape
    rng = np.random.default_rng(1234 + B * 7 + d)
    nb = sum(-(-L // bs) for L in lens) + 5
    tables, k_log, v_log, q, M = build_case(rng, B, Hq, Hkv, d, bs, lens, nb)
    cache = oracle.Cache(nb, Hkv, d, bs)
    fill_cache(cache, tables, k_log, v_log, bs)
    scale = 1.0 / math.sqrt(d)
    got = oracle.decode_attention(cache, q, tables, np.array(lens, np.int32), Hq, scale)
    ref = dense_reference(q, k_log, v_log, Hq, Hkv, scale)
    assert np.max(np.abs(got - ref)) <= 1e-12


def test_permutation_invariance_bit_identical():
    B, Hq, Hkv, d, bs, lens = 4, 8, 2, 64, 16, [1, 17, 50, 100]
    nb = 40
    outs = []
    for seed in (1, 2, 3):
        rng_data = np.random.default_rng(99)            # same values every time
        rng_perm = np.random.default_rng(seed)          # different physical placement
        perm = rng_perm.permutation(nb)
        tables, k_log, v_log, q, M = build_case(rng_data, B, Hq, Hkv, d, bs, lens, nb, perm=perm)
        cache = oracle.Cache(nb, Hkv, d, bs)
        fill_cache(cache, tables, k_log, v_log, bs)
        outs.append(oracle.decode_attention(cache, q, tables, np.array(lens, np.int32), Hq, 0.125))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_cached_equals_causal_last_row_and_wrong_values_break_it():
    """The hands-on identity: 7 positions of width 4, projections Wq/Wk/Wv."""
    rng = np.random.default_rng(124)
    x = rng.standard_normal((7, 4))
    Wq, Wk, Wv = (rng.standard_normal((4, 4)) for _ in range(3))
    # the oracle consumes bf16 operands: round the projections once, use them on both sides
    qa = bf16_f64(bf16_round(x @ Wq))
    ka = bf16_round(x @ Wk)
    va = bf16_round(x @ Wv)
    bs, nb = 2, 8
    perm = np.array([5, 2, 7, 0], dtype=np.int32)
    tables = perm[None, :]
    cache = oracle.Cache(nb, 1, 4, bs)
    for t in range(7):
        slot = oracle.slot_mapping(tables, np.zeros(1, np.int32), np.array([t], np.int32), bs)
        cache.append(ka[t:t + 1, None, :], va[t:t + 1, None, :], slot)
        q_t = bf16_round(qa[t:t + 1])[:, None, :]
        cached = oracle.decode_attention(cache, q_t, tables, np.array([t + 1], np.int32), 1, 0.5)
        # full causal attention over the first t+1 positions, last row
        Kf, Vf = bf16_f64(ka[: t + 1]), bf16_f64(va[: t + 1])
        Qf = qa[: t + 1]
        sc = Qf @ Kf.T / math.sqrt(4)
        sc[np.triu(np.ones_like(sc, dtype=bool), 1)] = -np.inf
        w = np.exp(sc - sc.max(axis=1, keepdims=True))
        full = (w / w.sum(axis=1, keepdims=True)) @ Vf
        assert np.allclose(cached[0, 0], full[-1], atol=1e-12, rtol=0)
    # wrong prefix values (V + 1 in the cache) break the identity
    cache.v[...] = bf16_round(bf16_f64(torch.from_numpy(cache.v.view(np.int16)).view(torch.bfloat16)) + 1) \
        .view(torch.int16).numpy().view(np.uint16)
    wrong = oracle.decode_attention(cache, bf16_round(qa[6:7])[:, None, :], tables,
                                    np.array([7], np.int32), 1, 0.5)
    assert not np.allclose(wrong[0, 0], full[-1], atol=1e-6)


def _single(lens, k_rows, v_rows, q_row, scale, bs=4):
    L = len(k_rows)
    tables = np.arange(max(1, -(-L // bs)), dtype=np.int32)[None, :]
    cache = oracle.Cache(tables.shape[1], 1, len(q_row), bs)
    if L:
        slots = oracle.slot_mapping(tables, np.zeros(L, np.int32), np.arange(L, dtype=np.int32), bs)
        cache.append(bf16_round(np.array(k_rows))[:, None, :], bf16_round(np.array(v_rows))[:, None, :],
                     slots)
    return oracle.decode_attention(cache, bf16_round(np.array([q_row]))[:, None, :], tables,
                                   np.array([lens], np.int32), 1, scale)[0, 0]


def test_one_token_returns_v_exactly():
    out = _single(1, [[0.5, -2.0, 3.0]], [[1.25, -0.75, 7.0]], [1.0, 2.0, 3.0], 0.37)
    assert np.array_equal(out, np.array([1.25, -0.75, 7.0]))


def test_equal_scores_give_mean_of_v():
    rng = np.random.default_rng(5)
    V = bf16_f64(bf16_round(rng.standard_normal((13, 8))))
    K = np.tile(rng.standard_normal(8), (13, 1))
    out = _single(13, K, V, rng.standard_normal(8), 0.3)
    assert np.max(np.abs(out - V.mean(axis=0))) <= 1e-12
    # scale 0 makes every score equal whatever the keys
    out0 = _single(13, rng.standard_normal((13, 8)), V, rng.standard_normal(8), 0.0)
    assert np.max(np.abs(out0 - V.mean(axis=0))) <= 1e-12


def test_dominant_score_selects_its_row():
    K = np.zeros((9, 4))
    K[6] = [64.0, 0, 0, 0]
    V = np.arange(36, dtype=np.float64).reshape(9, 4)
    out = _single(9, K, V, [1.0, 0, 0, 0], 1.0)
    # weight of the other rows is 8 * exp(-64)
    assert np.max(np.abs(out - V[6])) <= 36 * 8 * math.exp(-64)


def test_gqa_heads_read_their_group_kv_head():
    """Query head i uses KV head i // G: make KV head 1's V constant 5, head 0's constant -3."""
    Hq, Hkv, d, bs, L = 6, 2, 8, 4, 7
    tables = np.arange(2, dtype=np.int32)[None, :]
    cache = oracle.Cache(2, Hkv, d, bs)
    rng = np.random.default_rng(0)
    k = bf16_round(rng.standard_normal((L, Hkv, d)))
    v = np.zeros((L, Hkv, d))
    v[:, 0, :] = -3.0
    v[:, 1, :] = 5.0
    slots = oracle.slot_mapping(tables, np.zeros(L, np.int32), np.arange(L, dtype=np.int32), bs)
    cache.append(k, bf16_round(v), slots)
    q = bf16_round(rng.standard_normal((1, Hq, d)))
    out = oracle.decode_attention(cache, q, tables, np.array([L], np.int32), Hq, 0.35)
    assert np.max(np.abs(out[0, :3] + 3.0)) <= 1e-12 and np.max(np.abs(out[0, 3:] - 5.0)) <= 1e-12


@pytest.mark.parametrize("part", [1, 2, 3, 7, 64])
def test_split_merge_equals_unsplit(part):
    B, Hq, Hkv, d, bs, lens = 4, 8, 2, 32, 16, [1, 40, 100, 257]
    rng = np.random.default_rng(77)
    nb = sum(-(-L // bs) for L in lens) + 3
    tables, k_log, v_log, q, M = build_case(rng, B, Hq, Hkv, d, bs, lens, nb)
    cache = oracle.Cache(nb, Hkv, d, bs)
    fill_cache(cache, tables, k_log, v_log, bs)
    L = np.array(lens, np.int32)
    ref = oracle.decode_attention(cache, q, tables, L, Hq, 0.2)
    got = oracle.decode_attention(cache, q, tables, L, Hq, 0.2, part_blocks=part)
    assert np.max(np.abs(got - ref)) <= 1e-12


def test_zero_length_sequence_gives_zero_row():
    rng = np.random.default_rng(3)
    tables, k_log, v_log, q, M = build_case(rng, 2, 2, 1, 8, 4, [0, 5], 4)
    cache = oracle.Cache(4, 1, 8, 4)
    fill_cache(cache, tables, k_log, v_log, 4)
    out = oracle.decode_attention(cache, q, tables, np.array([0, 5], np.int32), 2, 0.5)
    assert np.all(out[0] == 0.0)
    assert np.max(np.abs(out[1] - dense_reference(q[1:], k_log[1:], v_log[1:], 2, 1, 0.5)[0])) <= 1e-12


def test_bad_block_id_is_rejected():
    cache = oracle.Cache(4, 1, 8, 4)
    tables = np.array([[0, 9]], np.int32)
    q = bf16_round(np.ones((1, 1, 8)))
    with pytest.raises(ValueError):
        oracle.decode_attention(cache, q, tables, np.array([6], np.int32), 1, 0.5)


def test_threaded_equals_serial():
    rng = np.random.default_rng(8)
    lens = [3, 50, 17, 64, 1, 33]
    tables, k_log, v_log, q, M = build_case(rng, 6, 4, 2, 16, 16, lens, 20)
    cache = oracle.Cache(20, 2, 16, 16)
    fill_cache(cache, tables, k_log, v_log, 16)
    L = np.array(lens, np.int32)
    a = oracle.decode_attention(cache, q, tables, L, 4, 0.25)
    b = oracle.decode_attention(cache, q, tables, L, 4, 0.25, threads=4)
    assert np.array_equal(a, b)
