"""pa_kv_append through the C ABI against the oracle: bit-exact cache bytes and scales."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_294_gb300 as pa
import workloads
from tests.gpu_util import cache_bytes, oracle_out, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("8b", dict(B=6, seq_len=700)),
                                     ("70b", dict(B=8, seq_len=400)),
                                     ("fp8prefix", dict(B=6, seq_len=600)),
                                     ("8b-int8", dict(B=6, seq_len=700)),
                                     ("8b-int4", dict(B=6, seq_len=700))])
def test_workload_caches_bit_exact(name, kw):
    w = workloads.make(name, **kw)
    layer = run_gpu(w)
    st, _ = oracle_out(w)
    assert pa.pa_get_device_error() == 0
    assert np.array_equal(cache_bytes(layer.k_cache), st.cache.k.reshape(layer.k_cache.shape))
    assert np.array_equal(cache_bytes(layer.v_cache), st.cache.v.reshape(layer.v_cache.shape))
    if w.kv != "bf16":
        assert np.array_equal(layer.k_scale.cpu().numpy().view(np.uint32), st.cache.k_scale.view(np.uint32))
        assert np.array_equal(layer.v_scale.cpu().numpy().view(np.uint32), st.cache.v_scale.view(np.uint32))


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


class Pair:
    """The same cache on the GPU (through the C ABI) and in the oracle."""

    def __init__(self, nb, hkv, d, bs, kv):
        self.o = oracle.Cache(nb, hkv, d, bs, kv)
        dt = {"bf16": torch.bfloat16, "fp8": torch.uint8, "int8": torch.int8, "int4": torch.uint8}[kv]
        self.k = torch.zeros((nb, hkv, bs, d // 2 if kv == "int4" else d), dtype=dt, device="cuda")
        self.v = torch.zeros_like(self.k)
        self.ks = torch.zeros((nb, hkv), dtype=torch.float32, device="cuda") if kv != "bf16" else None
        self.vs = torch.zeros_like(self.ks) if kv != "bf16" else None

    def append(self, k, v, slots):
        slots = np.asarray(slots, np.int64)
        pa.pa_kv_append(self.k, self.v, self.ks, self.vs, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda())
        self.o.append(k, v, slots)

    def check(self):
        torch.cuda.synchronize()
        assert np.array_equal(cache_bytes(self.k), self.o.k)
        assert np.array_equal(cache_bytes(self.v), self.o.v)
        if self.ks is not None:
            assert np.array_equal(self.ks.cpu().numpy().view(np.uint32), self.o.k_scale.view(np.uint32))
            assert np.array_equal(self.vs.cpu().numpy().view(np.uint32), self.o.v_scale.view(np.uint32))


@pytest.mark.parametrize("d,bs", [(64, 16), (128, 16), (128, 32), (64, 32)])
def test_bf16_scatter_with_skips(d, bs):
    rng = np.random.default_rng(d + bs)
    p = Pair(9, 3, d, bs, "bf16")
    T = 40
    slots = rng.permutation(9 * bs)[:T].astype(np.int64)
    slots[::7] = -1
    k = _bf16(rng.standard_normal((T, 3, d)))
    v = _bf16(rng.standard_normal((T, 3, d)))
    p.append(k, v, slots)
    p.check()
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("kv", ["fp8", "int8", "int4"])
@pytest.mark.parametrize("bs", [16, 32])
def test_one_byte_growth_restart_and_runs(bs, kv):
    rng = np.random.default_rng(bs)
    p = Pair(6, 2, 128, bs, kv)
    # a prefill run across three blocks, with a skipped token in the middle of the call
    k = _bf16(rng.standard_normal((2 * bs + 5, 2, 128)))
    slots = np.concatenate([np.arange(bs, 3 * bs), [-1], np.arange(4 * bs, 4 * bs + 4)])
    p.append(k, k, slots)
    p.check()
    # decode appends: first smaller (no growth), then larger (growth re-encodes older rows)
    for mult, off in ((0.01, 5), (20.0, 6), (1.0, 7), (300.0, 8)):
        x = _bf16(rng.standard_normal((1, 2, 128)) * mult)
        p.append(x, x, np.array([4 * bs + off], np.int64))
        p.check()
    # a write at offset 0 restarts block 1
    x = _bf16(rng.standard_normal((1, 2, 128)) * 0.5)
    p.append(x, x, np.array([bs], np.int64))
    p.check()
    # all-zero values into a fresh block: scale 0, codes 0
    z = _bf16(np.zeros((3, 2, 128)))
    p.append(z, z, np.array([5 * bs, 5 * bs + 1, 5 * bs + 2], np.int64))
    p.check()
    # extreme magnitudes saturate nothing beyond rounding
    big = _bf16(np.concatenate([rng.standard_normal((2, 2, 128)) * 1e30,
                                rng.standard_normal((2, 2, 128)) * 1e-30]))
    p.append(big[:2], big[2:], np.array([2, 3], np.int64))
    p.check()
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("kv", ["fp8", "int8", "int4"])
def test_one_byte_one_token_per_sequence_many_blocks(kv):
    rng = np.random.default_rng(11)
    p = Pair(64, 4, 128, 32, kv)
    hist = _bf16(rng.standard_normal((64 * 20, 4, 128)))
    slots = np.concatenate([np.arange(b * 32, b * 32 + 20) for b in range(64)])
    p.append(hist, hist, slots)
    new = _bf16(rng.standard_normal((64, 4, 128)) * rng.uniform(0.1, 3.0, size=(64, 1, 1)))
    p.append(new, new, np.arange(64) * 32 + 20)
    p.check()


def test_empty_append_is_a_noop():
    p = Pair(2, 1, 128, 16, "bf16")
    p.append(_bf16(np.zeros((0, 1, 128))), _bf16(np.zeros((0, 1, 128))), np.zeros(0, np.int64))
    p.check()
