"""The oracle and the product share no code, and the product has no CPU path.

Checked statically over the sources: nothing in the product package, the C
header or the kernels names the oracle; nothing in the oracle names the
product, its header or its kernels; the shared input generators import
neither.  And a device entry point given CPU tensors refuses them instead of
computing anything on the host.
"""
import os
import re

import pytest
import torch

import paged_kv_cache_294_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC_EXT = (".py", ".cu", ".cuh", ".cpp", ".h", ".c")


def _sources(*dirs):
    for d in dirs:
        for dp, dn, fn in os.walk(os.path.join(ROOT, d)):
            dn[:] = [x for x in dn if x not in ("__pycache__", "_build", "build")]
            for f in fn:
                if f.endswith(SRC_EXT):
                    yield os.path.join(dp, f)


def test_product_never_names_the_oracle():
    for path in _sources("paged_kv_cache_294_gb300", "include"):
        text = open(path, encoding="utf-8").read()
        assert not re.search(r"\boracle\b", text, re.I), path


def test_oracle_never_names_the_product():
    for path in _sources("oracle"):
        text = open(path, encoding="utf-8").read()
        for token in ("paged_kv_cache_294_gb300", "pa.h", "csrc", "libpagedattn", "workloads"):
            assert token not in text, (path, token)


def test_input_generators_import_neither_side():
    text = open(os.path.join(ROOT, "workloads.py"), encoding="utf-8").read()
    imports = re.findall(r"^\s*(?:import|from)\s+([\w.]+)", text, re.M)
    assert not any(m.split(".")[0] in ("oracle", "paged_kv_cache_294_gb300") for m in imports), imports


def test_device_calls_refuse_host_tensors():
    bf = torch.bfloat16
    q = torch.zeros(1, 8, 128, dtype=bf)
    out = torch.zeros_like(q)
    kc = torch.zeros(4, 2, 16, 128, dtype=bf)
    tables = torch.zeros(1, 4, dtype=torch.int32)
    lens = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        pa.pa_decode_attention(out, q, kc, kc.clone(), None, None, tables, lens, 0.1)
    with pytest.raises(ValueError, match="CUDA"):
        pa.pa_kv_append(kc, kc.clone(), None, None, torch.zeros(1, 2, 128, dtype=bf),
                        torch.zeros(1, 2, 128, dtype=bf), torch.zeros(1, dtype=torch.int64))
