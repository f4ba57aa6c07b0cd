"""Helpers for the GPU parity tests: run a workload through the C ABI and the oracle."""
import numpy as np
import torch

import oracle
import oracle.run
import paged_kv_cache_294_gb300 as pa
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer

BF16_TOL = 1e-2     # max |err| of bf16-cache attention outputs
FP8_TOL = 5e-2      # max |err| of fp8-cache outputs against the oracle on the stored fp8 cache


def tol(w):
    return FP8_TOL if w.kv == "fp8" else BF16_TOL


def run_gpu(w, num_splits=0, device="cuda"):
    layer = PagedDecodeLayer.from_workload(w, device)
    pa.pa_get_device_error(clear=True)
    layer.step(num_splits=num_splits)
    torch.cuda.synchronize()
    return layer


def oracle_out(w, seqs=None, tables=None):
    st = oracle.run.OracleStep(w, seqs=seqs, tables=tables)
    st.append()
    return st, st.decode(threads=8)


def gpu_out_f64(layer, seqs=None):
    o = layer.out.float().cpu().numpy().astype(np.float64)
    return o if seqs is None else o[np.asarray(sorted(set(int(s) for s in seqs)))]


def cache_bytes(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()
