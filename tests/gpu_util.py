"""Helpers for the GPU parity tests: run a workload through the C ABI and the oracle."""
import numpy as np
import torch

import oracle
import oracle.run
import paged_kv_cache_294_gb300 as pa
from paged_kv_cache_294_gb300.engine import PagedDecodeLayer

BF16_TOL = 1e-2     # max |err| of bf16-cache attention outputs
FP8_TOL = 5e-2      # max |err| of fp8-cache outputs against the oracle on the stored fp8 cache
INT8_TOL = 1e-2     # int8 / int4 caches: codes are exact in f16, so the bf16 output bound applies


def tol(w):
    return {"fp8": FP8_TOL, "int8": INT8_TOL, "int4": INT8_TOL}.get(w.kv, BF16_TOL)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of the bf16 grid (8 significant bits) in the binade of |x|."""
    a = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


# Bound on the kernel's error before the output's final rounding to bf16 (fp32
# accumulation; the probabilities enter P.V as 16-bit operands).  Only used
# where half a bf16 spacing at ref plus this exceeds atol.
ROUND_EPS = 2.0 ** -10


def allowed_err(ref: np.ndarray, atol: float) -> np.ndarray:
    """Per-output bound: atol, or half a bf16 spacing of the reference plus
    ROUND_EPS, whichever is larger.  The outputs are bf16: a correctly rounded
    output misses the exact value by up to half a spacing, so where that half
    spacing exceeds atol (|ref| >= 4 for 1e-2, >= 16 for 5e-2) no kernel can
    meet atol itself.  Below those magnitudes the bound is atol exactly."""
    return np.maximum(atol, 0.5 * bf16_ulp(ref) + ROUND_EPS)


def worst(got: np.ndarray, ref: np.ndarray, atol: float) -> str:
    """The output furthest outside (or closest to) its bound, for failure messages."""
    if not got.size:
        return "no outputs"
    r = np.abs(got - ref) / allowed_err(ref, atol)
    i = np.unravel_index(int(np.argmax(r)), r.shape)
    return "worst at %s: ref %.6g got %.6g |err| %.3g bound %.3g (%.3f of it)" % (
        tuple(int(x) for x in i), float(ref[i]), float(got[i]), float(abs(got[i] - ref[i])),
        float(allowed_err(ref[i], atol)), float(r[i]))


def excess(got: np.ndarray, ref: np.ndarray, atol: float) -> float:
    """max over outputs of |got - ref| / allowed_err; parity holds when <= 1."""
    return float(np.max(np.abs(got - ref) / allowed_err(ref, atol))) if got.size else 0.0


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
    return t.cpu().numpy().view(np.uint8)
