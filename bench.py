"""Benchmark: paged decode attention on one GB300 (or N independent replicas).

A step is one decode iteration of one attention layer over the whole batch:
the append of every sequence's new token, attention and the split-K merge,
in one launch (pa_decode_step).  The metric is the KV-read bandwidth of that
step, counted from the algorithmic bytes (K/V of every cached token read once,
q read, out written), also reported as sequence-steps per second and as a
fraction of the measured HBM peak.

    python bench.py [--workload all|8b|70b|long|fp8prefix|8b-int8|8b-int4|tiny]
                    [--steps K] [--warmup W] [--splits S] [--impl ours|reference]
                    [--gpus N]

The default run measures every workload and prints them under "workloads";
the line's headline (value, config, roofline, e2e) is the Llama-3-70B-shaped
continuous-batching step.  The long-context workload is also timed at every
split count from 1 to 64 ("long_split_sweep").  Before timing, each
workload's step is checked against the fp64 oracle on every output of every
sequence.  Prints one JSON line (rank 0).  With torchrun (N > 1) every rank
runs independent replicas of the workloads on its own GPU (the path has no
exchange step); value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged decode attention KV-read GB/s (% of GB300 HBM peak), seq-steps/sec"
UNIT = "GB/s"
FALLBACK_BF16 = 1900.0
FALLBACK_HBM = 6800.0


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM, "fallback"


def row_bytes(w):
    """Bytes of one token row of one kv head: 2 per element (bf16), 1 (fp8, int8), 1/2 (int4)."""
    return {"bf16": 2 * w.d, "int4": w.d // 2}.get(w.kv, w.d)


def algorithmic_bytes(w):
    """K/V bytes of every cached token of every sequence (logical, once per sequence),
    plus q read and out written.  Unique-physical KV bytes reported beside it."""
    tok = 2 * w.Hkv * row_bytes(w)
    lens = np.asarray(w.seq_lens, dtype=np.int64)
    qo = 2 * w.B * w.Hq * w.d * 2
    return int(lens.sum()) * tok + qo, int(lens.sum()) * tok, qo


def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16, "fallback"


def prefill_flops(w):
    """Causal multi-query attention FLOPs: query i of a C-token chunk over L cached
    positions scores L - C + i + 1 keys; 2 d FLOPs per score for Q K^T, 2 d for P V."""
    tot = 0
    for b in range(w.B):
        C = int(w.q_start[b + 1] - w.q_start[b])
        L = int(w.seq_lens[b])
        tot += C * (L - C) + C * (C + 1) // 2
    return 4 * w.d * w.Hq * tot


def unique_kv_bytes(w, tables):
    """K/V bytes of distinct cached tokens: a physical block shared by several
    sequences (a common prefix) counts once, with as many tokens as its longest
    user fills.  Equals the logical count when no block is shared."""
    used = {}
    for b, L in enumerate(w.seq_lens):
        L = int(L)
        for j in range(-(-L // w.bs)):
            p = int(tables[b, j])
            used[p] = max(used.get(p, 0), min(w.bs, L - j * w.bs))
    return sum(used.values()) * 2 * w.Hkv * row_bytes(w)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            sel = str(device_index)
        self.cmd = ["nvidia-smi", "-i", sel, "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                    "-lms", "200"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_source_hash():
    """Hash of the decode kernel's sources without comments and blank lines, so
    that a comment edit keeps the recorded ncu traffic while any code change
    drops it."""
    h = hashlib.sha256()
    for f in ("pa_decode.cu", "pa_device.cuh", "pa_fp8.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_294_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        lines = [ln.rstrip() for ln in src.splitlines()]
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload, splits_used):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken
    on the current kernel source for this workload; else None."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel_hash") == kernel_source_hash() and e.get("splits") == splits_used:
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        return dist, dist.get_rank(), ws
    return None, 0, 1


def max_over_ranks(t: float, dist, device="cpu") -> float:
    """The slowest rank's time (every rank gets it); t itself on one process."""
    if not dist:
        return t
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt[0])


HEADLINE = "70b"
ALL_WORKLOADS = ("8b", "70b", "long", "fp8prefix", "8b-int8", "8b-int4")
SPLIT_SWEEP = (1, 2, 4, 8, 16, 32, 64)


def oracle_sample(w):
    """The sequences both CPU arms time per step: a seeded eighth of the batch
    (at least one).  One helper, so that the CPU baseline and the reference
    arm time the same work."""
    n = max(1, w.B // 8)
    return sorted(np.random.default_rng(294).permutation(w.B)[:n].tolist())


def sample_bytes(w, seqs):
    lens = np.asarray(w.seq_lens, dtype=np.int64)[seqs]
    return int(lens.sum()) * 2 * w.Hkv * row_bytes(w) + 2 * len(seqs) * w.Hq * w.d * 2


def cpu_oracle_baseline(w, tables, budget_s=10.0, threads=None):
    """The fp64 oracle's step (append of the new token + decode attention) on
    oracle_sample(w), repeated for about budget_s of wall time."""
    import oracle.run
    threads = threads or os.cpu_count() or 1
    seqs = oracle_sample(w)
    st = oracle.run.OracleStep(w, seqs=seqs, tables=tables)
    reps, total = 0, 0.0
    while (total < budget_s or reps < 2) and reps < 1000:
        # re-appending the same token rewrites the same cache bytes: every rep is the same step
        t0 = time.perf_counter()
        st.append()
        st.decode(threads=threads)
        total += time.perf_counter() - t0
        reps += 1
    per_step = total / reps
    # the same step on one thread, once (a few seconds)
    t0 = time.perf_counter()
    st.append()
    st.decode(threads=1)
    one = time.perf_counter() - t0
    return {"value": sample_bytes(w, seqs) / per_step / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "%d of %d sequences (%d tokens; the same sample as the reference arm), fp64 C oracle "
                      "append+decode, %d reps, %.1f s" % (len(seqs), w.B, int(np.sum(np.asarray(w.seq_lens)[seqs])),
                                                          reps, total),
            "seq_steps_per_s": len(seqs) / per_step,
            "one_thread": {"value": sample_bytes(w, seqs) / one / 1e9, "unit": UNIT, "reps": 1},
            "cpu": cpu_model()}


def cpu_model():
    """The host CPU's name as /proc/cpuinfo gives it (x86 'model name'; Arm
    implementer / part codes), else the platform's."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k = k.strip()
                if k and k not in fields:
                    fields[k] = v.strip()
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return "%s, implementer %s, part %s" % (platform.machine(), fields.get("CPU implementer", "?"),
                                                 fields["CPU part"])
    return platform.processor() or platform.machine()


def run_reference(args):
    """The oracle arm: the fp64 CPU oracle timed on the host cores, rank 0 only,
    on the workload and metric of our arm's headline, each step oracle_sample(w)."""
    dist, rank, world = dist_init()
    if rank != 0:
        return
    name = HEADLINE if args.workload == "all" else args.workload
    w = workloads.make(name, device="cpu", B=args.batch)
    import oracle.run
    tables = oracle.run.tables_of(w)
    threads = os.cpu_count() or 1
    seqs = oracle_sample(w)
    times = []
    st = oracle.run.OracleStep(w, seqs=seqs, tables=tables)
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        st.append()
        st.decode(threads=threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    t = sum(times)
    value = sample_bytes(w, seqs) * len(times) / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "seq_steps_per_s": len(seqs) * len(times) / t,
            "config": {"workload": name, "desc": w.desc, "sample_sequences": len(seqs)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": "%d of %d sequences per step (the same sample as our arm's cpu_baseline), "
                                       "fp64 C oracle append+decode" % (len(seqs), w.B)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


class Bench:
    """Timing machinery shared by every measurement of one run."""

    def __init__(self, args, dev, dist):
        self.args, self.dev, self.dist = args, dev, dist
        self.flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)   # > 2 x L2
        self.stream = torch.cuda.current_stream(dev)
        self.clock_lines = []

    def flush_l2(self):
        # write then read 512 MiB: evicts the previous step's lines and leaves no
        # dirty lines whose write-back would overlap the timed region
        self.flush.fill_(1)
        self.flush.sum(dtype=torch.int32)

    def timed(self, fn, K):
        """Per-step CUDA-event time (s, summed over K steps), L2 flushed before each (untimed)."""
        for _ in range(self.args.warmup):
            self.flush_l2()
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        if self.dist:
            self.dist.barrier()
        torch.cuda.synchronize()
        for i in range(K):
            self.flush_l2()
            ev[i][0].record(self.stream)
            fn()
            ev[i][1].record(self.stream)
        torch.cuda.synchronize()
        self.last_steps_ms = [x.elapsed_time(y) for x, y in ev]
        t = sum(self.last_steps_ms) / 1e3
        return max_over_ranks(t, self.dist, self.dev)

    def step_stats(self):
        """Median and 90th percentile of the last timed() call's steps (µs, this rank)."""
        v = np.asarray(self.last_steps_ms) * 1e3
        return {"median_us": float(np.median(v)), "p90_us": float(np.percentile(v, 90)), "steps": int(v.size)}


def parity_bound(ref, tol):
    """Per-output bound: tol, or half a bf16 spacing of ref plus 2^-10 where
    that is larger (the outputs are bf16: only for |ref| >= 4 at tol 1e-2)."""
    a = np.maximum(np.abs(ref), 2.0 ** -126)
    return np.maximum(tol, 0.5 * 2.0 ** (np.floor(np.log2(a)) - 7) + 2.0 ** -10)


def parity_full(w, out, ref, flags):
    """Every output of every sequence against the oracle's (fp64)."""
    got = out.float().cpu().numpy().astype(np.float64)
    tol = {"fp8": 5e-2}.get(w.kv, 1e-2)
    err = np.abs(got - ref)
    ex = float(np.max(err / parity_bound(ref, tol))) if err.size else 0.0
    return {"max_abs_err": float(err.max()) if err.size else 0.0, "max_err_over_bound": ex, "tol": tol,
            "sequences": "all %d" % w.B, "outputs": int(err.size),
            "ok": bool(ex <= 1.0 and flags == 0 and np.all(np.isfinite(got)))}


def clock_summary(lines):
    cs = ClockSampler.__new__(ClockSampler)
    cs.lines = lines
    return ClockSampler.summary(cs)


def e2e_measure(bn, layer, K, world, alg):
    """The step through the public API with host buffers: each step copies its
    inputs (q, new K/V, tables, lengths) in from pinned host memory and its
    output back, all inside the timed region.  Returns (pipelined, serial)."""
    dev, stream, args = bn.dev, bn.stream, bn.args
    parts = [layer.q, layer.k_new, layer.v_new, layer.block_tables, layer.seq_lens]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_sets = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]

    def view(buf, i):
        t = parts[i]
        n = t.numel() * t.element_size()
        return buf[offs[i]:offs[i] + n].view(t.dtype).view(t.shape)

    for i, t in enumerate(parts):
        view(h_buf, i).copy_(t.cpu())
    d_views = [[view(buf, i) for i in range(len(parts))] for buf in d_sets]
    outs = [torch.empty_like(layer.out) for _ in range(2)]
    h_outs = [torch.empty(tuple(layer.out.shape), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d, d2h = total, h_outs[0].numel() * h_outs[0].element_size()

    def serial_step():
        d_sets[0].copy_(h_buf, non_blocking=True)
        q_, kn_, vn_, tab_, len_ = d_views[0]
        layer.fused_step(q=q_, k_new=kn_, v_new=vn_, out=outs[0], num_splits=args.splits, tables=tab_, lens=len_)
        h_outs[0].copy_(outs[0], non_blocking=True)

    t_serial = bn.timed(serial_step, K)

    # as a serving loop issues the steps: two sets of device buffers, one stream
    # per copy direction, so step i+1's input copy and step i-1's output copy run
    # while step i's kernel runs; the timed region ends when the last output has
    # reached the host.  The cache each step reads is far larger than L2, so the
    # steps run back to back without flushes.
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]

    def pipelined(n, start_ev):
        h2d_stream.wait_event(start_ev)
        for i in range(n):
            s_ = i % 2
            if i >= 2:   # this buffer set was last used by step i-2
                h2d_stream.wait_event(ev_done[s_])
            with torch.cuda.stream(h2d_stream):
                d_sets[s_].copy_(h_buf, non_blocking=True)
            ev_in[s_].record(h2d_stream)
            stream.wait_event(ev_in[s_])
            if i >= 2:
                stream.wait_event(ev_read[s_])
            q_, kn_, vn_, tab_, len_ = d_views[s_]
            layer.fused_step(q=q_, k_new=kn_, v_new=vn_, out=outs[s_], num_splits=args.splits,
                             tables=tab_, lens=len_, stream=stream)
            ev_done[s_].record(stream)
            d2h_stream.wait_event(ev_done[s_])
            with torch.cuda.stream(d2h_stream):
                h_outs[s_].copy_(outs[s_], non_blocking=True)
            ev_read[s_].record(d2h_stream)
        stream.wait_event(ev_read[(n - 1) % 2])

    w0 = torch.cuda.Event()
    w0.record(stream)
    pipelined(max(args.warmup, 2), w0)
    torch.cuda.synchronize()
    if bn.dist:
        bn.dist.barrier()
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    pipelined(K, p0)
    p1.record(stream)
    torch.cuda.synchronize()
    # the last step's output as read back on the host equals the step's result
    assert torch.equal(h_outs[(K - 1) % 2].view(torch.int16), outs[(K - 1) % 2].cpu().view(torch.int16))
    t_pipe = max_over_ranks(p0.elapsed_time(p1) / 1e3, bn.dist, dev)
    e2e = {"value": round(world * alg * K / t_pipe / 1e9, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "us_per_step": 1e6 * t_pipe / K,
           "how": "pa_decode_step through the Python API; each step copies its inputs in from pinned host memory "
                  "and its output back, the copies on one stream per direction overlapping the neighbouring steps"}
    serial = {"value": round(world * alg * K / t_serial / 1e9, 2), "unit": UNIT, "us_per_step": 1e6 * t_serial / K,
              "how": "copy in, step, copy out back to back; L2 flushed between steps"}
    return e2e, serial


def measure_workload(bn, name, world, local, sweep=None, cuda_core=False, shared=False):
    """Build one workload, check its step against the oracle on every output,
    then time it.  Returns the workload's entry of the JSON line."""
    import oracle.run
    from paged_kv_cache_294_gb300.engine import PagedDecodeLayer
    import paged_kv_cache_294_gb300 as pa
    args, dev = bn.args, bn.dev
    K = args.steps
    w = workloads.make(name, device=dev, B=args.batch)
    layer = PagedDecodeLayer.from_workload(w, dev)
    S = layer.num_splits(args.splits)
    layer.ensure_workspace(args.splits)
    alg, kv_bytes, qo_bytes = algorithmic_bytes(w)
    uniq = unique_kv_bytes(w, layer.tables_host)

    # parity before timing: the timed launch (pa_decode_step, this split plan)
    # against the oracle on every output of every sequence
    layer.out.fill_(float("nan"))   # a row the launch does not write fails the check
    pa.pa_get_device_error(clear=True)
    layer.fused_step(num_splits=args.splits)
    torch.cuda.synchronize()
    flags = pa.pa_get_device_error()
    st = oracle.run.OracleStep(w, tables=layer.tables_host)
    st.append()
    ref = st.decode(threads=os.cpu_count() or 1)
    parity = parity_full(w, layer.out, ref, flags)
    if not parity["ok"]:
        print("parity check failed on %s: %s flags=%#x" % (name, parity, flags), file=sys.stderr)
        sys.exit(3)

    # every step does identical work: re-appending the same token to the same slot
    # rewrites identical bytes (bf16) and keeps a coded block's scale
    with ClockSampler(local) as clocks:
        t_step = bn.timed(lambda: layer.fused_step(num_splits=args.splits), K)
        step_stats = bn.step_stats()
        t_two = bn.timed(lambda: (layer.append_step(), layer.decode(num_splits=args.splits)), K)
        t_attn = bn.timed(lambda: layer.decode(num_splits=args.splits), K)
        e2e, e2e_serial = e2e_measure(bn, layer, K, world, alg)
    bn.clock_lines.extend(clocks.lines)
    peak, peak_kind = hbm_peak()
    dec_gbs = (uniq + qo_bytes) * K / t_step / 1e9
    value = world * alg * K / t_step / 1e9
    traffic = ncu_traffic(name, S) if args.batch is None else None
    entry = {
        "value": round(value, 2), "unit": UNIT, "ms_per_step": 1e3 * t_step / K, "us_per_step": 1e6 * t_step / K,
        "seq_steps_per_s": world * w.B * K / t_step, "step_time": step_stats,
        "config": {"workload": name if args.batch is None else "%s-B%d" % (name, w.B), "desc": w.desc,
                   "batch": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.d, "block_size": w.bs, "kv": w.kv,
                   "num_splits": S, "tokens": int(np.sum(w.seq_lens)),
                   "parallelism": "replicas" if world > 1 else "1 gpu",
                   "l2": "512 MiB write+read between timed steps (untimed); step reads > L2"},
        "dtype": {"fp8": "fp8_e4m3-cache/f16-mma/f32-softmax", "int8": "int8-cache/f16-mma/f32-softmax",
                  "int4": "int4-cache/f16-mma/f32-softmax"}.get(w.kv, "bf16-cache/bf16-mma/f32-softmax"),
        "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(dec_gbs / peak, 4), "traffic": traffic, "peak_source": peak_kind,
                     "kernel": "paged_decode_kernel via pa_decode_step (append + attention + split-K merge, "
                               "one launch)"},
        "bytes_per_step": {"algorithmic_logical": alg, "kv_logical": kv_bytes, "q_out": qo_bytes,
                           "kv_distinct": uniq},
        "two_launch_step": {"GBps": alg * K / t_two / 1e9, "us": 1e6 * t_two / K,
                            "calls": "pa_kv_append + pa_decode_attention"},
        "attention_only": {"GBps": alg * K / t_attn / 1e9, "us": 1e6 * t_attn / K,
                           "calls": "pa_decode_attention"},
        "e2e": e2e, "e2e_serial": e2e_serial, "parity": parity, "clocks": clocks.summary(),
        "gpu_launches": K,
    }
    if sweep:
        # split-K partition counts (explicit), each checked against the same oracle output
        rows = []
        with ClockSampler(local) as sclocks:
            for Sx in sweep:
                layer.out.fill_(float("nan"))   # a row the launch does not write fails the check
                pa.pa_get_device_error(clear=True)
                layer.fused_step(num_splits=Sx)
                torch.cuda.synchronize()
                par = parity_full(w, layer.out, ref, pa.pa_get_device_error())
                if not par["ok"]:
                    print("parity check failed on %s S=%d: %s" % (name, Sx, par), file=sys.stderr)
                    sys.exit(3)
                t = bn.timed(lambda: layer.fused_step(num_splits=Sx), K)
                g = (uniq + qo_bytes) * K / t / 1e9
                rows.append({"splits": layer.num_splits(Sx), "us": 1e6 * t / K, "GBps": round(g, 1),
                             "frac": round(g / peak, 4), "max_err_over_bound": par["max_err_over_bound"]})
        bn.clock_lines.extend(sclocks.lines)
        rows.append({"splits": "auto (%d)" % S, "us": entry["us_per_step"], "GBps": entry["roofline"]["achieved"],
                     "frac": entry["roofline"]["frac"], "max_err_over_bound": parity["max_err_over_bound"]})
        entry["split_sweep"] = rows
    if cuda_core:
        # the same kernel with its CUDA-core page step (packed fp32 FMAs) in place
        # of the tensor-core MMAs: parity first, then the same timings
        os.environ["PA_DECODE_FMA"] = "1"
        try:
            layer.out.fill_(float("nan"))   # a row the launch does not write fails the check
            pa.pa_get_device_error(clear=True)
            layer.fused_step(num_splits=args.splits)
            torch.cuda.synchronize()
            par = parity_full(w, layer.out, ref, pa.pa_get_device_error())
            if not par["ok"]:
                print("parity check failed on %s (CUDA-core step): %s" % (name, par), file=sys.stderr)
                sys.exit(3)
            with ClockSampler(local) as fclocks:
                tf_step = bn.timed(lambda: layer.fused_step(num_splits=args.splits), K)
                tf_attn = bn.timed(lambda: layer.decode(num_splits=args.splits), K)
            bn.clock_lines.extend(fclocks.lines)
        finally:
            del os.environ["PA_DECODE_FMA"]
        g = (uniq + qo_bytes) * K / tf_step / 1e9
        entry["cuda_core_variant"] = {
            "what": "PA_DECODE_FMA=1: the page step's Q.K^T and P.V as packed fp32 FMAs on the CUDA cores "
                    "instead of m16n8k16 MMAs; same kernel otherwise",
            "step_us": 1e6 * tf_step / K, "step_GBps": round(g, 1), "frac": round(g / peak, 4),
            "attention_only_us": 1e6 * tf_attn / K,
            "tensor_core_step_us": entry["us_per_step"], "tensor_core_attention_only_us": entry["attention_only"]["us"],
            "parity": par}
    if shared:
        # the step through pa_decode_step_shared: the blocks several sequences
        # share are read once per chunk of 8 / G of them (plan: pa_share_plan)
        plan = layer.plan_sharing()
        pa.pa_get_device_error(clear=True)
        layer.out.fill_(float("nan"))   # a row the launch does not write fails the check
        layer.shared_step(num_splits=args.splits)
        torch.cuda.synchronize()
        par = parity_full(w, layer.out, ref, pa.pa_get_device_error())
        if not par["ok"]:
            print("parity check failed on %s (shared prefixes): %s" % (name, par), file=sys.stderr)
            sys.exit(3)
        with ClockSampler(local) as sclocks:
            ts_step = bn.timed(lambda: layer.shared_step(num_splits=args.splits), K)
            ts_attn = bn.timed(lambda: layer.shared_step(append=False, num_splits=args.splits), K)
        bn.clock_lines.extend(sclocks.lines)
        g = (uniq + qo_bytes) * K / ts_step / 1e9
        entry["shared_prefix_step"] = {
            "calls": "pa_share_plan (host) + pa_decode_step_shared (one launch)",
            "chunks": len(plan["chunk_blocks"]), "shared_blocks": plan["max_chunk_blocks"],
            "sequences_sharing": int((plan["chunk_of"] >= 0).sum()),
            "us_per_step": 1e6 * ts_step / K, "value": round(world * alg * K / ts_step / 1e9, 2), "unit": UNIT,
            "seq_steps_per_s": world * w.B * K / ts_step, "attention_only_us": 1e6 * ts_attn / K,
            "roofline": {"bound": "hbm", "achieved": round(g, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(g / peak, 4), "peak_source": peak_kind, "bytes": "distinct K/V + q + out"},
            "parity": par}
    cpu = None
    if name == bn.headline and world == 1 and not args.no_cpu_baseline and bn.rank == 0:
        cpu = cpu_oracle_baseline(w, layer.tables_host, budget_s=args.cpu_seconds)
    del layer, st, ref
    torch.cuda.empty_cache()
    return entry, cpu


def measure_extras(bn):
    """Secondary measurements on the Llama-3-8B layer shape: block copies
    (copy-on-write), the host prefix cache, and multi-query attention
    (chunked prefill, speculative verify)."""
    import paged_kv_cache_294_gb300 as pa
    from paged_kv_cache_294_gb300.engine import BlockManager, PagedDecodeLayer
    args, dev, K = bn.args, bn.dev, bn.args.steps
    base = workloads.CONFIGS["8b"]
    Hkv, bs, d = base["Hkv"], base["bs"], base["d"]
    out = {}

    # copy-on-write block copies (pa_copy_blocks): 4096 random source blocks into
    # 4096 others of a separate pool
    nb_copy = 4096
    ck = torch.empty((2 * nb_copy, Hkv, bs, d), dtype=torch.bfloat16, device=dev)
    cv = torch.empty_like(ck)
    ck.view(torch.uint8).fill_(3)
    cv.view(torch.uint8).fill_(5)
    perm = torch.from_numpy(np.random.default_rng(1).permutation(2 * nb_copy).astype(np.int32)).to(dev)
    c_src, c_dst = perm[:nb_copy].contiguous(), perm[nb_copy:].contiguous()
    t_copy = bn.timed(lambda: pa.pa_copy_blocks(ck, cv, None, None, c_src, c_dst), K)
    copy_bytes = 2 * 2 * nb_copy * ck[0].numel() * ck.element_size()   # K and V, read + write
    copy_gbs = copy_bytes * K / t_copy / 1e9
    out["copy_blocks"] = {"GBps": round(copy_gbs, 1), "frac": round(copy_gbs / hbm_peak()[0], 4),
                          "us": 1e6 * t_copy / K, "blocks": nb_copy, "bytes": copy_bytes,
                          "calls": "pa_copy_blocks (copy-on-write of whole K/V pages, 8b layer shape)"}
    del ck, cv

    # host prefix cache through BlockManager: 1000 requests, each one of 8 system
    # prompts of 2304 tokens plus its own U[1, 512] tokens; admit, commit, free
    prng = np.random.default_rng(11)
    prompts = [[int(x) for x in prng.integers(0, 32000, 2304)] for _ in range(8)]
    reqs = [np.array(prompts[int(prng.integers(0, 8))] +
                     [int(x) for x in prng.integers(32000, 64000, int(prng.integers(1, 513)))], dtype=np.int32)
            for _ in range(1000)]
    mgr = BlockManager(base["num_blocks"], bs)
    reused = 0
    t0 = time.perf_counter()
    for i, toks in enumerate(reqs):
        reused += mgr.add(i, toks)
        mgr.commit(i)
        mgr.free(i)
    t_host = time.perf_counter() - t0
    out["prefix_cache_host"] = {"requests": len(reqs), "us_per_request": 1e6 * t_host / len(reqs),
                                "reused_token_fraction": reused / sum(len(t) for t in reqs),
                                "calls": "BlockManager.add (pa_seq_admit), commit (pa_prefix_insert), free"}

    # multi-query attention (pa_prefill_attention): a chunked-prefill batch (16
    # sequences, 2048 cached + a 2048-token chunk) and a speculative-verify batch
    # (64 sequences, 4 proposals + 1, U[128, 4096] cached), 8b and 70b layers on
    # the bf16 cache, the 8b layer on the int8 and int4 caches
    mq = {}
    rng = np.random.default_rng(7)
    cases = {"prefill": ([2048] * 16, [2048] * 16),
             "verify": ([int(x) for x in rng.integers(128, 4097, 64)], [5] * 64)}
    for layer_name in args.mq_layers.split(","):
        for case, (ctx, chunk) in cases.items():
            pw = workloads.make_prefill(layer_name, ctx, chunk, seed=31, device=dev)
            pl = PagedDecodeLayer.from_workload(pw, dev)
            pq = pw.q_chunk.to(dev)
            po = torch.empty_like(pq)
            pqs = torch.from_numpy(pw.q_start).to(dev)
            fn = lambda: pa.pa_prefill_attention(po, pq, pl.k_cache, pl.v_cache, pl.k_scale, pl.v_scale,
                                                 pl.block_tables, pl.seq_lens, pqs, pw.max_q, pw.scale)
            pa.pa_get_device_error(clear=True)
            t_p = bn.timed(fn, K)
            flops = prefill_flops(pw)
            kvb = int(np.sum(pw.seq_lens.astype(np.int64))) * 2 * pw.Hkv * row_bytes(pw) + 2 * pq.numel() * 2
            e = {"layer": layer_name, "kv": pw.kv, "sequences": pw.B,
                 "cached": "2048" if case == "prefill" else "U[128,4096]", "chunk": chunk[0],
                 "us": 1e6 * t_p / K, "TFLOPs": flops * K / t_p / 1e12, "kv_GBps": kvb * K / t_p / 1e9,
                 "flops": flops, "kv_bytes": kvb, "device_error": pa.pa_get_device_error()}
            if case == "prefill":
                pk, pk_kind = bf16_peak()
                e["bound"], e["frac"] = "tensor", round(e["TFLOPs"] / pk, 4)
                e["peak"] = "%s bf16 %.1f TFLOP/s" % (pk_kind, pk)
            else:
                e["bound"], e["frac"] = "hbm", round(e["kv_GBps"] / hbm_peak()[0], 4)
                e["peak"] = "%s HBM %.1f GB/s" % hbm_peak()[::-1]
            mq["%s_%s" % (case, layer_name)] = e
            del pl, pq, po
            torch.cuda.empty_cache()
    out["multi_query_attention"] = mq
    return out


def run_ours(args):
    import paged_kv_cache_294_gb300 as pa

    dist, rank, world = dist_init()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.load()
    bn = Bench(args, dev, dist)
    bn.rank = rank
    names = ALL_WORKLOADS if args.workload == "all" else (args.workload,)
    if args.extras_only:
        names = ()
    bn.headline = HEADLINE if args.workload == "all" else args.workload
    entries, cpu = {}, None
    wall0 = time.perf_counter()
    for name in names:
        sweep = SPLIT_SWEEP if (name == "long" and args.workload == "all" and args.batch is None) else None
        if args.sweep_splits:
            sweep = tuple(int(x) for x in args.sweep_splits.split(","))
        cuda_core = name in ("8b", "70b") and args.workload == "all" and args.batch is None
        entries[name], c = measure_workload(bn, name, world, local, sweep, cuda_core, shared=name == "fp8prefix")
        cpu = c or cpu
    extras = measure_extras(bn) if not args.no_extras else {}
    wall = time.perf_counter() - wall0
    if rank != 0:
        return
    if args.extras_only:
        print(json.dumps(dict(extras, wall_s=wall, note="secondary measurements only (--extras-only)")))
        return
    h = entries[bn.headline]
    peak, peak_kind = hbm_peak()
    line = {
        "metric": METRIC, "value": h["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": h["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": h["dtype"], "data": "synthetic",
        "config": h["config"], "seq_steps_per_s": h["seq_steps_per_s"],
        "hbm_frac_of_%s" % peak_kind: (h["value"] / world) / peak,
        "us_per_step": h["us_per_step"], "roofline": h["roofline"], "e2e": h["e2e"], "e2e_serial": h["e2e_serial"],
        "two_launch_step": h["two_launch_step"], "attention_only": h["attention_only"],
        "bytes_per_step": h["bytes_per_step"], "parity": h["parity"],
        "gpu_launches": h["gpu_launches"],
        "clocks": clock_summary(bn.clock_lines),
        "workloads": entries,
        "wall_s": wall,
    }
    if "long" in entries and "split_sweep" in entries["long"]:
        line["long_split_sweep"] = entries["long"]["split_sweep"]
    line.update(extras)
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="all", choices=["all"] + sorted(workloads.CONFIGS))
    ap.add_argument("--splits", type=int, default=0, help="split-K partitions (0 = automatic)")
    ap.add_argument("--batch", type=int, default=None,
                    help="fewer sequences of the same workload recipe (profiling cases); default: full")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the secondary measurements (block copy, host prefix cache, multi-query attention)")
    ap.add_argument("--extras-only", action="store_true",
                    help="only the secondary measurements (profiling their kernels)")
    ap.add_argument("--sweep-splits", default="",
                    help="comma-separated split counts to time (each parity-checked) on every workload run")
    ap.add_argument("--mq-layers", default="8b,70b,8b-int8,8b-int4",
                    help="layer shapes (workload names) of the multi-query attention measurements")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.batch is not None and args.workload == "all":
        ap.error("--batch needs one --workload")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
