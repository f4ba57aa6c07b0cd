"""Benchmark: paged decode attention on one GB300 (or N independent replicas).

A step is one decode iteration of one attention layer over the whole batch:
pa_kv_append of every sequence's new token, then pa_decode_attention (and its
split-K merge when the plan has more than one partition).  The metric is the
KV-read bandwidth of that step, counted from the algorithmic bytes (K/V of
every cached token read once, q read, out written) and also reported as
sequence-steps per second and as a fraction of the measured HBM peak.

    python bench.py [--workload 8b|70b|long|fp8prefix] [--steps K] [--warmup W]
                    [--splits S] [--impl ours|reference] [--gpus N]

Prints one JSON line (rank 0).  With torchrun (N > 1) every rank runs an
independent replica of the workload on its own GPU (the path has no exchange
step); value = all ranks' bytes / the slowest rank's time.
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


def cpu_oracle_baseline(w, tables, budget_s=10.0, threads=None):
    """The fp64 oracle's step (append of the new token + decode attention) on a bounded
    sample of the batch, repeated until ~budget_s of wall time.  Returns dict."""
    import oracle.run
    threads = threads or os.cpu_count() or 1
    rng = np.random.default_rng(0)
    order = rng.permutation(w.B)
    # grow the sample until one oracle step takes ~1/5 of the budget
    n = min(w.B, max(1, threads))
    while True:
        seqs = sorted(order[:n].tolist())
        st = oracle.run.OracleStep(w, seqs=seqs, tables=tables)
        t0 = time.perf_counter()
        st.append()
        st.decode(threads=threads)
        dt = time.perf_counter() - t0
        if dt > budget_s / 5 or n >= w.B:
            break
        n = min(w.B, n * 2)
    reps, total = 1, dt
    while total < budget_s and reps < 500:
        # re-appending the same token rewrites the same cache bytes: every rep is the same step
        t0 = time.perf_counter()
        st.append()
        st.decode(threads=threads)
        total += time.perf_counter() - t0
        reps += 1
    lens = np.asarray(w.seq_lens, dtype=np.int64)[seqs]
    byts = int(lens.sum()) * 2 * w.Hkv * row_bytes(w) + 2 * len(seqs) * w.Hq * w.d * 2
    per_step = total / reps
    return {"value": byts / per_step / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "%d of %d sequences (%d tokens), fp64 C oracle append+decode, %d reps, %.1f s" %
                      (len(seqs), w.B, int(lens.sum()), reps, total),
            "seq_steps_per_s": len(seqs) / per_step}


def run_reference(args):
    """The oracle arm: the fp64 CPU oracle timed on the host cores, rank 0 only."""
    dist, rank, world = dist_init()
    if rank != 0:
        return
    w = workloads.make(args.workload, device="cpu", B=args.batch)
    import oracle.run
    tables = oracle.run.tables_of(w)
    threads = os.cpu_count() or 1
    # per step: a bounded sample of the batch sized for ~2 s of CPU work
    rng = np.random.default_rng(1)
    n = max(1, min(w.B, threads))
    seqs = sorted(rng.permutation(w.B)[:n].tolist())
    times = []
    st = oracle.run.OracleStep(w, seqs=seqs, tables=tables)
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        st.append()
        st.decode(threads=threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    lens = np.asarray(w.seq_lens, dtype=np.int64)[seqs]
    byts = int(lens.sum()) * 2 * w.Hkv * row_bytes(w) + 2 * len(seqs) * w.Hq * w.d * 2
    t = sum(times)
    value = byts * len(times) / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "seq_steps_per_s": len(seqs) * len(times) / t,
            "config": {"workload": args.workload, "desc": w.desc, "sample_sequences": len(seqs)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": "%d of %d sequences per step, fp64 C oracle append+decode" %
                                       (len(seqs), w.B)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_ours(args):
    import paged_kv_cache_294_gb300 as pa
    from paged_kv_cache_294_gb300.engine import PagedDecodeLayer
    import oracle.run

    dist, rank, world = dist_init()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.load()

    w = workloads.make(args.workload, device=dev, B=args.batch)
    layer = PagedDecodeLayer.from_workload(w, dev)
    S = layer.num_splits(args.splits)
    layer.ensure_workspace(args.splits)
    alg, kv_bytes, qo_bytes = algorithmic_bytes(w)
    uniq = unique_kv_bytes(w, layer.tables_host)

    # parity once, before timing: the step's output on sampled sequences vs the oracle
    pa.pa_get_device_error(clear=True)
    layer.step(num_splits=args.splits)
    torch.cuda.synchronize()
    flags = pa.pa_get_device_error()
    sample = sorted({0, w.B - 1, w.B // 2})
    st = oracle.run.OracleStep(w, seqs=sample, tables=layer.tables_host)
    st.append()
    ref = st.decode(threads=os.cpu_count() or 1)
    err = float(np.max(np.abs(layer.out.float().cpu().numpy()[sample] - ref)))
    tol = {"fp8": 5e-2, "int8": 1e-2, "int4": 1e-2}.get(w.kv, 1e-2)
    parity = {"max_abs_err": err, "tol": tol, "sequences": sample, "ok": bool(err <= tol and flags == 0)}
    if not parity["ok"]:
        print("parity check failed: %s flags=%#x" % (parity, flags), file=sys.stderr)
        sys.exit(3)

    # the cache must hold exactly the history before each timed append: re-running the
    # append of the same token to the same slot rewrites identical bytes (bf16) and, for
    # fp8, keeps the block scale (max(old, same absmax)) -- every step does identical work.
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)   # > 2 x L2
    stream = torch.cuda.current_stream(dev)
    launches_per_step = 1   # pa_decode_step: append, attention and split-K merge in one kernel

    def flush_l2():
        # write then read 512 MiB: evicts the previous step's lines and leaves no dirty
        # lines whose write-back would overlap the timed region
        flush.fill_(1)
        flush.sum(dtype=torch.int32)

    def timed(fn, K, sampler=None):
        """Per-step CUDA-event time (s, summed over K steps), L2 flushed before each (untimed)."""
        for _ in range(args.warmup):
            flush_l2()
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(K):
            flush_l2()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t = sum(x.elapsed_time(y) for x, y in ev) / 1e3
        return max_over_ranks(t, dist, dev)

    K = args.steps
    # the step: pa_decode_step (append of every new token + attention, one launch)
    wall0 = time.perf_counter()
    with ClockSampler(local) as clocks:
        t_step = timed(lambda: layer.fused_step(num_splits=args.splits), K)
    wall = time.perf_counter() - wall0
    # the same step as two launches (pa_kv_append, then pa_decode_attention)
    t_two = timed(lambda: (layer.append_step(), layer.decode(num_splits=args.splits)), K)
    # pa_decode_attention alone
    t_attn = timed(lambda: layer.decode(num_splits=args.splits), K)
    value = world * alg * K / t_step / 1e9
    # roofline of the step's only kernel: distinct KV bytes (a shared prefix once) + q + out
    dec_gbs = (uniq + qo_bytes) * K / t_step / 1e9
    peak, peak_kind = hbm_peak()

    # end to end through the public API with host buffers: the step's inputs (q,
    # new K/V, slots, tables, lengths) packed in one pinned buffer and copied
    # host->device in one transfer, append + decode, the output copied back,
    # all inside the timed region
    parts = [layer.q, layer.k_new, layer.v_new, layer.step_slots, layer.block_tables, layer.seq_lens]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, i):
        t = parts[i]
        n = t.numel() * t.element_size()
        return buf[offs[i]:offs[i] + n].view(t.dtype).view(t.shape)

    for i, t in enumerate(parts):
        view(h_buf, i).copy_(t.cpu())
    d_q, d_kn, d_vn, d_slots, d_tab, d_len = (view(d_buf, i) for i in range(len(parts)))
    h_out = torch.empty(tuple(layer.out.shape), dtype=torch.bfloat16).pin_memory()
    h2d = total
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_buf.copy_(h_buf, non_blocking=True)
        layer.fused_step(q=d_q, k_new=d_kn, v_new=d_vn, num_splits=args.splits, tables=d_tab, lens=d_len)
        h_out.copy_(layer.out, non_blocking=True)

    t_e2e_serial = timed(e2e_step, K)
    e2e_serial = world * alg * K / t_e2e_serial / 1e9

    # the same steps as a serving loop issues them: two sets of device buffers, one
    # stream per copy direction, so step i+1's input copy and step i-1's output
    # copy run while step i's kernel runs.  Every step still copies its inputs in
    # from pinned host memory and its output back, all inside the timed region
    # (which ends when the last output has reached the host).  The cache the step
    # reads (hundreds of MB) is far larger than L2, so steps run back to back
    # without flushes.
    e2e_how = ("pa_decode_step through the Python API; each step copies its inputs in from pinned host memory "
               "and its output back, the copies on one stream per direction overlapping the neighbouring steps")
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    d_sets = [d_buf, torch.empty(total, dtype=torch.uint8, device=dev)]
    d_views = [[view(buf, i) for i in range(len(parts))] for buf in d_sets]
    outs = [torch.empty_like(layer.out) for _ in range(2)]
    h_outs = [h_out, torch.empty_like(h_out).pin_memory()]
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
            q_, kn_, vn_, _, tab_, len_ = d_views[s_]
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
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    pipelined(K, p0)
    p1.record(stream)
    torch.cuda.synchronize()
    # the last step's output as read back on the host equals the step's result
    assert torch.equal(h_outs[(K - 1) % 2].view(torch.int16), outs[(K - 1) % 2].cpu().view(torch.int16))
    t_e2e = max_over_ranks(p0.elapsed_time(p1) / 1e3, dist, dev)
    e2e_value = world * alg * K / t_e2e / 1e9

    # copy-on-write block copies (pa_copy_blocks) on this layer's page shape:
    # 4096 random source blocks into 4096 others of a separate pool
    nb_copy = 4096
    ck = torch.empty((2 * nb_copy,) + tuple(layer.k_cache.shape[1:]), dtype=layer.k_cache.dtype, device=dev)
    cv = torch.empty_like(ck)
    ck.view(torch.uint8).fill_(3)
    cv.view(torch.uint8).fill_(5)
    cks = torch.ones((2 * nb_copy, w.Hkv), dtype=torch.float32, device=dev) if w.kv != "bf16" else None
    cvs = torch.ones_like(cks) if cks is not None else None
    perm = torch.from_numpy(np.random.default_rng(1).permutation(2 * nb_copy).astype(np.int32)).to(dev)
    c_src, c_dst = perm[:nb_copy].contiguous(), perm[nb_copy:].contiguous()
    t_copy = timed(lambda: pa.pa_copy_blocks(ck, cv, cks, cvs, c_src, c_dst,
                                             kv_dtype=pa.PA_KV_INT4 if w.kv == "int4" else None), K)
    page = ck[0].numel() * ck.element_size()
    copy_bytes = 2 * 2 * nb_copy * (page + (4 * w.Hkv if cks is not None else 0))   # K and V, read + write
    copy_gbs = copy_bytes * K / t_copy / 1e9
    del ck, cv, cks, cvs

    # host prefix cache (pa_prefix_match + pa_prefix_insert through BlockManager):
    # 1000 requests, each one of 8 system prompts of 2304 tokens plus its own
    # U[1, 512] tokens; admit (match + allocate), commit (insert), free
    prefix = None
    if not args.no_extras:
        from paged_kv_cache_294_gb300.engine import BlockManager
        prng = np.random.default_rng(11)
        prompts = [[int(x) for x in prng.integers(0, 32000, 2304)] for _ in range(8)]
        reqs = [np.array(prompts[int(prng.integers(0, 8))] +
                         [int(x) for x in prng.integers(32000, 64000, int(prng.integers(1, 513)))], dtype=np.int32)
                for _ in range(1000)]
        mgr = BlockManager(w.num_blocks, w.bs)
        reused = 0
        t0 = time.perf_counter()
        for i, toks in enumerate(reqs):
            reused += mgr.add(i, toks)
            mgr.commit(i)
            mgr.free(i)
        t_host = time.perf_counter() - t0
        prefix = {"requests": len(reqs), "us_per_request": 1e6 * t_host / len(reqs),
                  "reused_token_fraction": reused / sum(len(t) for t in reqs),
                  "calls": "BlockManager.add (pa_prefix_match + pa_block_alloc), commit (pa_prefix_insert), free"}

    # multi-query attention (pa_prefill_attention) on this workload's layer shape:
    # a chunked-prefill batch (16 sequences, 2048 cached + a 2048-token chunk) and
    # a speculative-verify batch (64 sequences, 4 proposals + 1, U[128, 4096] cached)
    extras = {}
    if not args.no_extras and w.kv == "bf16" and w.d == 128:
        base = args.workload if args.workload in ("8b", "70b", "long") else "8b"
        rng = np.random.default_rng(7)
        cases = {"prefill": ([2048] * 16, [2048] * 16),
                 "verify": ([int(x) for x in rng.integers(128, 4097, 64)], [5] * 64)}
        for name, (ctx, chunk) in cases.items():
            pw = workloads.make_prefill(base, ctx, chunk, seed=31, device=dev)
            pl = PagedDecodeLayer.from_workload(pw, dev)
            pq = pw.q_chunk.to(dev)
            po = torch.empty_like(pq)
            pqs = torch.from_numpy(pw.q_start).to(dev)
            fn = lambda: pa.pa_prefill_attention(po, pq, pl.k_cache, pl.v_cache, None, None, pl.block_tables,
                                                 pl.seq_lens, pqs, pw.max_q, pw.scale)
            pa.pa_get_device_error(clear=True)
            t_p = timed(fn, K)
            flops = prefill_flops(pw)
            kvb = int(np.sum(pw.seq_lens.astype(np.int64))) * 2 * pw.Hkv * pw.d * 2 + 2 * pq.numel() * 2
            e = {"layer": base, "sequences": pw.B, "cached": "%s" % ("2048" if name == "prefill" else "U[128,4096]"),
                 "chunk": chunk[0], "us": 1e6 * t_p / K, "TFLOPs": flops * K / t_p / 1e12,
                 "kv_GBps": kvb * K / t_p / 1e9, "flops": flops, "kv_bytes": kvb,
                 "device_error": pa.pa_get_device_error()}
            if name == "prefill":
                pk, pk_kind = bf16_peak()
                e["bound"], e["frac"] = "tensor", round(e["TFLOPs"] / pk, 4)
                e["peak"] = "%s bf16 %.1f TFLOP/s" % (pk_kind, pk)
            else:
                e["bound"], e["frac"] = "hbm", round(e["kv_GBps"] / hbm_peak()[0], 4)
                e["peak"] = "%s HBM %.1f GB/s" % hbm_peak()[::-1]
            extras[name] = e
            del pl, pq, po

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_baseline(w, layer.tables_host, budget_s=args.cpu_seconds)
    clk = clocks.summary()
    traffic = ncu_traffic(args.workload, S) if args.batch is None else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_step / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp8": "fp8_e4m3-cache/f16-mma/f32-softmax",
                  "int8": "int8-cache/f16-mma/f32-softmax",
                  "int4": "int4-cache/f16-mma/f32-softmax"}.get(w.kv, "bf16-cache/bf16-mma/f32-softmax"),
        "data": "synthetic",
        "config": {"workload": args.workload if args.batch is None else "%s-B%d" % (args.workload, w.B),
                   "desc": w.desc, "batch": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                   "head_dim": w.d, "block_size": w.bs, "kv": w.kv, "num_splits": S,
                   "tokens": int(np.sum(w.seq_lens)), "parallelism": "replicas" if world > 1 else "1 gpu",
                   "l2": "512 MiB write+read between timed steps (untimed); step reads > L2"},
        "seq_steps_per_s": world * w.B * K / t_step,
        "hbm_frac_of_%s" % peak_kind: (value / world) / peak,
        "us_per_step": 1e6 * t_step / K,
        "two_launch_step": {"GBps": alg * K / t_two / 1e9, "us": 1e6 * t_two / K,
                            "calls": "pa_kv_append + pa_decode_attention"},
        "attention_only": {"GBps": alg * K / t_attn / 1e9, "us": 1e6 * t_attn / K,
                           "calls": "pa_decode_attention"},
        "multi_query_attention": extras,
        "prefix_cache_host": prefix,
        "copy_blocks": {"GBps": round(copy_gbs, 1), "frac": round(copy_gbs / hbm_peak()[0], 4),
                        "us": 1e6 * t_copy / K, "blocks": nb_copy, "bytes": copy_bytes,
                        "calls": "pa_copy_blocks (copy-on-write of whole K/V pages)"},
        "bytes_per_step": {"algorithmic_logical": alg, "kv_logical": kv_bytes, "q_out": qo_bytes,
                           "kv_distinct": uniq},
        "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(dec_gbs / peak, 4), "traffic": traffic,
                     "peak_source": peak_kind, "kernel": "paged_decode_kernel via pa_decode_step (append + attention + split-K merge, one launch)"},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_step": 1e6 * t_e2e / K,
                "how": e2e_how},
        "e2e_serial": {"value": round(e2e_serial, 2), "unit": UNIT, "us_per_step": 1e6 * t_e2e_serial / K,
                       "how": "copy in, step, copy out back to back; L2 flushed between steps"},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "parity": parity,
        "wall_s_timed_region": wall,
    }
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="8b", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--splits", type=int, default=0, help="split-K partitions (0 = automatic)")
    ap.add_argument("--batch", type=int, default=None,
                    help="fewer sequences of the same workload recipe (profiling cases); default: full")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the secondary measurements (block copy, prefill / verify attention)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
