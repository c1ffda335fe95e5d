"""Throughput of the QuantWM 2-bit KV-cache hot path on one GB300 (or N, as
independent replicas).

One step is one pass of the whole path over one chunk of a 12-head video
world-model cache (21 latent frames of 1,560 tokens held, 3-frame chunks):
  qwm_calibrate  (1,024 historical queries per head, PSAC rank 16)
  qwm_append     (4,680 new tokens: QSAC over 256 centroids, INT2, PSAC e)
  qwm_attend     (4,680 query rows over the 32,760 cached tokens)
after which the cache is rewound to its 6-chunk prefix (host bookkeeping),
so every step does the same work.  L2 is flushed between steps.

`value` is the attention algorithmic throughput of the whole step,
H (4 M N d + 2 M N r + 2 M d r) flops per step / step time, in TFLOP/s;
the kernel-only numbers (attend TFLOP/s and cache GB/s, append Mtokens/s)
are reported beside it.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same step on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_kv_cache_qwm_gb300 import synth  # noqa: E402

WORKLOAD = "bf16-h12-n32760"
METRIC = "qwm_attend TFLOP/s & cache GB/s (% roofline); qwm_append Mtokens/s"
L2_FLUSH_BYTES = 256 << 20   # twice the 129 MB L2


def profiled_traffic(summary, source):
    """DRAM bytes (read + write) per launch of the attention kernel from a
    committed ncu summary, when the summary records the sha256 of the kernel
    source it was captured on and that source is unchanged; else None."""
    try:
        with open(summary) as f:
            text = f.read()
        want = re.search(r"source sha256: ([0-9a-f]{64})", text).group(1)
        nbytes = float(re.search(r"dram bytes per launch: ([0-9.eE+]+)", text).group(1))
        with open(source, "rb") as f:
            have = hashlib.sha256(f.read()).hexdigest()
    except (OSError, AttributeError, ValueError):
        return None
    return nbytes if have == want else None


def attend_flops(H, M, N, d, r):
    return H * (4.0 * M * N * d + 2.0 * M * N * r + 2.0 * M * d * r)


def max_over_ranks(value: float, device) -> float:
    """The largest `value` over all ranks (the step time that bounds the job)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, world: int, max_ms: float) -> float:
    """Work of all replicas divided by the slowest rank's step time."""
    return world * flops_per_rank_step / (max_ms * 1e-3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while it runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# the CPU oracle, timed on a bounded sample (reference arm and cpu_baseline)
# --------------------------------------------------------------------------

def oracle_step_seconds(wl, sample_tokens=256, sample_rows=64, head=0):
    """Seconds the fp64 oracle needs for one whole step, extrapolated from one
    head: calibrate (whole), append of `sample_tokens` keys, attention of
    `sample_rows` query rows over the full cache.  Heads, tokens and rows are
    independent, so the work scales linearly in each."""
    from oracle import qwm_oracle as O
    H, d, r, C = wl.heads, wl.head_dim, wl.rank, wl.n_centroids
    kf = synth.kmeans_keys(wl, [head])[0]
    cent = synth.round_to_dtype(kf[synth.kmeans_init_rows(wl, head, kf.shape[1], C)], wl.dtype)
    qh = synth.hist_queries(wl, 0, [head])[0]
    t0 = time.perf_counter()
    s = O.sensitivity(qh).astype(np.float32)
    U, _, _ = O.psac_basis(qh, r)
    w = O.group_weights(s)
    t_cal = time.perf_counter() - t0
    # cache of the 6-chunk prefix (untimed set-up)
    segs = [O.append_head(synth.keys(wl, ch, [head])[0], synth.values(wl, ch, [head])[0], cent, w, U)
            for ch in range(wl.n_chunks - 1)]
    k = synth.keys(wl, wl.n_chunks - 1, [head])[0]
    v = synth.values(wl, wl.n_chunks - 1, [head])[0]
    t0 = time.perf_counter()
    O.append_head(k[:sample_tokens], v[:sample_tokens], cent, w, U)
    t_app = (time.perf_counter() - t0) * wl.chunk / sample_tokens
    segs.append(O.append_head(k, v, cent, w, U))
    q = synth.queries(wl, 0, [head], m=sample_rows)[0]
    t0 = time.perf_counter()
    O.attend_head(q, segs, {0: U}, 1.0 / np.sqrt(d))
    t_att = (time.perf_counter() - t0) * wl.n_query / sample_rows
    per_head = t_cal + t_app + t_att
    return per_head * H, {"calibrate_s": t_cal * H, "append_s": t_app * H, "attend_s": t_att * H}


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    wl = synth.workload(args.workload)
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_step_seconds(wl, sample_tokens=64, sample_rows=16)
    times = []
    for _ in range(args.steps):
        sec, parts = oracle_step_seconds(wl)
        times.append(sec)
    step = float(np.mean(times))
    N = wl.n_tokens
    value = attend_flops(wl.heads, wl.n_query, N, wl.head_dim, wl.rank) / step / 1e12
    sample = (f"1 of {wl.heads} heads: calibrate whole, append 256 of {wl.chunk} tokens, attention "
              f"of 64 of {wl.n_query} query rows over {N} tokens; scaled linearly (extrapolated)")
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "heads": wl.heads, "head_dim": wl.head_dim,
                       "cached_tokens": N, "query_rows": wl.n_query, "chunk": wl.chunk,
                       "n_centroids": wl.n_centroids, "rank": wl.rank},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "breakdown_s": parts}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------

def run_gpu(args):
    import torch
    import torch.distributed as dist
    from bit_kv_cache_qwm_gb300 import build as B
    B.build()
    from bit_kv_cache_qwm_gb300 import qwm

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    wl = synth.workload(args.workload)
    H, d, r, C = wl.heads, wl.head_dim, wl.rank, wl.n_centroids
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    n_prefix = wl.n_chunks - 1

    def T(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev, tdt)

    # inputs: every rank holds its own replica of the workload (weak scaling)
    kf = synth.kmeans_keys(wl)
    rows = np.stack([synth.kmeans_init_rows(wl, h, kf.shape[1], C) for h in range(H)]).astype(np.int32)
    tiles = wl.n_chunks * ((wl.chunk + 127) // 128)
    ctx = qwm.Qwm(H, d, r, C, dtype=wl.dtype, max_tokens=tiles * 128, max_versions=2,
                  max_hist=wl.n_hist, device=dev)
    # the centroids: 25 Lloyd iterations on the keys of frame 0, on the GPU
    cent = qwm.qwm_kmeans(T(kf), torch.from_numpy(rows).to(dev), C, iters=25)
    ctx.set_centroids(cent)
    ctx.set_attend_kernel({"auto": 0, "simt": 1, "mma": 2, "tc": 3, "tc2": 4}[args.kernel])
    qh = T(synth.hist_queries(wl, 0))
    ctx.calibrate(qh)
    for ch in range(n_prefix):
        ctx.append(T(synth.keys(wl, ch)), T(synth.values(wl, ch)))
    k_new, v_new = T(synth.keys(wl, n_prefix)), T(synth.values(wl, n_prefix))
    q = T(synth.queries(wl, 0))
    out = torch.empty_like(q)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    assert ctx.status() == 0, "device status bits after set-up"

    N = wl.n_tokens
    if args.only:
        # profiling mode: the cache holds the full workload, then only the named
        # call runs, --steps times (no timing, no JSON line)
        if args.only == "attend":
            ctx.append(k_new, v_new)
            for _ in range(args.steps):
                ctx.attend(q, out)
        elif args.only == "append":
            for _ in range(args.steps):
                ctx.append(k_new, v_new)
                ctx.rewind(n_prefix)
        else:
            for _ in range(args.steps):
                ctx.calibrate(qh)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        return
    flops = attend_flops(H, wl.n_query, N, d, r)
    cache_bytes = H * N * ctx.layout.bytes_per_token
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ctx.calibrate(qh)
        if ev is not None:
            ev[1].record(stream)
        ctx.append(k_new, v_new)
        if ev is not None:
            ev[2].record(stream)
        ctx.attend(q, out)
        if ev is not None:
            ev[3].record(stream)
        ctx.rewind(n_prefix)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            step(evs[i])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    st = ctx.status()
    cal = [e[0].elapsed_time(e[1]) for e in evs]
    app = [e[1].elapsed_time(e[2]) for e in evs]
    att = [e[2].elapsed_time(e[3]) for e in evs]
    stp = [e[0].elapsed_time(e[3]) for e in evs]
    ms_step = max_over_ranks(float(np.mean(stp)), dev)

    # end to end through the public API with host buffers (pinned): every
    # step's inputs go host -> device and its output comes back, all inside
    # the timed region.  The copies run on a second stream, double-buffered:
    # the inputs of step i+1 go up and the output of step i-1 comes back
    # while step i computes (the calls themselves stay in order on one stream)
    h_in = [x.cpu().pin_memory() for x in (qh, k_new, v_new, q)]
    h_out = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    d_in = [[torch.empty_like(x) for x in (qh, k_new, v_new, q)] for _ in range(2)]
    d_out = [torch.empty_like(out) for _ in range(2)]
    copy = torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in_ready", "in_free", "out_ready", "out_free")}

    def upload(i):
        b = i & 1
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(ev["in_free"][b])
            for dst, src in zip(d_in[b], h_in):
                dst.copy_(src, non_blocking=True)
            ev["in_ready"][b].record(copy)

    def pipelined(n):
        """n end-to-end steps; milliseconds per step."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        copy.wait_event(e0)
        upload(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                upload(i + 1)
            stream.wait_event(ev["in_ready"][b])
            if i >= 2:
                stream.wait_event(ev["out_free"][b])
            flush.zero_()
            d_qh, d_k, d_v, d_q = d_in[b]
            ctx.calibrate(d_qh)
            ctx.append(d_k, d_v)
            ctx.attend(d_q, d_out[b])
            ev["in_free"][b].record(stream)
            ev["out_ready"][b].record(stream)
            ctx.rewind(n_prefix)
            with torch.cuda.stream(copy):
                copy.wait_event(ev["out_ready"][b])
                h_out[b].copy_(d_out[b], non_blocking=True)
                ev["out_free"][b].record(copy)
        stream.wait_stream(copy)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / n

    if args.warmup > 0:
        pipelined(args.warmup)
    e2e_step = max_over_ranks(pipelined(args.steps), dev)
    # the last end-to-end output is the device-timed steps' output (same inputs)
    e2e_same = bool(torch.equal(h_out[(args.steps - 1) & 1], out.cpu()))
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = h_out[0].numel() * h_out[0].element_size()

    peaks = load_peaks()
    att_ms = float(np.mean(att))
    achieved = flops / (att_ms * 1e-3) / 1e12
    value = whole_job_tflops(flops, world, ms_step)
    kernel = {0: "auto", 1: "simt", 2: "mma", 3: "tcgen05", 4: "tcgen05-2tile"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "heads": H, "head_dim": d, "cached_tokens": N,
                   "query_rows": wl.n_query, "chunk": wl.chunk, "n_centroids": C, "rank": r,
                   "hist_queries": wl.n_hist, "parallelism": f"replicas x{world}",
                   "l2": "flushed between steps (256 MiB write)",
                   "centroids": "k-means on frame 0 (25 Lloyd iterations, GPU)"},
        "components": {"calibrate_ms": float(np.mean(cal)), "append_ms": float(np.mean(app)),
                       "attend_ms": att_ms, "attend_tflops": achieved,
                       "cache_gbs": cache_bytes / (att_ms * 1e-3) / 1e9,
                       "append_mtok_s": wl.chunk / (float(np.mean(app)) * 1e-3) / 1e6,
                       "append_gbs": H * wl.chunk * (4 * d + ctx.layout.bytes_per_token) / (float(np.mean(app)) * 1e-3) / 1e9,
                       "attend_kernel": kernel.get(ctx.resolved_attend_kernel, "?")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"],
                     "traffic": profiled_traffic(os.path.join(ROOT, "profiles", f"attend_tc2_{wl.name}.md"),
                                                 os.path.join(ROOT, "bit_kv_cache_qwm_gb300", "csrc", "attend_tc.cu"))
                     if ctx.resolved_attend_kernel == 4 else None,
                     "kernel": "qwm_attend", "peak_source": peaks["source"] + " burst bf16"},
        "e2e": {"value": world * flops / (e2e_step * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_step,
                "copies": "second stream, double-buffered: inputs of step i+1 and output of step i-1 "
                          "move while step i computes", "output_matches_device_timed": e2e_same},
        # gram, gram sum, A^2, eig, weights, append, attend (A^2 only when r > 0)
        # gram, gram_sum, [square], eig, weights, append, [append_e], attend
        "gpu_launches": args.steps * (8 if r > 0 else 6),
        "clocks": clk.summary(),
        "wall_s": t_wall,
        "device_status": int(st),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sec, parts = oracle_step_seconds(wl)
        line["cpu_baseline"] = {
            "value": flops / sec / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": "1 head: calibrate whole, append 256 of 4680 tokens, attention of 64 of 4680 rows "
                      "over 32760 tokens; scaled to 12 heads (extrapolated)", "step_s": sec}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_small_m(args):
    """Few query rows (--small-m M) over the workload's whole cache: the
    attention is bound by reading the packed cache, so the metric is cache
    GB/s against the measured HBM copy bandwidth.  Prints its own JSON line."""
    import torch
    from bit_kv_cache_qwm_gb300 import build as B
    B.build()
    from bit_kv_cache_qwm_gb300 import qwm
    wl = synth.workload(args.workload)
    H, d, r, C, M = wl.heads, wl.head_dim, wl.rank, wl.n_centroids, args.small_m
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev, torch.bfloat16)
    kf = synth.kmeans_keys(wl)
    rows = np.stack([synth.kmeans_init_rows(wl, h, kf.shape[1], C) for h in range(H)]).astype(np.int32)
    tiles = wl.n_chunks * ((wl.chunk + 127) // 128)
    ctx = qwm.Qwm(H, d, r, C, dtype=wl.dtype, max_tokens=tiles * 128, max_hist=wl.n_hist, device=dev)
    ctx.set_centroids(qwm.qwm_kmeans(T(kf), torch.from_numpy(rows).to(dev), C, iters=25))
    ctx.calibrate(T(synth.hist_queries(wl, 0)))
    for ch in range(wl.n_chunks):
        ctx.append(T(synth.keys(wl, ch)), T(synth.values(wl, ch)))
    ctx.set_attend_kernel({"auto": 0, "simt": 1, "mma": 2, "tc": 3, "tc2": 4}[args.kernel])
    q = T(synth.queries(wl, 0, m=M))
    out = torch.empty_like(q)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    assert ctx.status() == 0, "device status bits after set-up"
    N = wl.n_tokens
    nbytes = H * N * ctx.layout.bytes_per_token + 2 * q.numel() * q.element_size()   # cache + Q + O
    kern = ctx.attend_kernel_for(M)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.zero_()
        ctx.attend(q, out)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(0) as clk:
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            ctx.attend(q, out)
            e1.record(stream)
        torch.cuda.synchronize()
    ms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs]))
    st = ctx.status()
    # end to end: Q from pinned host memory, O back to it, inside the timed region
    h_q = q.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    d_q = torch.empty_like(q)
    e2e = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        d_q.copy_(h_q, non_blocking=True)
        ctx.attend(d_q, out)
        h_out.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e.append(e0.elapsed_time(e1))
    e2e_ms = float(np.mean(e2e))
    peaks = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {
        "metric": f"qwm_attend cache GB/s, {M} query rows", "value": gbs, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "heads": H, "head_dim": d, "cached_tokens": N, "query_rows": M,
                   "n_centroids": C, "rank": r, "l2": "flushed between steps (256 MiB write)",
                   "attend_kernel": kern},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"],
                     "traffic": profiled_traffic(os.path.join(ROOT, "profiles", f"attend_small_{wl.name}_m{M}.md"),
                                                 os.path.join(ROOT, "bit_kv_cache_qwm_gb300", "csrc", "attend_small.cu"))
                     if kern == 5 else None,
                     "kernel": "qwm_attend",
                     "bytes_per_launch": nbytes, "peak_source": peaks["source"] + " HBM copy"},
        "e2e": {"value": nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": q.numel() * q.element_size(),
                "d2h_bytes_per_step": out.numel() * out.element_size(), "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * (3 if kern == 5 else 1),
        "clocks": clk.summary(),
        "device_status": int(st),
        "attend_tflops": attend_flops(H, M, N, d, r) / (ms * 1e-3) / 1e12,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="qwm", choices=["qwm", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="", choices=["", "attend", "append", "calibrate"],
                    help="profiling mode: set up the workload, then run only this call --steps times")
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "mma", "tc", "tc2"],
                    help="attention kernel (auto picks the fastest that applies)")
    ap.add_argument("--small-m", type=int, default=0,
                    help="few-row attention: M query rows over the workload's whole cache (GB/s line)")
    args = ap.parse_args()
    if args.small_m > 0 and args.impl != "reference":
        run_small_m(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
