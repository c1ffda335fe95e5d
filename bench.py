"""Throughput of the QuantWM 2-bit KV-cache hot path on one GB300 (or N).

Default workload: the long streaming video world-model cache, 24 heads,
d = 128, 256 centroids, PSAC rank 16, 240 latent frames of 1,560 tokens held
(374,400 cached tokens after the step).  The cache is first built as a real
stream: 79 steps of {qwm_calibrate on the 4,096-query ring of the previous
chunk, qwm_append of 4,680 tokens}, so it holds 79 segments, each with its
own PSAC basis version.  One timed step is then the 80th step of the stream:
  qwm_calibrate  (the 4,096-query ring, PSAC rank 16)
  qwm_append     (4,680 new tokens: QSAC over 256 centroids, INT2, PSAC e)
  qwm_attend     (the chunk's 4,680 query rows over all 374,400 tokens)
after which the cache is rewound to its 79-segment prefix (host bookkeeping),
so every timed step does the same work.  L2 is flushed between steps.

`value` is the attention algorithmic throughput of the whole step,
H (4 M N d + 2 M N r + 2 M d r) flops per step / step time, in TFLOP/s.
`roofline` is the attention kernel's rate against the measured bf16 peak;
`roofline_append` the append kernels' HBM rate (timed alone, after the main
loop) against the measured HBM copy bandwidth.

Other modes: `--workload NAME` (any synthetic workload), `--sweep` (the
append-only sweep: chunk length x centroids x rank, one JSON line per point),
`--small-m M` (few query rows, cache GB/s), `--only CALL` (profiling runs).
`--impl reference` times the fp64 CPU oracle on a bounded sample.

With N ranks (torchrun), every rank owns its own shard of heads of an N-times
larger job (rank i: heads [i H, (i+1) H) of the synthetic stream), so the
per-GPU work is fixed (weak scaling) and no data crosses ranks; the only
collectives are a barrier and the max-over-ranks of the step time.
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
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_kv_cache_qwm_gb300 import synth  # noqa: E402

WORKLOAD = "bf16-h24-stream-n374400"
METRIC = "qwm_attend TFLOP/s & cache GB/s (% roofline); qwm_append Mtokens/s"
L2_FLUSH_BYTES = 256 << 20   # twice the 129 MB L2
KERNEL_IDS = {"auto": 0, "simt": 1, "mma": 2, "tc": 3, "tc2": 4, "tc3": 6, "tc3few": 7}
KERNEL_NAMES = {0: "auto", 1: "simt", 2: "mma", 3: "tcgen05", 4: "tcgen05-2tile", 5: "few-row",
                6: "tcgen05-f16-split", 7: "tcgen05-f16-split-few-row"}
# the committed ncu summary and the source of each large-M attention kernel
KERNEL_PROFILES = {4: ("attend_tc2_{}.md", "attend_tc.cu"), 6: ("attend_tc3_{}.md", "attend_tc3.cu")}


def profiled_traffic(summary, source):
    """DRAM bytes (read + write) per launch of a kernel from a committed ncu
    summary, when the summary records the sha256 of the kernel source it was
    captured on and that source is unchanged; else None."""
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


def append_bytes_per_token_head(d, bytes_per_token, in_elem=2):
    """HBM bytes one appended token of one head moves: k and v in, packed out."""
    return 2 * d * in_elem + bytes_per_token


def alu_roofline(token_heads_per_s: float, n_centroids: int, d: int, sms: int, sm_mhz: float) -> dict:
    """The exhaustive QSAC search does 3 C d float32 operations per
    token-head (one subtraction, and a max and a min per channel and
    centroid).  Peak: one scalar float32 operation per lane per cycle on the
    128 lanes of every SM at the maximum SM clock (packed two-wide adds and
    three-input min/max can exceed it)."""
    ops = 3.0 * n_centroids * d
    peak = 128.0 * sms * sm_mhz * 1e6
    achieved = token_heads_per_s * ops
    return {"bound": "alu", "ops_per_token_head": ops, "achieved": achieved / 1e12, "peak": peak / 1e12,
            "unit": "Tops/s", "frac": achieved / peak}


def shard_heads(rank: int, world: int, heads: int) -> list:
    """Global head indices of `rank`'s shard: every rank owns `heads` heads of
    a job of world * heads heads (weak scaling; disjoint shards)."""
    if not (0 <= rank < world) or heads < 1:
        raise ValueError("rank must lie in [0, world) and heads be positive")
    return list(range(rank * heads, (rank + 1) * heads))


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
    """Work of all shards divided by the slowest rank's step time."""
    return world * flops_per_rank_step / (max_ms * 1e-3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "sm_max_mhz": j.get("sm_max_mhz", 2070.0),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
            "source": "fallback"}


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

SAMPLE_TOKENS, SAMPLE_ROWS, SAMPLE_SEGMENTS = 512, 128, 16


def oracle_sample(wl, head=0):
    """Untimed set-up of the oracle's bounded sample of one step of `wl` for
    one head: centroids, the historical queries, the last chunk's keys and
    values, the query rows, and up to SAMPLE_SEGMENTS encoded segments of the
    cache the attention reads."""
    from oracle import qwm_oracle as O
    C = wl.n_centroids
    kf = synth.kmeans_keys(wl, [head])[0]
    cent = synth.round_to_dtype(kf[synth.kmeans_init_rows(wl, head, kf.shape[1], C)], wl.dtype)
    last = wl.n_chunks - 1
    qh = synth.hist_queries(wl, last if wl.steps else 0, [head])[0]
    s = O.sensitivity(qh).astype(np.float32)
    U, _, _ = O.psac_basis(qh, wl.rank)
    w = O.group_weights(s)
    n_seg = min(SAMPLE_SEGMENTS, wl.n_chunks)
    segs = [O.append_head(synth.keys(wl, ch, [head])[0], synth.values(wl, ch, [head])[0], cent, w, U)
            for ch in range(wl.n_chunks - n_seg, wl.n_chunks)]
    return {"qh": qh, "cent": cent, "w": w, "U": U, "segs": segs, "n_seg": n_seg,
            "k": synth.keys(wl, last, [head], n=min(SAMPLE_TOKENS, wl.chunk))[0],
            "v": synth.values(wl, last, [head], n=min(SAMPLE_TOKENS, wl.chunk))[0],
            "q": synth.queries(wl, last if wl.steps else 0, [head], m=min(SAMPLE_ROWS, wl.n_query))[0]}


def oracle_step(wl, smp):
    """Time the oracle on the sample: calibrate (whole), append of
    SAMPLE_TOKENS keys, attention of SAMPLE_ROWS rows over the sampled
    segments.  Returns (seconds actually spent, extrapolated seconds of the
    whole step of all heads, breakdown).  Heads, appended tokens, query rows
    and cached segments are independent, so the work scales linearly."""
    from oracle import qwm_oracle as O
    t0 = time.perf_counter()
    s = O.sensitivity(smp["qh"]).astype(np.float32)
    U, _, _ = O.psac_basis(smp["qh"], wl.rank)
    w = O.group_weights(s)
    t1 = time.perf_counter()
    O.append_head(smp["k"], smp["v"], smp["cent"], w, U)
    t2 = time.perf_counter()
    O.attend_head(smp["q"], smp["segs"], {0: U}, 1.0 / np.sqrt(wl.head_dim))
    t3 = time.perf_counter()
    H = wl.heads
    cal = (t1 - t0) * H
    app = (t2 - t1) * H * wl.chunk / smp["k"].shape[0]
    att = (t3 - t2) * H * (wl.n_query / smp["q"].shape[0]) * (wl.n_chunks / smp["n_seg"])
    return t3 - t0, cal + app + att, {"calibrate_s": cal, "append_s": app, "attend_s": att}


def oracle_sample_text(wl, smp):
    return (f"1 of {wl.heads} heads: calibrate on {smp['qh'].shape[0]} queries (whole), append of "
            f"{smp['k'].shape[0]} of {wl.chunk} tokens, attention of {smp['q'].shape[0]} of {wl.n_query} "
            f"query rows over {smp['n_seg']} of {wl.n_chunks} cached segments; scaled linearly to the "
            f"whole step (extrapolated)")


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def one_thread_step_seconds(wl):
    """Extrapolated seconds of the same oracle step with every BLAS and OpenMP
    pool limited to one thread, timed in a child process (the thread counts of
    numpy's BLAS are fixed when it loads), or None if that fails."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1")
    code = ("import sys; sys.path.insert(0, %r); import bench; from bit_kv_cache_qwm_gb300 import synth; "
            "wl = synth.workload(%r); smp = bench.oracle_sample(wl); bench.oracle_step(wl, smp); "
            "print(bench.oracle_step(wl, smp)[1])" % (ROOT, wl.name))
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        return float(out.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError, OSError):
        return None


def run_reference(args):
    wl = synth.workload(args.workload)
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    smp = oracle_sample(wl)
    for _ in range(args.warmup):
        oracle_step(wl, smp)
    spent, extrap = [], []
    for _ in range(args.steps):
        sec, full, parts = oracle_step(wl, smp)
        spent.append(sec)
        extrap.append(full)
    step = float(np.mean(extrap))
    N = wl.n_tokens
    value = attend_flops(wl.heads, wl.n_query, N, wl.head_dim, wl.rank) / step / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": float(np.mean(spent)) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "heads": wl.heads, "head_dim": wl.head_dim,
                       "cached_tokens": N, "query_rows": wl.n_query, "chunk": wl.chunk,
                       "n_centroids": wl.n_centroids, "rank": wl.rank},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": oracle_sample_text(wl, smp)},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "extrapolated_ms_per_step": step * 1e3,
            "note": "ms_per_step is the time of the sampled step actually run; value is the whole "
                    "step's work over the extrapolated whole-step time",
            "breakdown_s": parts}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------

def _gpu_init(args):
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
    return torch, dist, qwm, world, rank, local, dev


def _generate(fn, items, threads=16):
    """Draw synthetic arrays in parallel threads (numpy's generators release
    the GIL while filling); the results are in `items` order."""
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))


def build_stream(torch, qwm, wl, heads, dev, kernel):
    """Context for `heads` of workload `wl` holding the cache of its first
    n_chunks - 1 steps.  Streaming workloads recalibrate before every append
    (one basis version per segment); the others calibrate once.  Returns
    (ctx, inputs of the last step as device tensors)."""
    H, d, r, C = len(heads), wl.head_dim, wl.rank, wl.n_centroids
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    n_prefix = wl.n_chunks - 1

    def T(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev, tdt)

    kf = synth.kmeans_keys(wl, heads)
    rows = np.stack([synth.kmeans_init_rows(wl, h, kf.shape[1], C) for h in heads]).astype(np.int32)
    tiles = wl.n_chunks * ((wl.chunk + 127) // 128)
    ctx = qwm.Qwm(H, d, r, C, dtype=wl.dtype, max_tokens=tiles * 128,
                  max_versions=(wl.n_chunks + 1) if wl.steps else 2, max_hist=wl.n_hist, device=dev)
    # the centroids: 25 Lloyd iterations on the keys of frame 0, on the GPU
    ctx.set_centroids(qwm.qwm_kmeans(T(kf), torch.from_numpy(rows).to(dev), C, iters=25))
    ctx.set_attend_kernel(KERNEL_IDS[kernel])

    def draw(ch):
        qh = synth.hist_queries(wl, ch, heads) if (wl.steps or ch == 0) else None
        return qh, synth.keys(wl, ch, heads), synth.values(wl, ch, heads)

    # drawn 16 steps at a time (bounded host memory), appended in order
    for b0 in range(0, n_prefix, 16):
        for ch, (qh, k, v) in zip(range(b0, n_prefix), _generate(draw, range(b0, min(b0 + 16, n_prefix)))):
            if qh is not None:
                ctx.calibrate(T(qh))
            ctx.append(T(k), T(v))
    last = n_prefix
    qh, k, v = draw(last)
    if qh is None:
        qh = synth.hist_queries(wl, 0, heads)
    inp = {"qh": T(qh), "k": T(k), "v": T(v), "q": T(synth.queries(wl, last if wl.steps else 0, heads))}
    return ctx, inp


def run_gpu(args):
    torch, dist, qwm, world, rank, local, dev = _gpu_init(args)
    wl = synth.workload(args.workload)
    heads = shard_heads(rank, world, wl.heads)
    H, d, r, C = wl.heads, wl.head_dim, wl.rank, wl.n_centroids
    n_prefix = wl.n_chunks - 1
    ctx, inp = build_stream(torch, qwm, wl, heads, dev, args.kernel)
    qh, k_new, v_new, q = inp["qh"], inp["k"], inp["v"], inp["q"]
    out = torch.empty_like(q)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    assert ctx.status() == 0, "device status bits after set-up"

    N = wl.n_tokens
    if args.only:
        # profiling mode: the cache holds the prefix; only the named call runs,
        # --steps times (no timing, no JSON line)
        if args.only == "attend":
            ctx.calibrate(qh)
            ctx.append(k_new, v_new)
            for _ in range(args.steps):
                ctx.attend(q, out)
        elif args.only == "append":
            ctx.calibrate(qh)
            for _ in range(args.steps):
                ctx.append(k_new, v_new)
                ctx.rewind(n_prefix)
        else:
            for _ in range(args.steps):
                ctx.calibrate(qh)
                ctx.rewind(n_prefix)
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
    out_ref = out.clone()

    # the append kernels alone (quantisation and PSAC coefficients), with the
    # step's calibration already in place: the HBM roofline of the append
    ctx.calibrate(qh)
    torch.cuda.synchronize()
    app_alone = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ctx.append(k_new, v_new)
        e1.record(stream)
        ctx.rewind(n_prefix)
        if i >= args.warmup:
            app_alone.append((e0, e1))
    torch.cuda.synchronize()
    app_ms = float(np.mean([a.elapsed_time(b) for a, b in app_alone]))
    ctx.rewind(n_prefix)

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
    e2e_same = bool(torch.equal(h_out[(args.steps - 1) & 1], out_ref.cpu()))
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = h_out[0].numel() * h_out[0].element_size()
    st = st | ctx.status()

    peaks = load_peaks()
    att_ms = float(np.mean(att))
    achieved = flops / (att_ms * 1e-3) / 1e12
    value = whole_job_tflops(flops, world, ms_step)
    kern = ctx.resolved_attend_kernel
    in_elem = 2 if wl.dtype == "bf16" else 4
    app_bytes = H * wl.chunk * append_bytes_per_token_head(d, ctx.layout.bytes_per_token, in_elem)
    app_gbs = app_bytes / (app_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "heads": H, "head_dim": d, "cached_tokens": N,
                   "query_rows": wl.n_query, "chunk": wl.chunk, "n_centroids": C, "rank": r,
                   "hist_queries": wl.n_hist, "basis_versions_in_cache": wl.n_chunks if wl.steps else 1,
                   "parallelism": f"head shards x{world} (heads {heads[0]}-{heads[-1]} on rank {rank})",
                   "l2": "flushed between steps (256 MiB write)",
                   "centroids": "k-means on frame 0 (25 Lloyd iterations, GPU)"},
        "components": {"calibrate_ms": float(np.mean(cal)), "append_ms": float(np.mean(app)),
                       "attend_ms": att_ms, "attend_tflops": achieved,
                       "cache_gbs": cache_bytes / (att_ms * 1e-3) / 1e9,
                       "append_alone_ms": app_ms,
                       "append_mtok_s": wl.chunk / (app_ms * 1e-3) / 1e6,
                       "append_token_heads_per_s": H * wl.chunk / (app_ms * 1e-3),
                       "attend_kernel": KERNEL_NAMES.get(kern, "?")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"],
                     "traffic": profiled_traffic(os.path.join(ROOT, "profiles", KERNEL_PROFILES[kern][0].format(wl.name)),
                                                 os.path.join(ROOT, "bit_kv_cache_qwm_gb300", "csrc",
                                                              KERNEL_PROFILES[kern][1]))
                     if kern in KERNEL_PROFILES else None,
                     "kernel": "qwm_attend", "peak_source": peaks["source"] + " burst bf16",
                     "work": "H (4 M N d + 2 M N r + 2 M d r) flops per launch"},
        "roofline_append": {"bound": "hbm", "achieved": app_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": app_gbs / peaks["hbm_gbs"], "kernel": "qwm_append",
                            "bytes_per_token_head": append_bytes_per_token_head(d, ctx.layout.bytes_per_token,
                                                                                in_elem),
                            "traffic": profiled_traffic(os.path.join(ROOT, "profiles", f"append_{wl.name}.md"),
                                                        os.path.join(ROOT, "bit_kv_cache_qwm_gb300", "csrc",
                                                                     "append.cu")),
                            "peak_source": peaks["source"] + " HBM copy",
                            "alu": alu_roofline(H * wl.chunk / (app_ms * 1e-3), C, d,
                                                torch.cuda.get_device_properties(dev).multi_processor_count,
                                                peaks["sm_max_mhz"])},
        "e2e": {"value": world * flops / (e2e_step * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_step,
                "copies": "second stream, double-buffered: inputs of step i+1 and output of step i-1 "
                          "move while step i computes", "output_matches_device_timed": e2e_same},
        # gram, gram_sum, [square], eig, weights, append, [append_e], attend
        "gpu_launches": args.steps * (8 if r > 0 else 6),
        "clocks": clk.summary(),
        "wall_s": t_wall,
        "device_status": int(st),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = oracle_sample(wl)
        oracle_step(wl, smp)                          # warm-up
        runs = []
        while sum(x[0] for x in runs) < 10.0:        # about 10 s of CPU work
            runs.append(oracle_step(wl, smp))
        spent = float(np.mean([x[0] for x in runs]))
        full = float(np.mean([x[1] for x in runs]))
        parts = {k: float(np.mean([x[2][k] for x in runs])) for k in runs[0][2]}
        one = one_thread_step_seconds(wl)
        line["cpu_baseline"] = {
            "value": flops / full / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": oracle_sample_text(wl, smp) + f"; {len(runs)} repetitions averaged",
            "step_s": full, "sample_s": spent, "breakdown_s": parts,
            "value_1_thread": (flops / one / 1e12) if one else None}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_sweep(args):
    """The append-only sweep: for every (chunk length, centroids, rank) point,
    one JSON line with the append's Mtokens/s and its HBM fraction."""
    torch, dist, qwm, world, rank, local, dev = _gpu_init(args)
    wl = synth.workload("bf16-h24-append-sweep")
    heads = shard_heads(rank, world, wl.heads)
    H, d = wl.heads, wl.head_dim
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev, torch.bfloat16)
    n_max = max(wl.sweep["chunk"])
    k_all, v_all = T(synth.keys(wl, 1, heads, n=n_max)), T(synth.values(wl, 1, heads, n=n_max))
    qh = T(synth.hist_queries(wl, 0, heads))
    kf = synth.kmeans_keys(wl, heads)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peaks = load_peaks()
    stream = torch.cuda.current_stream()
    points = [(n, C, r) for C in wl.sweep["n_centroids"] for r in wl.sweep["rank"] for n in wl.sweep["chunk"]]
    if args.sweep_points:
        points = points[: args.sweep_points]
    cents = {}
    for n, C, r in points:
        if C not in cents:
            rows = np.stack([synth.kmeans_init_rows(wl, h, kf.shape[1], C) for h in heads]).astype(np.int32)
            cents[C] = qwm.qwm_kmeans(T(kf), torch.from_numpy(rows).to(dev), C, iters=25)
        ctx = qwm.Qwm(H, d, r, C, dtype="bf16", max_tokens=((n + 127) // 128) * 128, max_versions=2,
                      max_hist=wl.n_hist, device=dev)
        ctx.set_centroids(cents[C])
        ctx.calibrate(qh)
        k, v = k_all[:, :n].contiguous(), v_all[:, :n].contiguous()
        evs = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ctx.append(k, v)
            e1.record(stream)
            ctx.rewind(0)
            if i >= args.warmup:
                evs.append((e0, e1))
        torch.cuda.synchronize()
        st = ctx.status()
        ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in evs])), dev)
        bpt = append_bytes_per_token_head(d, ctx.layout.bytes_per_token)
        gbs = world * H * n * bpt / (ms * 1e-3) / 1e9
        line = {"metric": "qwm_append Mtokens/s", "value": world * n / (ms * 1e-3) / 1e6, "unit": "Mtokens/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic",
                "config": {"workload": wl.name, "heads": H, "head_dim": d, "chunk": n, "n_centroids": C,
                           "rank": r, "l2": "flushed between steps (256 MiB write)"},
                "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": gbs / peaks["hbm_gbs"], "bytes_per_token_head": bpt,
                             "peak_source": peaks["source"] + " HBM copy",
                             "alu": alu_roofline(world * H * n / (ms * 1e-3), C, d,
                                                 torch.cuda.get_device_properties(dev).multi_processor_count,
                                                 peaks["sm_max_mhz"])},
                "token_heads_per_s": world * H * n / (ms * 1e-3),
                "gpu_launches": args.steps * (2 if r > 0 else 1), "device_status": int(st)}
        ctx.close()
        if rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_small_m(args):
    """Few query rows (--small-m M) over the workload's whole cache: the
    attention is bound by reading the packed cache, so the metric is cache
    GB/s against the measured HBM copy bandwidth.  Prints its own JSON line."""
    torch, dist, qwm, world, rank, local, dev = _gpu_init(args)
    wl = synth.workload(args.workload)
    heads = shard_heads(rank, world, wl.heads)
    H, d, r, C, M = wl.heads, wl.head_dim, wl.rank, wl.n_centroids, args.small_m
    ctx, inp = build_stream(torch, qwm, wl, heads, dev, args.kernel)
    ctx.calibrate(inp["qh"])
    ctx.append(inp["k"], inp["v"])
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    q = torch.from_numpy(synth.queries(wl, wl.n_chunks - 1 if wl.steps else 0, heads, m=M)).to(dev, tdt)
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
    if world > 1:
        dist.barrier()
    with ClockSampler(local) as clk:
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            ctx.attend(q, out)
            e1.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs])), dev)
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
    e2e_ms = max_over_ranks(float(np.mean(e2e)), dev)
    peaks = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {
        "metric": f"qwm_attend cache GB/s, {M} query rows", "value": world * gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "heads": H, "head_dim": d, "cached_tokens": N, "query_rows": M,
                   "n_centroids": C, "rank": r, "l2": "flushed between steps (256 MiB write)",
                   "attend_kernel": kern},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"],
                     "traffic": profiled_traffic(os.path.join(ROOT, "profiles", f"attend_small_{wl.name}_m{M}.md"),
                                                 os.path.join(ROOT, "bit_kv_cache_qwm_gb300", "csrc", "attend_small.cu"))
                     if kern == 5 else
                     profiled_traffic(os.path.join(ROOT, "profiles", f"attend_tc3few_{wl.name}_m{M}.md"),
                                      os.path.join(ROOT, "bit_kv_cache_qwm_gb300", "csrc", "attend_tc3.cu"))
                     if kern == 7 else None,
                     "kernel": "qwm_attend",
                     "bytes_per_launch": nbytes, "peak_source": peaks["source"] + " HBM copy"},
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": q.numel() * q.element_size(),
                "d2h_bytes_per_step": out.numel() * out.element_size(), "ms_per_step": e2e_ms},
        # kernel 5: the QC table, the split attention and the merge; kernel 7:
        # the split attention and the merge
        "gpu_launches": args.steps * {5: 3, 7: 2}.get(kern, 1),
        "clocks": clk.summary(),
        "device_status": int(st),
        "attend_tflops": attend_flops(H, M, N, d, r) / (ms * 1e-3) / 1e12,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="qwm", choices=["qwm", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="", choices=["", "attend", "append", "calibrate"],
                    help="profiling mode: set up the workload, then run only this call --steps times")
    ap.add_argument("--kernel", default="auto", choices=sorted(KERNEL_IDS),
                    help="attention kernel (auto picks the fastest that applies)")
    ap.add_argument("--small-m", type=int, default=0,
                    help="few-row attention: M query rows over the workload's whole cache (GB/s line)")
    ap.add_argument("--sweep", action="store_true", help="the append-only sweep, one JSON line per point")
    ap.add_argument("--sweep-points", type=int, default=0, help="only the first N sweep points")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    elif args.small_m > 0:
        run_small_m(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
