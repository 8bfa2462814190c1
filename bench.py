"""Benchmark of the streaming chunk-attention hot path on GB300.

The default workload is the 720p chunk (40 heads x 128, 45x80 latent grid,
two-frame chunks, sinks of 4112 tokens, an 8-frame ring), the largest
configuration that fits one GPU, in steady state (ring full): per chunk, for
each of the two denoising steps, RoPE-3D on the chunk's Q/K and the chunk
attention over sink bank + ring + chunk; then the ring commit. A bench step is
several chunks (8 at 720p, about 50 ms), so that the clock sampler sees the GPU
under load throughout the timed steps. Inputs are seeded synthetic bf16 N(0,1),
resident in HBM before the timed region. Two independent sessions are used
alternately, so every chunk reads inputs that were last touched more than an
L2's worth of traffic ago. ``--config 2`` runs the 832x480 chunk instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 2|3]
                    [--workload steady|rhythm|window|graph|decoder|batch|long]

``--workload rhythm`` times the pages' unit rhythm instead (chunks of 3 and 2
latent frames at the 832x480 frame size) and ``--workload window`` the
page-faithful window (recomputed history rows as queries), ``--workload graph``
a chunk issued eagerly against one CUDA-graph replay, ``--workload decoder``
the streaming decoder's window attention per layer; each prints its own line.

Multi-GPU: the path has no exchange step, so N ranks run N independent
replicas (weak scaling, no collective on the data path); rank 0 prints the
aggregate. ``--impl reference`` times the float64 CPU oracle on the host
cores on a bounded sample of the same workload (the reference arm).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

import synthetic as syn

METRIC = "chunk-attention ms/step and TFLOP/s on 1 GB300; % of bf16 tensor peak"
# chunks per bench step of the steady workload, per config (about 50 ms per step)
CHUNKS_PER_STEP = {2: 64, 3: 8}
UNIT = "TFLOP/s"


# The part's nominal dense figures, reported beside the measured peaks and
# labelled as such: bf16 tensor throughput without sparsity, and HBM3e bandwidth.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["hbm_gbs"]), "measured"
    return 1900.0, 6800.0, "fallback"


def _sustained_bf16():
    """The bf16 GEMM rate held for seconds under the power cap: the peak of a
    kernel timed inside a long, back-to-back step."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured"
    return 1700.0, "fallback"



def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device) -> float:
    """Job time = the slowest rank's time (replicas run the same work)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, seconds: float, world: int) -> float:
    """Whole-job throughput of N replicas: every rank's units over the max time."""
    return world * units_per_rank / seconds


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _make_session(shape, config, sess_id, dev):
    import chunked_kv_cache_gb300 as sr
    W = shape.window_frames
    sink = lambda tid: syn.device_normal_bf16((shape.n_steps, shape.n_sink, shape.n_heads, shape.head_dim), dev,
                                              config, sess_id, 0, 0, tid)
    s = sr.Session(shape.n_heads, shape.head_dim, shape.grid_h, shape.grid_w, shape.chunk_frames, W,
                   shape.n_sink, shape.n_steps, sink_k=sink(syn.T_SINK_K), sink_v=sink(syn.T_SINK_V), device=dev)
    s.ring_k.copy_(syn.device_normal_bf16(tuple(s.ring_k.shape), dev, config, sess_id, 0, 0, syn.T_RING_K))
    s.ring_v.copy_(syn.device_normal_bf16(tuple(s.ring_v.shape), dev, config, sess_id, 0, 0, syn.T_RING_V))
    s.slot_frame.copy_(torch.arange(W, dtype=torch.int32, device=dev))
    s.restore(W)                                   # steady state: ring full
    x = syn.chunk_inputs_device(shape, config, dev, session=sess_id, chunk=0)
    x["o"] = [torch.empty_like(x["q"][0]) for _ in range(shape.n_steps)]
    return s, x


def _chunk(s, x, n_steps):
    """One streaming chunk through the library: 2 x (RoPE + attention) + commit."""
    for st in range(n_steps):
        s.rope3d_qk(x["q"][st], x["k"][st])
        s.chunk_attention(st, x["q"][st], x["k"][st], x["v"][st], out=x["o"][st])
    s.cache_commit(x["clean_k"], x["clean_v"])


def run_ours(args):
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from chunked_kv_cache_gb300 import build
    build.build()
    shape = syn.SHAPES[args.config]
    full = shape.window_frames
    flops_attn = shape.attention_flops(full)               # one denoising step
    flops_chunk = shape.n_steps * flops_attn
    commit_bytes = 4 * shape.lq * shape.n_heads * shape.head_dim * 2
    sessions = [_make_session(shape, args.config, i + 10 * rank, dev) for i in range(2)]
    session_mb = sum(t.numel() * t.element_size() for t in
                     [sessions[0][0].sink_k, sessions[0][0].sink_v, sessions[0][0].ring_k, sessions[0][0].ring_v] +
                     [v for val in sessions[0][1].values() for v in (val if isinstance(val, list) else [val])]) / 1e6
    # A bench step is R chunks, enough for tens of milliseconds, so that the
    # clock sampler sees the GPU under load many times over the timed steps.
    R = args.chunks_per_step or CHUNKS_PER_STEP[args.config]
    torch.cuda.synchronize()
    for i in range(args.warmup * R):
        s, x = sessions[i % 2]
        _chunk(s, x, shape.n_steps)
    torch.cuda.synchronize()

    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    # Events bracket only the attention launches, whose duration the roofline
    # needs: an event recorded between two launches sits between them in the
    # stream and can hold back the second one's early (programmatic) start. The
    # RoPE and commit kernels are timed back to back after the loop.
    n_chunks = args.steps * R
    per = [[mk() for _ in range(shape.n_steps)] for _ in range(n_chunks)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clk:
        t0.record()
        for i in range(n_chunks):
            s, x = sessions[i % 2]
            p = per[i]
            for st in range(shape.n_steps):
                s.rope3d_qk(x["q"][st], x["k"][st])
                p[st][0].record()
                s.chunk_attention(st, x["q"][st], x["k"][st], x["v"][st], out=x["o"][st])
                p[st][1].record()
            s.cache_commit(x["clean_k"], x["clean_v"])
        t1.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    elapsed = t0.elapsed_time(t1) / 1e3
    attn_ms = [a[0].elapsed_time(a[1]) for p in per for a in p]
    for s, _ in sessions:
        if s.error_status() != 0:
            raise RuntimeError("device error word set during the bench")
    elapsed = max_over_ranks(elapsed, dev)

    # end to end through the public API: pinned host inputs in, result out
    e2e = run_e2e(shape, args, dev, sessions[0][0]) if not args.profile else {"seconds": 1.0, "chunks": 0,
                                                                              "h2d": 0, "d2h": 0}
    e2e["seconds"] = max_over_ranks(e2e["seconds"], dev)
    clocks = clk.summary()
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peak_tf, peak_gbs, peak_kind = _peaks()
    sus_tf, sus_kind = _sustained_bf16()
    attn_avg = statistics.mean(attn_ms)
    achieved = flops_attn / (attn_avg / 1e3) / 1e12
    value = aggregate_throughput(n_chunks * flops_chunk, elapsed, world) / 1e12
    # The two HBM-bound kernels last ~20 us, close to the event timer's
    # granularity; time them again over 16 back-to-back launches each, cycling
    # through six input pairs of the two sessions (230 MB at 832x480, more than
    # the L2) so the inputs of a launch are not in L2.
    rope_avg, commit_avg = hbm_kernel_times(sessions, shape)
    cpu = cpu_baseline(shape, args) if world == 1 and not args.profile else None
    traffic = _profiled_traffic("chunk_attention", args.config)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "ms_per_chunk": round(elapsed / n_chunks * 1e3, 4), "chunks_per_step": R,
        "config": {"workload": shape.name + f", steady state (ring full), one step = {R} chunks, each "
                               "2 x (RoPE-3D + chunk attention) + ring commit",
                   "heads": shape.n_heads, "head_dim": shape.head_dim, "lq": shape.lq,
                   "lk": shape.lk(full), "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: two sessions of {session_mb:.0f} MB used alternately"},
        "attention_ms_per_denoise_step": round(attn_avg, 4),
        "attention_ms_p10_p50_p90": [round(float(np.percentile(attn_ms, q)), 4) for q in (10, 50, 90)],
        "attention_tflops": round(achieved, 2),
        # the attention launches run back to back for about a second under the
        # power cap: the sustained bf16 rate is their peak (burst beside it)
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": sus_tf, "unit": "TFLOP/s",
                     "frac": round(achieved / sus_tf, 4), "traffic": traffic,
                     "kernel": "attn_kernel (sr_chunk_attention)",
                     "peak_kind": f"{sus_kind} bf16 dense sustained (seconds-long GEMM loop under the power cap)",
                     "burst_peak": peak_tf, "frac_of_burst": round(achieved / peak_tf, 4),
                     "frac_of_nominal": round(achieved / NOMINAL_BF16_TFLOPS, 4),
                     "nominal_peak": f"{NOMINAL_BF16_TFLOPS:.0f} TFLOP/s nominal dense bf16 (spec, not measured)"},
        "kernels": {
            "commit": {"us": round(commit_avg * 1e3, 2), "GB/s": round(commit_bytes / (commit_avg / 1e3) / 1e9, 1),
                       "frac_hbm": round(commit_bytes / (commit_avg / 1e3) / 1e9 / peak_gbs, 4),
                       "frac_hbm_nominal": round(commit_bytes / (commit_avg / 1e3) / 1e9 / NOMINAL_HBM_GBS, 4)},
            "rope3d_qk": {"us": round(rope_avg * 1e3, 2),
                          "GB/s": round(commit_bytes / (rope_avg / 1e3) / 1e9, 1),
                          "frac_hbm": round(commit_bytes / (rope_avg / 1e3) / 1e9 / peak_gbs, 4),
                          "frac_hbm_nominal": round(commit_bytes / (rope_avg / 1e3) / 1e9 / NOMINAL_HBM_GBS, 4)},
        },
        "e2e": {"value": round(aggregate_throughput(e2e["chunks"] * flops_chunk, e2e["seconds"], world) / 1e12, 2),
                "unit": UNIT,
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]},
        "cpu_baseline": cpu,
        "clocks": clocks,
        "gpu_launches": (2 * shape.n_steps + 1) * n_chunks,
    }
    print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def hbm_kernel_times(sessions, shape, reps: int = 16, rounds: int = 7):
    """Mean ms per launch of RoPE-3D (mode 0) and of the ring commit, each timed
    over `reps` back-to-back launches between one pair of events; the median of
    `rounds` such timings."""
    pairs = [(x["q"][st], x["k"][st]) for _, x in sessions for st in range(shape.n_steps)]
    pairs += [(x["clean_k"], x["clean_v"]) for _, x in sessions]
    out = []
    for kind in ("rope", "commit"):
        times = []
        for _ in range(rounds):
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            ev0.record()
            for i in range(reps):
                if kind == "rope":
                    s = sessions[i % len(sessions)][0]
                    q, k = pairs[i % len(pairs)]
                    s.rope3d_qk(q, k)
                else:
                    s, x = sessions[i % len(sessions)]
                    s.cache_commit(x["clean_k"], x["clean_v"])
            ev1.record()
            torch.cuda.synchronize()
            times.append(ev0.elapsed_time(ev1) / reps)
        out.append(statistics.median(times))
    return out[0], out[1]


def run_e2e(shape, args, dev, sess):
    """Same chunk through the public API with the step's inputs copied in from
    pinned host memory and both steps' outputs copied back, every step, each
    direction as one copy of a contiguous block. Uploads and read-backs run on
    two more streams (the host link is full duplex), over three buffer sets:
    chunk i+2's inputs go up and chunk i-1's outputs come back while chunk i
    computes; every chunk still moves all of its own inputs
    and outputs inside the timed region, which starts before the first upload
    and ends after the last read-back. Reported: the median of three such
    timed runs of n chunks."""
    n = max(3, args.steps)
    nbuf = 3
    dims = (shape.lq, shape.n_heads, shape.head_dim)
    g = torch.Generator().manual_seed(1234)
    n_in = 3 * shape.n_steps + 2
    # one contiguous block per buffer set and direction, so that a chunk's
    # inputs go up in one copy and its outputs come back in one copy
    host_in_blk = [torch.randn((n_in,) + dims, generator=g).to(torch.bfloat16).pin_memory() for _ in range(nbuf)]
    host_out_blk = [torch.empty((shape.n_steps,) + dims, dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    dev_in_blk = [torch.empty((n_in,) + dims, dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    dev_out_blk = [torch.empty((shape.n_steps,) + dims, dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    dev_in = [list(blk.unbind(0)) for blk in dev_in_blk]
    dev_out = [list(blk.unbind(0)) for blk in dev_out_blk]
    comp = torch.cuda.current_stream(dev)
    h2d = torch.cuda.Stream(dev)
    d2h = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()

    def run(chunks):
        up = [ev() for _ in range(chunks)]       # inputs of chunk i are on the device
        done = [ev() for _ in range(chunks)]     # chunk i computed
        down = [ev() for _ in range(chunks)]     # chunk i's outputs are back on the host
        def upload(i):
            b = i % nbuf
            with torch.cuda.stream(h2d):
                if i >= nbuf:
                    h2d.wait_event(done[i - nbuf])   # buffer set b is free again
                dev_in_blk[b].copy_(host_in_blk[b], non_blocking=True)
                up[i].record(h2d)
        for i in range(min(nbuf - 1, chunks)):
            upload(i)
        for i in range(chunks):
            b = i % nbuf
            if i + nbuf - 1 < chunks:
                upload(i + nbuf - 1)
            comp.wait_event(up[i])
            if i >= nbuf:
                comp.wait_event(down[i - nbuf])      # its output buffers have been read back
            for st in range(shape.n_steps):
                q, k, v = dev_in[b][3 * st], dev_in[b][3 * st + 1], dev_in[b][3 * st + 2]
                sess.rope3d_qk(q, k)
                sess.chunk_attention(st, q, k, v, out=dev_out[b][st])
            sess.cache_commit(dev_in[b][-2], dev_in[b][-1])
            done[i].record(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(done[i])
                host_out_blk[b].copy_(dev_out_blk[b], non_blocking=True)
                down[i].record(d2h)
        torch.cuda.synchronize()

    run(3)
    # the median of three timed runs: a single one of about 25 ms at 832x480
    # is exposed to host hiccups (one such run read 1.5x the others)
    secs = []
    for _ in range(3):
        t = time.perf_counter()
        run(n)
        secs.append(time.perf_counter() - t)
    sec = statistics.median(secs)
    per = dims[0] * dims[1] * dims[2] * 2
    return {"seconds": sec, "chunks": n, "h2d": per * n_in, "d2h": per * shape.n_steps}


def _profiled_traffic(kernel, config):
    """DRAM bytes per launch from the committed ncu summary, if it matches."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}/config{config}")
    return None if e is None or e.get("stale") else e.get("bytes_per_launch")


def _host_info():
    """The host's CPU model (lscpu) and BLAS thread count, for the oracle lines."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    threads = None
    try:
        from threadpoolctl import threadpool_info
        blas = [d for d in threadpool_info() if d.get("user_api") == "blas"]
        threads = blas[0]["num_threads"] if blas else None
    except ImportError:
        env = [os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS")]
        threads = next((int(v) for v in env if v), None)
    return {"cpu_model": model,
            "blas_threads": threads if threads is not None else f"library default ({os.cpu_count()} cores)"}


def cpu_baseline(shape, args, budget_s: float = 12.0):
    """The float64 oracle, as it stands, on this host's cores: attention of
    whole heads of one denoising step (full window) until the time budget is
    used; returns TFLOP/s scaled by the sampled fraction."""
    from oracle import attention, bf16_bits_to_f64
    full = shape.window_frames
    lk = shape.lk(full)
    g = np.random.default_rng(0)
    heads_done, t_used = 0, 0.0
    while t_used < budget_s and heads_done < shape.n_heads:
        q = g.standard_normal((shape.lq, 1, shape.head_dim))
        k = g.standard_normal((lk, 1, shape.head_dim))
        v = g.standard_normal((lk, 1, shape.head_dim))
        t = time.perf_counter()
        attention(q, k, v, 1.0 / math.sqrt(shape.head_dim))
        t_used += time.perf_counter() - t
        heads_done += 1
    flops = 4.0 * heads_done * shape.lq * lk * shape.head_dim
    extra = ("" if heads_done == shape.n_heads else
             f"; heads are independent, so the rate of the sampled heads stands for all {shape.n_heads} "
             "(extrapolated linearly)")
    return {"value": round(flops / t_used / 1e12, 5), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{heads_done} of {shape.n_heads} heads of one denoising step "
                      f"({shape.lq} queries x {lk} keys, float64 numpy), {t_used:.1f} s{extra}", **_host_info()}


def _oracle_attention_rate(parts, d, budget_s: float = 6.0):
    """The float64 oracle's attention on the host cores, one head at a time over
    the (queries, keys) shapes in `parts`, round robin until the time budget is
    used (at least one head each). Returns (flop/s, heads done, seconds)."""
    from oracle import attention
    g = np.random.default_rng(0)
    done, used, flops = 0, 0.0, 0.0
    while done < len(parts) or used < budget_s:
        lq, lk = parts[done % len(parts)]
        q = g.standard_normal((lq, 1, d))
        k = g.standard_normal((lk, 1, d))
        v = g.standard_normal((lk, 1, d))
        t = time.perf_counter()
        attention(q, k, v, 1.0 / math.sqrt(d))
        used += time.perf_counter() - t
        flops += 4.0 * lq * lk * d
        done += 1
    return flops / used, done, used


def _oracle_line(rate, done, used, what, value=None, unit=UNIT):
    """cpu_baseline object: TFLOP/s unless a converted value and unit are given."""
    return {"value": round(rate / 1e12, 5) if value is None else value, "unit": unit, "cores": os.cpu_count(),
            "kind": "oracle", "sample": f"{done} heads of {what} (float64 numpy), {used:.1f} s", **_host_info()}


def run_reference(args):
    """Reference arm: the float64 oracle on the host cores, each step a bounded
    sample (one head of one denoising step, full window) of the same workload."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    from oracle import OracleSession, attention
    shape = syn.SHAPES[args.config]
    full = shape.window_frames
    lk = shape.lk(full)
    g = np.random.default_rng(0)
    q = g.standard_normal((shape.lq, 1, shape.head_dim))
    k = g.standard_normal((lk, 1, shape.head_dim))
    v = g.standard_normal((lk, 1, shape.head_dim))
    scale = 1.0 / math.sqrt(shape.head_dim)
    for _ in range(args.warmup):
        attention(q, k, v, scale)
    t = time.perf_counter()
    for _ in range(args.steps):
        attention(q, k, v, scale)
    sec = time.perf_counter() - t
    flops = 4.0 * shape.lq * lk * shape.head_dim
    value = args.steps * flops / sec / 1e12
    sample = f"one head of one denoising step per bench step ({shape.lq} queries x {lk} keys, float64 numpy)"
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec / args.steps * 1e3, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": shape.name + ", steady state (ring full)", "heads": shape.n_heads,
                      "lq": shape.lq, "lk": lk},
           "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                            "sample": sample, **_host_info()},
           "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_rhythm(args):
    """The pages' unit rhythm at the 832x480 frame size: after the 9-latent
    first window, chunks alternate 3 latents (2 latents of history) and 2
    latents (3 of history); the ring holds W = 3 latent frames. One bench step
    = one chunk (2 x (RoPE + attention) + commit), steps alternating the two
    chunk kinds; two sessions are used alternately, as in the main workload."""
    import chunked_kv_cache_gb300 as sr
    world, rank, local = _dist()
    if rank != 0:
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from chunked_kv_cache_gb300 import build
    build.build()
    base = syn.SHAPES[2]
    W, Fmax = 3, 9
    T, H, d, S = base.tokens_per_frame, base.n_heads, base.head_dim, base.n_sink
    sessions = []
    for sid in range(2):
        sink = lambda tid: syn.device_normal_bf16((base.n_steps, S, H, d), dev, 5, sid, 0, 0, tid)
        s = sr.Session(H, d, base.grid_h, base.grid_w, 3, W, S, base.n_steps, sink_k=sink(syn.T_SINK_K),
                       sink_v=sink(syn.T_SINK_V), device=dev)
        xs = {}
        for F in (2, 3, Fmax):
            dims = (F * T, H, d)
            xs[F] = {k: [syn.device_normal_bf16(dims, dev, 5, sid, F, st, tid) for st in range(base.n_steps)]
                     for k, tid in (("q", syn.T_Q), ("k", syn.T_K), ("v", syn.T_V))}
            xs[F]["clean_k"] = syn.device_normal_bf16(dims, dev, 5, sid, F, 0, syn.T_CLEAN_K)
            xs[F]["clean_v"] = syn.device_normal_bf16(dims, dev, 5, sid, F, 0, syn.T_CLEAN_V)
            xs[F]["o"] = torch.empty(dims, dtype=torch.bfloat16, device=dev)
        sessions.append([s, xs, 0])          # session, inputs, next chunk index

    def chunk(entry, ev=None):
        s, xs, c = entry
        plan = sr.plan_chunk(c)
        F, h = plan["n_frames"], min(plan["hist_frames"], W)
        x = xs[F]
        for st in range(base.n_steps):
            s.rope3d_qk(x["q"][st], x["k"][st], frames=F)
            if ev is not None:
                ev[st][0].record()
            s.chunk_attention(st, x["q"][st], x["k"][st], x["v"][st], out=x["o"], frames=F, hist=h)
            if ev is not None:
                ev[st][1].record()
        s.cache_commit(x["clean_k"], x["clean_v"], frames=F)
        entry[2] = c + 1
        return F, h

    # first window, then warm-up chunks in pairs, so that every session's next
    # chunk is a 3-latent one and the timed steps alternate 3 and 2 latents
    for e in sessions:
        for _ in range(1 + 2 * max(2, args.warmup // 2)):
            chunk(e)
    torch.cuda.synchronize()
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    steps = max(2, args.steps - args.steps % 2)
    evs = [[mk() for _ in range(base.n_steps)] for _ in range(steps)]
    kinds = []
    t0, t1 = mk()
    with Clocks(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clk:
        t0.record()
        for i in range(steps):
            kinds.append(chunk(sessions[(i // 2) % 2], evs[i]))
        t1.record()
        torch.cuda.synchronize()
    for s, _, _ in sessions:
        if s.error_status() != 0:
            raise RuntimeError("device error word set during the bench")
    elapsed = t0.elapsed_time(t1) / 1e3
    peak_tf, _, peak_kind = _peaks()
    per_kind = {}
    tot_fl, tot_ms = 0.0, 0.0
    for (F, h), ev in zip(kinds, evs):
        lq, lk = F * T, S + h * T + F * T
        fl = 4.0 * H * lq * lk * d
        ms = [a.elapsed_time(b) for a, b in ev]
        k = f"{F}_latents"
        e = per_kind.setdefault(k, {"lq": lq, "lk": lk, "hist_frames": h, "attn_ms": [], "flops": fl})
        e["attn_ms"].extend(ms)
        tot_fl += fl * len(ms)
        tot_ms += sum(ms)
    for e in per_kind.values():
        m = statistics.mean(e.pop("attn_ms"))
        e["attention_ms_per_denoise_step"] = round(m, 4)
        e["attention_tflops"] = round(e.pop("flops") / (m / 1e3) / 1e12, 2)
    achieved = tot_fl / (tot_ms / 1e3) / 1e12
    out = {
        "metric": "unit-rhythm chunk attention TFLOP/s and ms per chunk on 1 GB300", "value": round(achieved, 2),
        "unit": UNIT, "n_gpus": 1, "steps": steps, "warmup": args.warmup,
        "ms_per_chunk": round(elapsed / steps * 1e3, 4), "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "832x480 latent frames (24x128, 30x52 grid, S=2072), the pages' unit rhythm: "
                               "9-latent first window, then chunks of 3 and 2 latents with 2 and 3 latents of "
                               "recent history, ring W=3; one step = one chunk: 2 x (RoPE-3D + attention) + commit",
                   "l2": "two sessions used alternately"},
        "chunks": per_kind,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tf, 4), "kernel": "attn_kernel (sr_chunk_attention_frames)",
                     "peak_kind": f"{peak_kind} bf16 dense burst"},
        "cpu_baseline": _oracle_line(*_oracle_attention_rate([(e["lq"], e["lk"]) for e in per_kind.values()], d),
                                     "one denoising step of the 3- and 2-latent chunks, alternately"),
        "clocks": clk.summary(),
        "gpu_launches": 5 * steps,
    }
    print(json.dumps(out), flush=True)


def run_window(args):
    """The page-faithful window at the 832x480 frame size under the unit rhythm:
    every chunk recomputes its moving rows (2 or 3 latents of history, then the
    3- or 2-latent chunk: 5 latent frames, 7800 rows) and attends them over the
    bank of the step and themselves; the prefix pass (2072 prefix rows over
    the bank alone) runs in the same launch on the first window only and is
    timed separately. One bench step = one chunk: 2 x (RoPE at the moving rows'
    frame times + window attention). No ring: this is what the ring caches."""
    import chunked_kv_cache_gb300 as sr
    world, rank, local = _dist()
    if rank != 0:
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from chunked_kv_cache_gb300 import build
    build.build()
    base = syn.SHAPES[2]
    T, H, d, S = base.tokens_per_frame, base.n_heads, base.head_dim, base.n_sink
    moving = 5
    M = moving * T
    sessions = []
    for sid in range(2):
        sink = lambda tid: syn.device_normal_bf16((base.n_steps, S, H, d), dev, 6, sid, 0, 0, tid)
        s = sr.Session(H, d, base.grid_h, base.grid_w, 3, 0, S, base.n_steps, sink_k=sink(syn.T_SINK_K),
                       sink_v=sink(syn.T_SINK_V), device=dev)
        x = {k: [syn.device_normal_bf16((M, H, d), dev, 6, sid, 1, st, tid) for st in range(base.n_steps)]
             for k, tid in (("q", syn.T_Q), ("k", syn.T_K), ("v", syn.T_V))}
        x["o"] = torch.empty((M, H, d), dtype=torch.bfloat16, device=dev)
        x["qp"] = syn.device_normal_bf16((S + M, H, d), dev, 6, sid, 2, 0, syn.T_Q)
        x["op"] = torch.empty_like(x["qp"])
        sessions.append((s, x))
    first = [9]

    def chunk(s, x, c, ev=None):
        plan = sr.plan_chunk(c)
        h, F = plan["hist_frames"], plan["n_frames"]
        assert h + F == moving
        for st in range(base.n_steps):
            s.rope3d_at(plan["first_frame"] - h, moving, x["q"][st], x["k"][st])
            if ev is not None:
                ev[st][0].record()
            s.window_attention(st, x["q"][st], x["k"][st], x["v"][st], moving, out=x["o"])
            if ev is not None:
                ev[st][1].record()

    for i in range(max(args.warmup, 3)):
        chunk(*sessions[i % 2], 1 + i)
    torch.cuda.synchronize()
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    evs = [[mk() for _ in range(base.n_steps)] for _ in range(args.steps)]
    t0, t1 = mk()
    with Clocks(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clk:
        t0.record()
        for i in range(args.steps):
            chunk(*sessions[i % 2], 1 + i, evs[i])
        t1.record()
        torch.cuda.synchronize()
    # the prefix pass of a first window: prefix and moving rows in one launch
    pe = mk()
    s, x = sessions[0]
    for _ in range(3):
        s.window_attention(0, x["qp"], x["k"][0], x["v"][0], moving, with_prefix=True, out=x["op"])
    torch.cuda.synchronize()
    pe[0].record()
    s.window_attention(0, x["qp"], x["k"][0], x["v"][0], moving, with_prefix=True, out=x["op"])
    pe[1].record()
    torch.cuda.synchronize()
    for s, _ in sessions:
        if s.error_status() != 0:
            raise RuntimeError("device error word set during the bench")
    elapsed = t0.elapsed_time(t1) / 1e3
    attn_ms = statistics.mean(a.elapsed_time(b) for ev in evs for a, b in ev)
    fl = 4.0 * H * M * (S + M) * d
    fl_pre = fl + 4.0 * H * S * S * d
    achieved = fl / (attn_ms / 1e3) / 1e12
    peak_tf, _, peak_kind = _peaks()
    pre_ms = pe[0].elapsed_time(pe[1])
    out = {
        "metric": "page-faithful window attention TFLOP/s and ms per chunk on 1 GB300", "value": round(achieved, 2),
        "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_chunk": round(elapsed / args.steps * 1e3, 4), "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "832x480 latent frames (24x128, 30x52 grid, S=2072 prefix rows), the pages' "
                               "window: per chunk 5 latent frames of moving rows (recomputed history + chunk, "
                               "7800 rows) over the bank and themselves; one step = one chunk: 2 x (RoPE at the "
                               "rows' frame times + window attention)",
                   "lq": M, "lk": S + M, "l2": "two sessions used alternately"},
        "attention_ms_per_denoise_step": round(attn_ms, 4),
        "prefix_pass": {"ms": round(pre_ms, 4), "rows": S + M,
                        "tflops": round(fl_pre / (pre_ms / 1e3) / 1e12, 2),
                        "what": "first window: 2072 prefix rows over the bank alone + 7800 moving rows, one launch"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tf, 4), "kernel": "attn_kernel (sr_window_attention)",
                     "peak_kind": f"{peak_kind} bf16 dense burst"},
        "cpu_baseline": _oracle_line(*_oracle_attention_rate([(M, S + M)], d),
                                     f"one denoising step's window attention ({M} moving rows x {S + M} keys)"),
        "clocks": clk.summary(),
        "gpu_launches": 4 * args.steps,
    }
    print(json.dumps(out), flush=True)


def run_graph(args):
    """Per-chunk sequence (2 x (RoPE + attention) + commit) issued eagerly
    through the device-state calls, against one CUDA-graph replay of the same
    sequence, in steady state (ring full). Two shapes: the 832x480 chunk, and a
    small one (4 heads x 64, 6x10 tokens per frame, 64 sink rows, W = 4) where
    launch and host overhead dominate. Reports device ms per chunk (CUDA events
    around K chunks) and host microseconds to issue one chunk."""
    import chunked_kv_cache_gb300 as sr
    world, rank, local = _dist()
    if rank != 0:
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from chunked_kv_cache_gb300 import build
    build.build()
    shapes = {"832x480": syn.SHAPES[2], "small 4x64 6x10 S=64 W=4": syn.SHAPES[1]}
    results = {}
    for name, sh in shapes.items():
        T, H, d, F, W = sh.tokens_per_frame, sh.n_heads, sh.head_dim, sh.chunk_frames, sh.window_frames
        sink = lambda tid: syn.device_normal_bf16((sh.n_steps, sh.n_sink, H, d), dev, 7, 0, 0, 0, tid)
        s = sr.Session(H, d, sh.grid_h, sh.grid_w, F, W, sh.n_sink, sh.n_steps, sink_k=sink(syn.T_SINK_K),
                       sink_v=sink(syn.T_SINK_V), device_state=True, device=dev)
        x = syn.chunk_inputs_device(sh, 7, dev, chunk=1)
        o = [torch.empty_like(x["q"][0]) for _ in range(sh.n_steps)]

        def chunk():
            for st in range(sh.n_steps):
                s.rope3d_qk_dev(x["q"][st], x["k"][st], F)
                s.chunk_attention_dev(st, x["q"][st], x["k"][st], x["v"][st], F, out=o[st])
            s.cache_commit_dev(x["clean_k"], x["clean_v"], F)

        for _ in range(W // F + max(args.warmup, 3)):      # fill the ring, then warm up
            chunk()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chunk()
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        res = {}
        for mode, fn in (("eager", chunk), ("graph", g.replay)):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            h0 = time.perf_counter()
            for _ in range(args.steps):
                fn()
            host_us = (time.perf_counter() - h0) / args.steps * 1e6
            b.record()
            torch.cuda.synchronize()
            res[mode] = {"ms_per_chunk": round(a.elapsed_time(b) / args.steps, 4), "host_us_per_chunk": round(host_us, 1)}
        if s.error_status() != 0:
            raise RuntimeError("device error word set during the bench")
        res["speedup"] = round(res["eager"]["ms_per_chunk"] / res["graph"]["ms_per_chunk"], 3)
        results[name] = res
        s.close()
    main = results["832x480"]
    sh = shapes["832x480"]
    lk = sh.lk(sh.window_frames)
    rate, done, used = _oracle_attention_rate([(sh.lq, lk)], sh.head_dim)
    chunk_ms = sh.n_steps * 4.0 * sh.n_heads * sh.lq * lk * sh.head_dim / rate * 1e3
    out = {
        "metric": "per-chunk time, eager calls vs CUDA-graph replay (device-resident chunk state), 1 GB300",
        "value": main["graph"]["ms_per_chunk"], "unit": "ms/chunk", "higher_is_better": False, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "steady state (ring full), one step = one chunk: 2 x (RoPE-3D + chunk attention) + "
                               "ring commit through the *_dev calls; eager vs one graph replay"},
        "shapes": results,
        "cpu_baseline": _oracle_line(rate, done, used, f"one 832x480 denoising step ({sh.lq} queries x {lk} keys); "
                                     "ms per chunk extrapolated to all heads and both steps, attention only",
                                     value=round(chunk_ms, 1), unit="ms/chunk"),
        "gpu_launches": 6 * args.steps,
    }
    print(json.dumps(out), flush=True)


def run_decoder(args):
    """The streaming decoder's window attention, one layer at a time, with a
    full cache (4 frames) and 5 global tokens: every 16x16-token window's 2-frame
    chunk (512 rows for a full window) over global tokens + its 4 cached frames +
    its chunk (1541 keys for a full window). Latent grids of the 720p and the
    pages' 768x1344 streams; 16 heads x 128 (a synthetic model shape: the pages
    give no head count). Plain and shifted layers (the shifted one has partial
    windows at the edges). A layer per chunk = the window gather of frame-major
    Q, K, V with RoPE (one launch), the batched attention (one launch) and the
    commit of the clean K, V into every window's ring (one launch); each part is
    also timed alone."""
    world, rank, local = _dist()
    if rank != 0:
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from chunked_kv_cache_gb300 import build
    build.build()
    from chunked_kv_cache_gb300.decoder import DecoderWindowLayer
    H, d, G, F = 16, 128, 5, 2
    grids = {"720p (45x80 tokens)": (45, 80), "768x1344 (48x84 tokens)": (48, 84)}
    results, lay_fl = {}, {}
    peak_tf, peak_gbs, peak_kind = _peaks()

    def timed(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps

    def replay_ms(fn):
        """Device time of one CUDA-graph replay of fn's launches (no host work per call)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        return timed(g.replay)

    for gname, (gh, gw) in grids.items():
        for shifted in (False, True):
            lay = DecoderWindowLayer(gh, gw, H, d, G, shifted=shifted, chunk_frames=F, device=dev)
            dims = (F, gh, gw, H, d)
            mk = lambda tid: syn.device_normal_bf16(dims, dev, 8, int(shifted), 0, 0, tid)
            q, k, v = mk(syn.T_Q), mk(syn.T_K), mk(syn.T_V)
            ck, cv = mk(syn.T_CLEAN_K), mk(syn.T_CLEAN_V)
            lay.set_global(syn.device_normal_bf16((G, H, d), dev, 8, 0, 0, 0, syn.T_SINK_K),
                           syn.device_normal_bf16((G, H, d), dev, 8, 0, 0, 0, syn.T_SINK_V))
            for _ in range(2):                     # fill the 4-frame caches
                lay.commit(ck, cv)
            packed = tuple(torch.empty((lay.rows, H, d), dtype=torch.bfloat16, device=dev) for _ in range(3))
            o = torch.empty_like(packed[0])

            def layer():
                qp, kp, vp = lay.gather_rope(q, k, v, out=packed)
                lay.attention(qp, kp, vp, out=o)
                lay.commit(ck, cv)

            for _ in range(max(args.warmup, 3)):
                layer()
            torch.cuda.synchronize()
            eager_ms = timed(layer)
            layer_ms = replay_ms(layer)
            gather_ms = replay_ms(lambda: lay.gather_rope(q, k, v, out=packed))
            attn_ms = replay_ms(lambda: lay.attention(*packed, out=o))
            commit_ms = replay_ms(lambda: lay.commit(ck, cv))
            fl = sum(4.0 * H * s.lq * (G + 6 * s.T) * d for s in lay.sessions)
            tok_bytes = F * gh * gw * H * d * 2                 # one tensor of the chunk
            gather_bytes, commit_bytes = 6 * tok_bytes, 4 * tok_bytes
            full = [s for s in lay.sessions if s.T == 256]
            name = f"{gname}, {'shifted' if shifted else 'plain'} layer"
            lay_fl[name] = fl
            results[name] = {
                "windows": len(lay.windows), "full_windows": len(full),
                "launches": len(lay.groups) + 2 * len(lay.layer_groups),
                "ms_per_layer": round(layer_ms, 4), "eager_ms_per_layer": round(eager_ms, 4),
                "attention_ms": round(attn_ms, 4), "attention_tflops": round(fl / (attn_ms / 1e3) / 1e12, 2),
                "gather_rope_us": round(gather_ms * 1e3, 2),
                "gather_rope_GBs": round(gather_bytes / (gather_ms / 1e3) / 1e9, 1),
                "gather_rope_frac_hbm": round(gather_bytes / (gather_ms / 1e3) / 1e9 / peak_gbs, 4),
                "commit_us": round(commit_ms * 1e3, 2),
                "commit_GBs": round(commit_bytes / (commit_ms / 1e3) / 1e9, 1),
                "commit_frac_hbm": round(commit_bytes / (commit_ms / 1e3) / 1e9 / peak_gbs, 4),
                "share_of_layer": {"gather_rope": round(gather_ms / layer_ms, 3),
                                   "attention": round(attn_ms / layer_ms, 3),
                                   "commit": round(commit_ms / layer_ms, 3)}}
            if lay.error_status() != 0:
                raise RuntimeError("device error word set during the bench")
            lay.close()
    key = "768x1344 (48x84 tokens), shifted layer"
    rate, done, used = _oracle_attention_rate([(512, G + 6 * 256)], d)
    out = {
        "metric": "decoder window-attention layer ms on 1 GB300 (window gather + RoPE, attention, cache commit)",
        "value": results[key]["ms_per_layer"],
        "unit": "ms/layer", "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "streaming decoder layer: 16x16-token windows, 2-frame chunk, 4 cached frames, "
                               "5 global tokens, 16 heads x 128 (synthetic); frame-major Q, K, V gathered per "
                               "window with RoPE in one launch, every window's attention in one launch (at most "
                               "24 windows), every window's cache commit in one launch; full cache; ms_per_layer "
                               "from a CUDA-graph replay of the layer's launches (eager_ms_per_layer: issued call "
                               "by call); each part also replayed alone"},
        "layers": results,
        "context": "pages: FlexAttention with a block mask, 6 ms per layer on GB200 (their 1.62B decoder)",
        "roofline": {"bound": "tensor", "achieved": results[key]["attention_tflops"], "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(results[key]["attention_tflops"] / peak_tf, 4),
                     "kernel": "attn_kernel<128,24> (sr_chunk_attention_batch)",
                     "peak_kind": f"{peak_kind} bf16 dense burst"},
        "cpu_baseline": _oracle_line(rate, done, used, "one full window (512 queries x 1541 keys); ms per layer "
                                     "extrapolated to every window and head of the " + key + " (attention only)",
                                     value=round(lay_fl[key] / rate * 1e3, 2), unit="ms/layer"),
        "gpu_launches": sum(v["launches"] for v in results.values()) * args.steps * 3,
    }
    print(json.dumps(out), flush=True)


def run_batch(args):
    """The multi-session serving batch: 8 independent 832x480 sessions whose
    rings hold 0, 1, 2, 3, 4, 5, 6 and 6 frames (ragged key lengths), their
    chunks packed along the rows and attended in one launch per denoising
    step. Reports aggregate TFLOP/s of the batched step and each session's
    step run alone, for comparison."""
    import chunked_kv_cache_gb300 as sr
    world, rank, local = _dist()
    if rank != 0:
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from chunked_kv_cache_gb300 import build
    build.build()
    base = syn.SHAPES[2]
    T, H, d, S, W, F = base.tokens_per_frame, base.n_heads, base.head_dim, base.n_sink, base.window_frames, \
        base.chunk_frames
    fills = [0, 1, 2, 3, 4, 5, 6, 6]
    sessions = []
    for sid, fill in enumerate(fills):
        sink = lambda tid: syn.device_normal_bf16((base.n_steps, S, H, d), dev, 9, sid, 0, 0, tid)
        s = sr.Session(H, d, base.grid_h, base.grid_w, F, W, S, base.n_steps, sink_k=sink(syn.T_SINK_K),
                       sink_v=sink(syn.T_SINK_V), device=dev)
        if fill:
            s.ring_k.copy_(syn.device_normal_bf16((W * T, H, d), dev, 9, sid, 1, 0, syn.T_K))
            s.ring_v.copy_(syn.device_normal_bf16((W * T, H, d), dev, 9, sid, 1, 0, syn.T_V))
            s.slot_frame.copy_(torch.tensor([f if f < fill else -1 for f in range(W)], dtype=torch.int32))
            s.restore(fill)
        sessions.append(s)
    rows = F * T * len(fills)
    mk = lambda tid: syn.device_normal_bf16((rows, H, d), dev, 9, 99, 2, 0, tid)
    q, k, v = mk(syn.T_Q), mk(syn.T_K), mk(syn.T_V)
    o = torch.empty_like(q)
    lq = F * T

    def timed(fn, reps):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    with Clocks(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clk:
        batch_ms = timed(lambda: sr.chunk_attention_batch(sessions, 0, q, k, v, out=o), args.steps)
    alone = []
    for i, s in enumerate(sessions):
        sl = slice(i * lq, (i + 1) * lq)
        alone.append(timed(lambda: s.chunk_attention(0, q[sl], k[sl], v[sl], out=o[sl]), max(5, args.steps // 3)))
    for s in sessions:
        if s.error_status() != 0:
            raise RuntimeError("device error word set during the bench")
    lks = [S + f * T + lq for f in fills]
    fl = sum(4.0 * H * lq * lk * d for lk in lks)
    achieved = fl / (batch_ms / 1e3) / 1e12
    peak_tf, _, peak_kind = _peaks()
    rate, done, used = _oracle_attention_rate([(lq, lk) for lk in lks], d)
    out = {
        "metric": "multi-session batch: chunk-attention TFLOP/s of one batched step on 1 GB300", "value": round(achieved, 2),
        "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "8 independent 832x480 sessions (24x128, 30x52 grid, S=2072, W=6) with ring fills "
                               "0,1,2,3,4,5,6,6 frames, chunks packed along the rows, one launch per denoising step",
                   "lq_total": rows, "lk": lks},
        "batch_ms_per_step": round(batch_ms, 4),
        "alone_ms_per_step": [round(x, 4) for x in alone],
        "alone_sum_ms": round(sum(alone), 4),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tf, 4), "kernel": "attn_kernel<128,24> (sr_chunk_attention_batch)",
                     "peak_kind": f"{peak_kind} bf16 dense burst"},
        "cpu_baseline": _oracle_line(rate, done, used, "one denoising step of each session, in turn"),
        "clocks": clk.summary(),
        "gpu_launches": (args.steps + max(args.warmup, 3)) + len(fills) * (max(5, args.steps // 3) + max(args.warmup, 3)),
    }
    print(json.dumps(out), flush=True)


def run_long(args):
    """A long session at the 832x480 shape: 240 consecutive chunks from an empty
    ring (2 x (RoPE + attention) + commit each), the ring filling and then
    evicting. Reports the steady-state chunk time (chunks from W/F on) and
    checks the slot table against its closed form at the end."""
    import chunked_kv_cache_gb300 as sr
    world, rank, local = _dist()
    if rank != 0:
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from chunked_kv_cache_gb300 import build
    build.build()
    base = syn.SHAPES[2]
    T, H, d, S, W, F = base.tokens_per_frame, base.n_heads, base.head_dim, base.n_sink, base.window_frames, \
        base.chunk_frames
    n_chunks = 240
    sink = lambda tid: syn.device_normal_bf16((base.n_steps, S, H, d), dev, 10, 0, 0, 0, tid)
    s = sr.Session(H, d, base.grid_h, base.grid_w, F, W, S, base.n_steps, sink_k=sink(syn.T_SINK_K),
                   sink_v=sink(syn.T_SINK_V), device=dev)
    xs = [syn.chunk_inputs_device(base, 10, dev, chunk=c) for c in range(4)]   # rotated through the stream
    o = torch.empty_like(xs[0]["q"][0])
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    evs = [mk() for _ in range(n_chunks)]
    with Clocks(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clk:
        for c in range(n_chunks):
            x = xs[c % len(xs)]
            evs[c][0].record()
            for st in range(base.n_steps):
                s.rope3d_qk(x["q"][st], x["k"][st])
                s.chunk_attention(st, x["q"][st], x["k"][st], x["v"][st], out=o)
            s.cache_commit(x["clean_k"], x["clean_v"])
            evs[c][1].record()
        torch.cuda.synchronize()
    if s.error_status() != 0:
        raise RuntimeError("device error word set during the bench")
    n = s.frames
    want = [max((g for g in range(n) if g % W == slot), default=-1) for slot in range(W)]
    slots_ok = s.slot_frame.cpu().tolist() == want and n == n_chunks * F
    ms = [a.elapsed_time(b) for a, b in evs]
    first_full = (W + F - 1) // F
    steady = ms[first_full:]
    lk_full = S + W * T + F * T
    fl_chunk = base.n_steps * 4.0 * H * F * T * lk_full * d
    steady_ms = statistics.median(steady)
    peak_tf, _, peak_kind = _peaks()
    achieved = fl_chunk / (steady_ms / 1e3) / 1e12
    rate, done, used = _oracle_attention_rate([(F * T, lk_full)], d)
    out = {
        "metric": "long session: steady-state ms per chunk over 240 chunks on 1 GB300", "value": round(steady_ms, 4),
        "unit": "ms/chunk", "n_gpus": 1, "steps": n_chunks, "warmup": 0, "higher_is_better": False,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "832x480 session (24x128, 30x52 grid, S=2072, W=6), 240 consecutive chunks from an "
                               "empty ring, one chunk = 2 x (RoPE-3D + chunk attention) + ring commit"},
        "first_chunks_ms": [round(x, 4) for x in ms[:first_full + 1]],
        "steady_ms_p10_p50_p90": [round(float(np.percentile(steady, q)), 4) for q in (10, 50, 90)],
        "all_chunks_mean_ms": round(statistics.mean(ms), 4),
        "slot_table_closed_form": slots_ok,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tf, 4), "what": "whole chunk (attention FLOPs) in steady state",
                     "peak_kind": f"{peak_kind} bf16 dense burst"},
        "cpu_baseline": _oracle_line(rate, done, used, f"one steady-state denoising step ({F * T} queries x "
                                     f"{lk_full} keys); ms per chunk extrapolated to all heads and both steps",
                                     value=round(fl_chunk / rate * 1e3, 1), unit="ms/chunk"),
        "clocks": clk.summary(),
        "gpu_launches": 5 * n_chunks,
    }
    if not slots_ok:
        raise RuntimeError("slot table does not match its closed form")
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, choices=[2, 3], default=3,
                    help="3: the 720p chunk (the largest single-GPU workload, default); 2: the 832x480 chunk")
    ap.add_argument("--chunks-per-step", type=int, default=0,
                    help="chunks per bench step of the steady workload (0: about 50 ms worth)")
    ap.add_argument("--workload", choices=["steady", "rhythm", "window", "graph", "decoder", "batch", "long"],
                    default="steady",
                    help="steady: the headline chunk workload; rhythm: the pages' 3/2-latent unit rhythm; "
                         "window: the page-faithful window (recomputed history rows as queries); "
                         "graph: eager calls vs CUDA-graph replay of a chunk; decoder: the streaming decoder's "
                         "window attention; batch: 8 ragged 832x480 sessions in one launch; long: 240 chunks of "
                         "one 832x480 session from an empty ring")
    ap.add_argument("--profile", action="store_true",
                    help="under a profiler: skip the end-to-end and CPU-baseline legs (their numbers are not reported)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "rhythm":
        run_rhythm(args)
    elif args.workload == "window":
        run_window(args)
    elif args.workload == "graph":
        run_graph(args)
    elif args.workload == "decoder":
        run_decoder(args)
    elif args.workload == "batch":
        run_batch(args)
    elif args.workload == "long":
        run_long(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
