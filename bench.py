"""Benchmark: causal-adjusted attention forward TFLOP/s on one GB300 (per rank).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step is one pass of the whole hot path (``ra_ring_sim_fwd`` for the workload's ring
size: attention steps, causal tile skipping and the in-kernel LSE merge) over one
batch of seeded synthetic inputs resident in HBM.  Each timed step is bracketed by CUDA
events on the launching stream; between steps a 256 MiB buffer (larger than the 129 MB
L2) is rewritten to flush L2.  ``value`` = FLOPs of all steps of all ranks / the slowest
rank's summed step time.  Under torchrun every rank runs an independent replica (no data
exchange), so scaling is weak.

``--impl reference`` times the oracle (plain fp64 C, all host cores) on a bounded sample
of the same workload and prints the same JSON shape with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

DEFAULT_WORKLOAD = "dense_causal_b2h32n4k"
METRIC = "attention fwd TFLOP/s (causal-adjusted) and % of GB300 dense BF16 peak"
KERNEL_SRC = os.path.join(ROOT, "exact_long_context_gb300", "csrc", "attn_tc.cu")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float) -> float:
    """The largest value of x over all ranks (identity without a process group)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def emit(args, line: dict):
    """The run's one JSON line on stdout, and appended to the --results JSON-lines file when
    one is given (one record per run: config, rates, roofline, baselines, clocks)."""
    text = json.dumps(line)
    print(text, flush=True)
    if getattr(args, "results", None):
        with open(args.results, "a") as f:
            f.write(text + "\n")


def whole_job_rate(units_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Units processed by all ranks per second of the slowest rank's timed region."""
    return units_per_rank_step * steps * world / (max_ms * 1e-3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p.get("bf16_tflops", 1900.0), p.get("hbm_gbs", 6800.0), "measured"
    return 1900.0, 6800.0, "fallback"


# Nominal dense bf16 tensor rates per GPU, from NVIDIA's published datasheets, where the
# FP16/BF16 figures are quoted with 2:4 structured sparsity (dense is half):
#   HGX B300 (8 GPUs): 36 PFLOP/s sparse -> 2.25 PFLOP/s dense per GPU;
#   GB300 NVL72 (72 GPUs): 360 PFLOP/s sparse -> 2.5 PFLOP/s dense per GPU.
SPEC_DENSE_BF16_TFLOPS = {"hgx_b300": 2250.0, "gb300_nvl72": 2500.0}
# workloads whose oracle is also timed on one core (the tiny and the dense workload)
SINGLE_CORE_WORKLOADS = ("tiny_ring4_fp32", "dense_causal_b2h32n4k")


def bf16_peak(launch_ms: float):
    """The measured bf16 rate a kernel is held to: the burst GEMM rate for a kernel timed
    alone for a short time, the sustained (power-capped) one for a launch of 50 ms or more."""
    burst, _, kind = peaks()
    if kind == "measured" and launch_ms >= 50.0:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            sus = json.load(f).get("bf16_tflops_sustained")
        if sus:
            return sus, "measured sustained"
    return burst, f"{kind} burst"


def kernel_flops(w, kernel: str) -> float:
    """Algorithmic FLOPs per step of one kernel of the path.  Forward attention: 4 d per
    visible (query, key) pair (two products).  Backward: the dQ kernel makes three products
    per visible pair (S, dP, dQ: 6 d FLOP), the dK/dV kernel four (S^T, dP^T, dV, dK: 8 d);
    the D = rowsum(dO * O) pass is bandwidth work (0 FLOP here)."""
    f = w.flops()  # 4 d per visible pair
    if kernel.startswith("attn_"):
        return f
    if kernel.startswith("bwd_dq"):
        return 1.5 * f
    if kernel.startswith("bwd_dkdv"):
        return 2.0 * f
    return 0.0


def peak_fractions(tflops: float) -> dict:
    """Percent of the measured burst and sustained bf16 GEMM rates and of the nominal
    dense bf16 rates, for a TFLOP/s figure."""
    burst, _, kind = peaks()
    sustained = None
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            sustained = json.load(f).get("bf16_tflops_sustained")
    out = {f"of_{kind}_burst": round(100 * tflops / burst, 2)}
    for name, tf in SPEC_DENSE_BF16_TFLOPS.items():
        out[f"of_nominal_dense_bf16_{name}"] = round(100 * tflops / tf, 2)
    if sustained:
        out["of_measured_sustained"] = round(100 * tflops / sustained, 2)
    return out


def kernel_hash():
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(workload: str):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu summary of this
    workload, if that summary was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"attn_tc_{workload}.json")
    try:
        with open(path) as f:
            prof = json.load(f)
    except (OSError, ValueError):
        return None
    if prof.get("workload") != workload or prof.get("kernel_src_sha256_16") != kernel_hash():
        return None
    return prof.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if self.t0 is not None and self.t0 - 0.15 <= ts <= self.t1 + 0.15]
        use = inside if inside else rows[-3:]
        if not use:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(p[2]) for p in use]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in use:
            for name, val in zip(names, p[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(num(p[3]) for p in use),
                "reasons": sorted(reasons), "samples": len(use),
                "power_w_max": max(num(p[4]) for p in use)}


def run_ours(args, w, ws, rank, local):
    from exact_long_context_gb300 import ra, synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    q, k, v = synth.workload_inputs(w, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=dev)
    need = ra.ring_sim_workspace_bytes(q, w.ring_size)
    wsbuf = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    varlen = isinstance(w, synth.VarlenWorkload)
    cu = w.cu_seqlens() if varlen else None
    bwd = args.pass_ == "bwd"
    if bwd:
        if varlen:
            raise SystemExit("--pass bwd times the ring (or single-pass) backward, not packed batches")
        ra.ring_sim_fwd(q, k, v, w.ring_size, w.layout, causal=w.causal, scale=w.scale, o=o, lse=lse,
                        workspace=wsbuf if need else None, stream=stream)
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed + 1000)
        dout = torch.randn(q.shape, generator=g, device=dev).to(q.dtype)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bws = torch.empty(max(16, ra.ring_sim_bwd_workspace_bytes(q, k, w.ring_size)), dtype=torch.uint8,
                          device=dev)

    def step():
        if bwd:
            ra.ring_sim_bwd(q, k, v, o, lse, dout, w.ring_size, w.layout, causal=w.causal, scale=w.scale,
                            dq=dq, dk=dk, dv=dv, workspace=bws, stream=stream)
            return
        if varlen:
            ra.attn_varlen_fwd(q, k, v, cu, causal=w.causal, scale=w.scale, o=o, lse=lse,
                               stream=stream)
        else:
            ra.ring_sim_fwd(q, k, v, w.ring_size, w.layout, causal=w.causal, scale=w.scale, o=o,
                            lse=lse, workspace=wsbuf if need else None, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    ra.check(stream)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    launches0 = ra.launch_count()
    clocks.mark("t0")
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clocks.mark("t1")
    if ws > 1:
        torch.distributed.barrier()
    launches = ra.launch_count() - launches0
    ra.check(stream)
    clk = clocks.stop()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(float(sum(times)))
    ms_per_step = total_ms / args.steps
    # backward: the conventional 2.5x of the forward (five products of the forward's size)
    flops = w.flops() * (2.5 if bwd else 1.0)
    value = whole_job_rate(flops, args.steps, ws, total_ms) / 1e12
    launches_per_step = launches / args.steps

    # end to end through the public call: pinned host inputs -> device -> host result
    e2e = None
    if args.e2e_steps > 0 and not bwd:
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        if not varlen:
            # the library's host-buffer call: it stages through device memory and overlaps
            # the copies in and out with the kernels, head group by head group
            hws = torch.empty(ra.ring_sim_fwd_host_workspace_bytes(hq, hk, w.ring_size), dtype=torch.uint8,
                              device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def e2e_step():
            if not varlen:
                ra.ring_sim_fwd_host(hq, hk, hv, w.ring_size, w.layout, causal=w.causal, scale=w.scale,
                                     o=ho, lse=hl, workspace=hws, stream=stream)
                return
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            ra.attn_varlen_fwd(dq, dk, dv, cu, causal=w.causal, scale=w.scale, o=o, lse=lse, stream=stream)
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        etot = 0.0
        for _ in range(args.e2e_steps):
            flush.zero_()
            es.record(stream)
            e2e_step()
            ee.record(stream)
            ee.synchronize()
            etot += es.elapsed_time(ee)
        ra.check(stream)
        etot = max_over_ranks(etot)
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
        e2e = {"value": round(flops * args.e2e_steps * ws / (etot * 1e-3) / 1e12, 2),
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(etot / args.e2e_steps, 4)}

    # The dominant kernel on its own: a few more steps (outside the timed region, L2 flushed
    # between steps as there) with every launch bracketed by its own CUDA events on the
    # launching stream, inside the library (ra_debug_time_launches).
    ra.time_launches(True)
    nk = max(3, min(10, args.steps))
    for _ in range(nk):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    ra.time_launches(False)
    per = {}
    for name, ms in ra.launch_times():
        per.setdefault(name, []).append(ms)
    ra.check(stream)
    dom = max(per, key=lambda n: sum(per[n]))
    dom_ms = sum(per[dom]) / nk  # per step
    dom_launch_ms = sum(per[dom]) / len(per[dom])
    achieved = kernel_flops(w, dom) / (dom_ms * 1e-3) / 1e12
    peak_tf, peak_kind = bf16_peak(dom_launch_ms)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 2), "peak": peak_tf,
                "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                "traffic": None if bwd else profiled_traffic(w.name), "peak_kind": peak_kind,
                "launches_per_step": round(len(per[dom]) / nk, 2), "ms_per_launch": round(dom_launch_ms, 5),
                "kernels_ms_per_step": {n: round(sum(t) / nk, 5) for n, t in per.items()}}
    return {
        "value": round(value, 2), "ms_per_step": round(ms_per_step, 5), "e2e": e2e,
        "roofline": roofline, "clocks": clk, "gpu_launches": launches,
        "wall_s_timed_region": round(wall, 4),
        "tokens_per_s": round(w.B * w.N * args.steps * ws / (total_ms * 1e-3), 1),
    }


def run_hbm_pass(args, w, ws, rank, local):
    """HBM-bound calls: the standalone LSE merge on the workload's whole running output
    (fp32 o_acc [B,Hq,N,D], bf16 o_blk, 1292 algorithmic bytes per row at D = 128) or the
    Ulysses exchange of the workload's Q (read + write of every element)."""
    from exact_long_context_gb300 import ra

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 7)
    stream = torch.cuda.current_stream(dev)
    if args.pass_ == "merge":
        shape = (w.B, w.Hq, w.N, w.D)
        o_acc = torch.randn(shape, generator=g, device=dev)
        o_blk = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
        lse_acc = torch.randn(shape[:3], generator=g, device=dev)
        lse_blk = torch.randn(shape[:3], generator=g, device=dev)
        rows = w.B * w.Hq * w.N
        nbytes = rows * (w.D * 4 * 2 + w.D * 2 + 4 * 3)

        def step():
            ra.lse_merge(o_acc, lse_acc, o_blk, lse_blk, stream=stream)
    else:
        sp = max(1, min(8, w.Hq))
        while w.Hq % sp or w.N % sp:
            sp -= 1
        x = torch.randn((sp, w.N // sp, w.Hq, w.D), generator=g, device=dev).to(w.dtype)
        y = torch.empty((sp, w.N, w.Hq // sp, w.D), dtype=w.dtype, device=dev)
        nbytes = 2 * x.numel() * x.element_size()

        def step():
            ra.ulysses_all_to_all(x, sp, to_heads=True, out=y, stream=stream)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        step()
    ra.check(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = ra.launch_count()
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    launches = ra.launch_count() - launches0
    ra.check(stream)
    total_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)))
    gbs = whole_job_rate(nbytes, args.steps, ws, total_ms) / 1e9
    _, hbm, kind = peaks()
    per_rank = gbs / ws
    return {"value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(total_ms / args.steps, 5),
            "gpu_launches": launches, "higher_is_better": True,
            "roofline": {"bound": "hbm", "achieved": round(per_rank, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(per_rank / hbm, 4), "traffic": None, "peak_kind": kind},
            "bytes_per_step": nbytes}


def run_hostlink(args, ws, rank, local):
    """Pinned host <-> device copy rates (one cudaMemcpyAsync per copy, through torch's
    non-blocking copy_) at 8 MiB .. 1 GiB, each direction alone and both at once on two
    streams: the bound of the end-to-end figure, whose step copies q, k, v in and o, lse out."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    out = {}
    for mib in (8, 32, 128, 512, 1024):
        n = mib << 20
        h_in = torch.empty(n, dtype=torch.uint8).pin_memory()
        h_out = torch.empty(n, dtype=torch.uint8).pin_memory()
        d_a = torch.empty(n, dtype=torch.uint8, device=dev)
        d_b = torch.empty(n, dtype=torch.uint8, device=dev)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        reps = max(3, min(20, (2048 // mib)))

        def timed(fn):
            for _ in range(2):
                fn()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            for _ in range(reps):
                fn()
            torch.cuda.synchronize(dev)
            return (time.perf_counter() - t0) / reps

        def h2d():
            with torch.cuda.stream(s_in):
                d_a.copy_(h_in, non_blocking=True)

        def d2h():
            with torch.cuda.stream(s_out):
                h_out.copy_(d_b, non_blocking=True)

        def both():
            h2d()
            d2h()

        t_in, t_out, t_both = timed(h2d), timed(d2h), timed(both)
        out[f"{mib}MiB"] = {"h2d_gbs": round(n / t_in / 1e9, 1), "d2h_gbs": round(n / t_out / 1e9, 1),
                            "both_gbs_each": round(n / t_both / 1e9, 1)}
        del h_in, h_out, d_a, d_b
    return {"value": max(v["h2d_gbs"] for v in out.values()), "unit": "GB/s", "sizes": out,
            "how": "wall time of reps back-to-back cudaMemcpyAsync copies of pinned memory per size"}


def host_cpu_desc():
    """The host CPU the oracle runs on: machine, model (or Arm part number) and the cores
    this process may use."""
    import platform
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key, _, val = ln.partition(":")
                key = key.strip().lower()
                if key == "model name" or (key == "cpu part" and not model):
                    model = (val.strip() if key == "model name" else f"CPU part {val.strip()}")
                    if key == "model name":
                        break
    except OSError:
        pass
    avail = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return f"{platform.machine()}{', ' + model if model else ''}, {avail} cores available"


def oracle_rate_sample(w, budget_s, seed=0, threads=None):
    """Time the oracle on rows sampled from the workload (all host cores unless `threads`
    is given); returns (flops, seconds, rows, threads)."""
    import oracle
    from exact_long_context_gb300 import synth

    q, k, v = synth.workload_inputs(w, device="cpu")

    def enc(t):
        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()

    qn, kn, vn = enc(q), enc(k), enc(v)
    threads = threads or oracle.default_threads()
    rng = np.random.default_rng(seed)

    def rows_for(n):
        b = rng.integers(0, w.B, n)
        h = rng.integers(0, w.Hq, n)
        i = rng.integers(0, w.N, n)
        return np.stack([b, h, i], 1).astype(np.int64)

    varlen = isinstance(w, synth.VarlenWorkload)
    cu = w.cu_seqlens() if varlen else None

    def run(rows):
        """Oracle over the rows; returns their causal-adjusted FLOPs."""
        if not varlen:
            oracle.attention(qn, kn, vn, w.causal, w.scale, rows=rows, nthreads=threads)
            vis = (rows[:, 2] + 1) if w.causal else np.full(len(rows), w.N)
            return float(np.sum(vis)) * 4.0 * w.D
        seq = np.searchsorted(np.array(cu), rows[:, 2], side="right") - 1
        flops = 0.0
        for s_ in np.unique(seq):
            sel = rows[seq == s_]
            a, b = cu[s_], cu[s_ + 1]
            oracle.attention(qn, kn, vn, w.causal, w.scale, kv_lo=a, kv_hi=b, rows=sel,
                             nthreads=threads)
            vis = (sel[:, 2] - a + 1) if w.causal else np.full(len(sel), b - a)
            flops += float(np.sum(vis)) * 4.0 * w.D
        return flops

    # calibrate on a small batch, then size the timed sample to the budget
    cal = rows_for(max(threads, 8))
    t0 = time.perf_counter()
    run(cal)
    dt = max(time.perf_counter() - t0, 1e-4)
    per_row = dt / len(cal)
    n = int(max(threads, min(200000, budget_s / per_row)))
    rows = rows_for(n)
    t0 = time.perf_counter()
    f = run(rows)
    sec = time.perf_counter() - t0
    return f, sec, len(rows), threads


def run_reference(args, w, ws, rank):
    """The oracle as it stands, on the host cores, a bounded sample per step."""
    if rank != 0:
        return None
    per_step = max(0.05, min(2.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_rate_sample(w, per_step, seed=1)
    tf = tsec = 0.0
    nrows = 0
    threads = 1
    for i in range(args.steps):
        f, s, n, threads = oracle_rate_sample(w, per_step, seed=100 + i)
        tf += f
        tsec += s
        nrows += n
    value = tf / tsec / 1e12
    sample = (f"{nrows} uniformly random query rows of {w.name} over {args.steps} steps "
              f"(fp64 oracle, causal-adjusted FLOPs of the rows' visible keys)")
    return {"value": round(value, 6), "ms_per_step": round(tsec / args.steps * 1e3, 3),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample, "cpu": host_cpu_desc()},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd", "merge", "ulysses", "hostlink"], default="fwd",
                    help="fwd (default): the hot path; bwd: its backward (ring schedule when ring_size > 1); "
                         "merge / ulysses: the HBM-bound LSE merge / Ulysses exchange; hostlink: pinned "
                         "host <-> device copy rates (the end-to-end figure's bound)")
    ap.add_argument("--results", default=None,
                    help="also append the JSON line to this JSON-lines file (rank 0)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from exact_long_context_gb300 import synth

    w = synth.WORKLOADS.get(args.workload) or synth.VARLEN_WORKLOADS[args.workload]
    ws, rank, local = dist_env()
    if ws > 1:
        torch.distributed.init_process_group("nccl" if args.impl == "ours" else "gloo")

    config = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "D": w.D,
              "causal": w.causal, "ring_size": w.ring_size, "layout": w.layout,
              **({"sequences": len(w.lengths())} if isinstance(w, synth.VarlenWorkload) else {}),
              "l2": "flushed between steps (256 MiB write)", "parallelism": f"replicas x{ws}"}
    metric = {"fwd": METRIC, "bwd": METRIC.replace("attention fwd", "attention bwd"),
              "merge": "lse_merge GB/s (algorithmic bytes) and % of measured HBM bandwidth",
              "ulysses": "Ulysses all-to-all GB/s and % of measured HBM bandwidth",
              "hostlink": "pinned host<->device copy GB/s"}[args.pass_]
    line = {"metric": metric, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
            "data": "synthetic (seeded N(0,1), rounded to bf16)", "config": config}

    if args.impl == "reference":
        res = run_reference(args, w, ws, rank)
        if ws > 1:
            torch.distributed.barrier()
        if res is None:
            return
        line.update(res)
        line["impl"] = "reference"
        emit(args, line)
        return

    if args.pass_ == "hostlink":
        if rank == 0:
            line.update(run_hostlink(args, ws, rank, local))
            line["config"] = {"workload": "pinned copies 8 MiB .. 1 GiB"}
            emit(args, line)
        return
    if args.pass_ in ("merge", "ulysses"):
        res = run_hbm_pass(args, w, ws, rank, local)
        if rank == 0:
            line.update(res)
            line["unit"] = "GB/s"
            line["dtype"] = "f32+bf16" if args.pass_ == "merge" else line["dtype"]
            emit(args, line)
        if ws > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return
    res = run_ours(args, w, ws, rank, local)
    if rank == 0:
        line.update(res)
        line["pct_of_peak"] = round(100 * res["roofline"]["frac"], 2)
        if line["unit"] == "TFLOP/s":
            line["pct_of_peaks"] = peak_fractions(line["value"])
        if args.pass_ == "bwd":
            line["cpu_baseline"] = None  # the oracle's timed leg is the forward
            emit(args, line)
            if ws > 1:
                torch.distributed.barrier()
                torch.distributed.destroy_process_group()
            return
        f, sec, nrows, threads = oracle_rate_sample(w, args.cpu_budget_s)
        line["cpu_baseline"] = {
            "value": round(f / sec / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{nrows} uniformly random query rows of {w.name} (fp64 oracle, "
                      f"{sec:.1f} s wall)",
            "cpu": host_cpu_desc()}
        if w.name in SINGLE_CORE_WORKLOADS and args.cpu_budget_s > 0:
            f1, sec1, nrows1, _ = oracle_rate_sample(w, min(5.0, args.cpu_budget_s), seed=1, threads=1)
            line["cpu_baseline"]["single_core"] = {
                "value": round(f1 / sec1 / 1e12, 7), "unit": "TFLOP/s", "cores": 1,
                "sample": f"{nrows1} uniformly random query rows of {w.name} (fp64 oracle, one thread, "
                          f"{sec1:.1f} s wall)"}
        emit(args, line)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
