"""Throughput of non-causal DiT attention on GB300: fused pass and p-chunk ring decomposition.

One step = the whole hot path once over one batch of synthetic input: the
fused attention pass (dit_attn_fwd) and the same attention as p KV chunks
(dit_attn_chunks_fwd: every virtual ring rank's local attention, partial O and
LSE per chunk, in one launch) merged by dit_attn_lse_merge.  The same chunk path
with one dit_attn_chunk_fwd launch per rank (bitwise the same partials) is
reported beside the step.  FLOPs counted per pass: 4*B*H*N^2*D (the two GEMMs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload wan22] [--impl reference]

Prints ONE JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload (weak scaling, no data-path collective); the timed
region is bracketed by a barrier + synchronize and the max over ranks is used.
`--impl reference` times the fp64 CPU oracle (the only reference this path
has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from diffusion_transformer_long_gb300 import synth  # noqa: E402

METRIC = "attention TFLOP/s & % of GB300 BF16 dense peak (H=24,N=27280,D=128)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129e6


def pct(xs):
    """median, min and 90th percentile of per-step times (ms)."""
    ys = sorted(xs)
    return {"median": statistics.median(ys), "min": ys[0],
            "p90": ys[min(len(ys) - 1, int(math.ceil(0.9 * len(ys))) - 1)], "n": len(ys)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_digest() -> str:
    """Digest of the attention kernel's code (comments and blank lines excluded, so that a
    comment edit does not orphan the profile summary taken on the same code)."""
    h = hashlib.sha256()
    for f in ("attn_kernel.cuh", "sm103_ptx.cuh", "attn_fwd.cu"):
        with open(os.path.join(ROOT, "diffusion_transformer_long_gb300", "csrc", f)) as fh:
            for line in fh:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary, if the
    summary was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"attn_fwd_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    digest = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    traffic = re.search(r"dram_bytes_per_launch_full_size:\s*([0-9.eE+]+)", text)
    if not digest or not traffic or digest.group(1) != kernel_source_digest():
        return None
    return float(traffic.group(1))


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock, power and throttle reasons; summary()
    keeps the samples taken between mark_start() and mark_end() (the timed region).  The
    driver refreshes its readings about every 100 ms, so each value appears about twice."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, device_index: int):
        self.proc = None
        self.out = None
        self.t_start = self.t_end = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(device_index)
        self.cmd = ["nvidia-smi", f"--id={ident}", f"--query-gpu={self.FIELDS}",
                    "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t_start = datetime.datetime.now()

    def mark_end(self):
        self.t_end = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)  # the sample covering the region's end
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def rows(self):
        """(time, sm MHz, max MHz, watts or None, [active, hw, hw_thermal, sw_thermal, power_cap])
        for every parsed sample."""
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 9:
                continue
            try:
                when = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                watts = float(parts[3])
            except ValueError:
                watts = None
            rows.append((when, sm, mx, watts, parts[4:]))
        return rows

    def summary(self):
        rows = self.rows()
        if self.t_start is not None and self.t_end is not None:
            inside = [r for r in rows if self.t_start <= r[0] <= self.t_end]
            window = "inside the timed region"
            if not inside:  # a region shorter than the sampling period
                inside = [min(rows, key=lambda r: abs((r[0] - self.t_end).total_seconds()))] \
                    if rows else []
                window = "the sample nearest the timed region's end"
        else:
            inside, window = rows, "whole run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[4][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        watts = [r[3] for r in inside if r[3] is not None]
        sm = [r[1] for r in inside]
        sm_max = max(r[2] for r in inside)
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm),
                "sm_max_mhz": sm_max,
                "frac_samples_below_max": sum(x < sm_max for x in sm) / len(sm),
                "reasons": sorted(reasons), "samples": len(inside),
                "sampling": f"nvidia-smi every {self.PERIOD_MS} ms, {window}",
                "power_w_max": max(watts) if watts else None}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def oracle_sample_tflops(w, q, k, v, target_s: float, rows_cap: int = 100000,
                         threads: int = 0):
    """Times the fp64 oracle on a bounded row sample of workload w (all heads, R query rows),
    on `threads` worker threads (0: every core this process may run on).
    Returns (tflops, seconds, rows_per_head, threads)."""
    import oracle
    threads = threads or len(os.sched_getaffinity(0))
    heads = w.B * w.H
    # calibrate on 2 rows per head
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, rows=list(range(2)), threads=threads)
    dt = max(time.perf_counter() - t0, 1e-3)
    per_row = dt / (2 * heads)
    R = int(max(2, min(rows_cap, target_s / (per_row * heads))))
    R = min(R, w.N)
    rows = synth.sample_rows(w.N, R, edge=min(16, R // 2), seed=w.seed)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, rows=rows, threads=threads)
    secs = time.perf_counter() - t0
    flops = 4.0 * heads * len(rows) * w.N * w.D
    used = oracle.threads_used(threads, heads * len(rows))
    return flops / secs / 1e12, secs, len(rows), used


def run_reference(args):
    """Reference arm: the fp64 CPU oracle on bounded samples of the same workload."""
    dist, rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    w = synth.WORKLOADS[args.workload]
    q, k, v = synth.make_qkv(w)
    per_step = []
    rows_used = threads = 0
    for i in range(args.warmup + args.steps):
        tf, secs, rows_used, threads = oracle_sample_tflops(w, q, k, v, target_s=args.ref_step_s)
        if i >= args.warmup:
            per_step.append((tf, secs))
    value = statistics.median(t for t, _ in per_step)
    ms = statistics.median(s for _, s in per_step) * 1e3
    sample = (f"{w.B * w.H} heads x {rows_used} query rows against all {w.N} keys per step "
              f"(fp64 oracle, one step ~{args.ref_step_s:.0f} s)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; no dataset exists for this path)",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": f"{w.name}: B={w.B} H={w.H} N={w.N} D={w.D} bf16 Q/K/V, non-causal, "
                        f"fused pass + p={w.p} KV chunks ({'/'.join(map(str, sorted(set(w.chunks))))})"
                        f" merged by LSE",
            "B": w.B, "H": w.H, "N": w.N, "D": w.D, "p": w.p, "chunks": list(w.chunks),
            "out_dtype": "fp32", "partial_dtype": "fp32",
            "l2": f"no flush: Q/K/V are {3 * w.B * w.H * w.N * w.D * 2 / 1e6:.0f} MB "
                  f"(> {L2_BYTES / 1e6:.0f} MB L2)" if 3 * w.B * w.H * w.N * w.D * 2 > L2_BYTES
                  else "L2 flushed between steps (256 MB write)",
            "parallelism": "replicas (one independent workload per GPU)"}


def run_gpu(args):
    from diffusion_transformer_long_gb300 import ditattn as da

    dist, rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    q_h, k_h, v_h = synth.make_qkv(w)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    B, H, N, D, p = w.B, w.H, w.N, w.D, w.p
    out_f = torch.empty((B, H, N, D), device=dev, dtype=torch.float32)
    lse_f = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    parts = torch.empty((p, B, H, N, D), device=dev, dtype=torch.float32)
    lses = torch.empty((p, B, H, N), device=dev, dtype=torch.float32)
    out_c = torch.empty_like(out_f)
    lse_c = torch.empty_like(lse_f)
    starts = synth.chunk_starts(w.chunks)
    small = 3 * B * H * N * D * 2 <= L2_BYTES
    flush = torch.empty(int(256e6) // 4, device=dev, dtype=torch.float32) if small else None
    stream = torch.cuda.current_stream(dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    fused_ev, merge_ev, chunk_ev = [], [], []

    def step(record=False):
        if record:
            e0, e1 = ev(), ev()
            e0.record(stream)
        da.attn_fwd(q, k, v, out=out_f, lse=lse_f, scale=w.scale)
        if record:
            e1.record(stream)
            fused_ev.append((e0, e1))
            c0 = ev()
            c0.record(stream)
        da.attn_chunks_fwd(q, k, v, w.chunks, partials=parts, lses=lses, scale=w.scale)
        if record:
            m0, m1 = ev(), ev()
            m0.record(stream)
        da.attn_lse_merge(parts, lses, out=out_c, lse=lse_c)
        if record:
            m1.record(stream)
            merge_ev.append((m0, m1))
            chunk_ev.append((c0, m1))

    launches_per_step = 3
    for _ in range(args.warmup):
        step()
        if flush is not None:
            flush.zero_()
    torch.cuda.synchronize(dev)
    da.check(dev)
    diff = (out_f - out_c).abs().max().item()

    # ---- timed region (device clock) ----
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        barrier(dist)
        torch.cuda.synchronize(dev)
        clk.mark_start()
        t0, t1 = ev(), ev()
        if flush is None:
            t0.record(stream)
            for _ in range(args.steps):
                step(record=True)
            t1.record(stream)
            torch.cuda.synchronize(dev)
            elapsed_ms = t0.elapsed_time(t1)
        else:
            elapsed_ms = 0.0
            for _ in range(args.steps):
                flush.zero_()
                s0, s1 = ev(), ev()
                s0.record(stream)
                step(record=True)
                s1.record(stream)
                torch.cuda.synchronize(dev)
                elapsed_ms += s0.elapsed_time(s1)
        clk.mark_end()
        barrier(dist)
    da.check(dev)
    ms_step = max_over_ranks(dist, elapsed_ms / args.steps)
    fused_all = [a.elapsed_time(b) for a, b in fused_ev]
    chunk_all = [a.elapsed_time(b) for a, b in chunk_ev]
    fused_ms = statistics.mean(fused_all)
    merge_ms = statistics.mean(a.elapsed_time(b) for a, b in merge_ev)
    chunk_ms = statistics.mean(chunk_all)
    fused_ms = max_over_ranks(dist, fused_ms)
    chunk_ms = max_over_ranks(dist, chunk_ms)
    merge_ms = max_over_ranks(dist, merge_ms)
    step_flops = 2 * w.flops  # the fused pass and the chunked pass each compute the attention
    value = step_flops * world / (ms_step * 1e-3) / 1e12

    # ---- small workloads (inputs below L2): warm steps and the step as one CUDA graph ----
    warm_ms = graph_ms = None
    graph_err = None
    if small:
        for _ in range(2):
            step()
        torch.cuda.synchronize(dev)
        w0, w1 = ev(), ev()
        w0.record(stream)
        for _ in range(args.steps):
            step()
        w1.record(stream)
        torch.cuda.synchronize(dev)
        warm_ms = max_over_ranks(dist, w0.elapsed_time(w1) / args.steps)
        try:
            graph = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                step()  # eager once on the capture stream
                torch.cuda.synchronize(dev)
                with torch.cuda.graph(graph, stream=cap):
                    step()
            stream.wait_stream(cap)
            graph.replay()
            torch.cuda.synchronize(dev)
            g0, g1 = ev(), ev()
            g0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            g1.record(stream)
            torch.cuda.synchronize(dev)
            da.check(dev)
            graph_ms = g0.elapsed_time(g1) / args.steps
        except Exception as e:  # reported, not fatal: the eager numbers stand
            graph_err = f"{type(e).__name__}: {str(e).splitlines()[0][:200]}"
        # collectives outside the try: every rank takes part whatever happened locally
        all_ok = sum_over_ranks(dist, 1.0 if graph_ms is not None else 0.0) == world
        slowest = max_over_ranks(dist, graph_ms if graph_ms is not None else 0.0)
        graph_ms = slowest if all_ok else None
        if not all_ok and graph_err is None:
            graph_err = "CUDA-graph capture failed on another rank"

    # ---- chunk-path variants (timed outside the step) ----
    parts16 = torch.empty((p, B, H, N, D), device=dev, dtype=torch.bfloat16)

    def chunk_bf16():
        # bf16 partials (a stated variant), all ranks in one launch
        da.attn_chunks_fwd(q, k, v, w.chunks, partials=parts16, lses=lses, scale=w.scale)
        da.attn_lse_merge(parts16, lses, out=out_c, lse=lse_c)

    def chunk_per_rank():
        # one dit_attn_chunk_fwd launch per virtual rank (the same partials, bit for bit)
        for c, (s, n) in enumerate(zip(starts, w.chunks)):
            da.attn_chunk_fwd(q, k[:, :, s:s + n], v[:, :, s:s + n], out=parts[c], lse=lses[c],
                              scale=w.scale)
        da.attn_lse_merge(parts, lses, out=out_c, lse=lse_c)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        b0, b1 = ev(), ev()
        b0.record(stream)
        n_rep = max(3, args.steps // 3)
        for _ in range(n_rep):
            fn()
        b1.record(stream)
        torch.cuda.synchronize(dev)
        da.check(dev)
        return max_over_ranks(dist, b0.elapsed_time(b1) / n_rep)

    chunk16_ms = timed(chunk_bf16)
    per_rank_ms = timed(chunk_per_rank)
    del parts16

    # ---- the fused pass without the LSE output (O only; bitwise the same O) ----
    out_nl = torch.empty_like(out_f)

    def fused_no_lse():
        da.attn_fwd(q, k, v, out=out_nl, scale=w.scale, with_lse=False)

    no_lse_ms = timed(fused_no_lse)
    no_lse_same = bool(torch.equal(out_nl, out_f))
    del out_nl

    # ---- hop-by-hop ring: each chunk pass merges into the running (O, lse) itself ----
    # The first hop writes the running state (dit_attn_chunk_fwd, fp32), the other p-1 fold
    # their chunk in (dit_attn_chunk_fwd_accumulate): no stacked partials, no merge pass.
    def ring():
        for c, (s, n) in enumerate(zip(starts, w.chunks)):
            kc, vc = k[:, :, s:s + n], v[:, :, s:s + n]
            if c == 0:
                da.attn_chunk_fwd(q, kc, vc, out=out_c, lse=lse_c, scale=w.scale)
            else:
                da.attn_chunk_fwd_accumulate(q, kc, vc, out_c, lse_c, scale=w.scale)

    for _ in range(args.warmup):
        ring()
    torch.cuda.synchronize(dev)
    r0, r1 = ev(), ev()
    r0.record(stream)
    nr = max(3, args.steps // 3)
    for _ in range(nr):
        ring()
    r1.record(stream)
    torch.cuda.synchronize(dev)
    da.check(dev)
    ring_ms = max_over_ranks(dist, r0.elapsed_time(r1) / nr)
    ring_diff = (out_f - out_c).abs().max().item()

    # ---- token-major (BSND) tensors: the re-shard transpose and attention on strided views ----
    q_s = da.bhnd_to_bsnd(q)                       # [B, N, H, D] memory
    k_s, v_s = da.bhnd_to_bsnd(k), da.bhnd_to_bsnd(v)
    out_s = torch.empty((B, N, H, D), device=dev, dtype=torch.float32)
    q_t = torch.empty_like(q)
    for _ in range(args.warmup):
        da.bsnd_to_bhnd(q_s, out=q_t)
        da.attn_fwd_strided(q_s.transpose(1, 2), k_s.transpose(1, 2), v_s.transpose(1, 2),
                            out=out_s.transpose(1, 2), lse=lse_c, scale=w.scale)
    torch.cuda.synchronize(dev)
    da.check(dev)
    bsnd_diff = (out_s.transpose(1, 2) - out_f).abs().max().item()
    t_0, t_1 = ev(), ev()
    nt = max(10, args.steps)
    t_0.record(stream)
    for _ in range(nt):
        da.bsnd_to_bhnd(q_s, out=q_t)
    t_1.record(stream)
    a_0, a_1 = ev(), ev()
    na = max(3, args.steps // 3)
    a_0.record(stream)
    for _ in range(na):
        da.attn_fwd_strided(q_s.transpose(1, 2), k_s.transpose(1, 2), v_s.transpose(1, 2),
                            out=out_s.transpose(1, 2), lse=lse_c, scale=w.scale)
    a_1.record(stream)
    torch.cuda.synchronize(dev)
    da.check(dev)
    transpose_ms = max_over_ranks(dist, t_0.elapsed_time(t_1) / nt)
    transpose_bytes = 2 * B * H * N * D * 2
    bsnd_ms = max_over_ranks(dist, a_0.elapsed_time(a_1) / na)
    del q_s, k_s, v_s, out_s, q_t

    # ---- stale-KV attention of one patch (displaced patch parallelism, p patches) ----
    m = w.chunks[0]
    kb, vb = k.clone(), v.clone()
    q_patch = q[:, :, :m].contiguous()
    k_new, v_new = k[:, :, :m].contiguous(), v[:, :, :m].contiguous()
    o_patch = torch.empty((B, H, m, D), device=dev, dtype=torch.float32)
    l_patch = torch.empty((B, H, m), device=dev, dtype=torch.float32)
    s_split, ws = da.splitkv_plan(B, H, m, N, D, dev)  # the library's split-KV suggestion

    def stale_ms_for(splits):
        for _ in range(args.warmup):
            da.stale_kv_attention(q_patch, k_new, v_new, kb, vb, 0, out=o_patch, lse=l_patch,
                                  scale=w.scale, splits=splits, workspace=ws)
        torch.cuda.synchronize(dev)
        st_0, st_1 = ev(), ev()
        ns = max(5, args.steps)
        st_0.record(stream)
        for _ in range(ns):
            da.stale_kv_attention(q_patch, k_new, v_new, kb, vb, 0, out=o_patch, lse=l_patch,
                                  scale=w.scale, splits=splits, workspace=ws)
        st_1.record(stream)
        torch.cuda.synchronize(dev)
        da.check(dev)
        return max_over_ranks(dist, st_0.elapsed_time(st_1) / ns)

    stale_ms = stale_ms_for(s_split)
    stale_ms_unsplit = stale_ms_for(1)
    stale_flops = 4.0 * B * H * m * N * D
    del kb, vb, q_patch, k_new, v_new, o_patch, l_patch, ws

    # ---- cross-attention shape: all N queries against 512 replicated text keys ----
    n_txt = 512
    kx, vx = k[:, :, :n_txt], v[:, :, :n_txt]
    for _ in range(args.warmup):
        da.attn_chunk_fwd(q, kx, vx, out=out_c, lse=lse_c, scale=w.scale)
    torch.cuda.synchronize(dev)
    x0, x1 = ev(), ev()
    x0.record(stream)
    nx = max(5, args.steps)
    for _ in range(nx):
        da.attn_chunk_fwd(q, kx, vx, out=out_c, lse=lse_c, scale=w.scale)
    x1.record(stream)
    torch.cuda.synchronize(dev)
    da.check(dev)
    cross_ms = max_over_ranks(dist, x0.elapsed_time(x1) / nx)
    cross_flops = 4.0 * B * H * N * n_txt * D
    # The same with bf16 output (what a DiT's cross-attention feeds its output projection).
    out_x16 = torch.empty((B, H, N, D), device=dev, dtype=torch.bfloat16)
    for _ in range(args.warmup):
        da.attn_chunk_fwd(q, kx, vx, out=out_x16, lse=lse_c, scale=w.scale, out_dtype=torch.bfloat16)
    torch.cuda.synchronize(dev)
    x0.record(stream)
    for _ in range(nx):
        da.attn_chunk_fwd(q, kx, vx, out=out_x16, lse=lse_c, scale=w.scale, out_dtype=torch.bfloat16)
    x1.record(stream)
    torch.cuda.synchronize(dev)
    da.check(dev)
    cross16_ms = max_over_ranks(dist, x0.elapsed_time(x1) / nx)
    del out_x16

    # ---- end to end through the public API with host buffers ----
    q_p, k_p, v_p = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    o1_h = torch.empty(out_f.shape, dtype=torch.float32, pin_memory=True)
    l1_h = torch.empty(lse_f.shape, dtype=torch.float32, pin_memory=True)
    o2_h = torch.empty(out_f.shape, dtype=torch.float32, pin_memory=True)
    l2_h = torch.empty(lse_f.shape, dtype=torch.float32, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in (q_p, k_p, v_p))
    d2h = sum(t.numel() * t.element_size() for t in (o1_h, l1_h, o2_h, l2_h))

    # Through the public host pipeline: head groups are uploaded, computed (fused pass and
    # chunk path) and downloaded with the copies overlapping the compute.
    flat_in = [t.reshape(B * H, N, D) for t in (q_p, k_p, v_p)]
    flat_out = [o1_h.view(B * H, N, D), l1_h.view(B * H, N), o2_h.view(B * H, N, D),
                l2_h.view(B * H, N)]
    groups = da.head_groups(B * H)

    # A group's chunk path runs on a second stream beside its fused pass, so that each launch
    # can fill the SMs the other's last wave leaves idle (small head groups are few waves).
    side = torch.cuda.Stream(dev)

    def both_paths(qg, kg, vg):
        q4, k4, v4 = qg.unsqueeze(0), kg.unsqueeze(0), vg.unsqueeze(0)
        cur = torch.cuda.current_stream(dev)
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            o2, l2 = da.chunk_attention(q4, k4, v4, w.chunks, scale=w.scale, batched=True)
        o1, l1 = da.attn_fwd(q4, k4, v4, scale=w.scale)
        cur.wait_stream(side)
        for t in (o2, l2, q4, k4, v4):
            t.record_stream(side)
        return o1[0], l1[0], o2[0], l2[0]

    def e2e_step():
        da.host_pipeline(both_paths, flat_in, flat_out, groups, dev)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_steps = max(5, args.steps // 2)
    barrier(dist)
    torch.cuda.synchronize(dev)
    a, b = ev(), ev()
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    da.check(dev)
    e2e_ms = max_over_ranks(dist, a.elapsed_time(b) / e2e_steps)
    e2e_value = step_flops * world / (e2e_ms * 1e-3) / 1e12
    # The host-pipelined results against the device-timed fused pass (same kernels per head,
    # so the fused output is bitwise the same; the chunk path differs by rounding).
    out_f_h = out_f.cpu()
    e2e_check = {"fused_bitwise_equal_to_device": bool(torch.equal(o1_h, out_f_h)),
                 "chunk_path_max_abs_vs_fused": float((o2_h - out_f_h).abs().max())}
    del out_f_h

    peaks, peak_src = load_peaks()
    peak_sust = float(peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"])
    peak_burst = float(peaks["bf16_tflops"])

    # ---- every configured workload's fused pass and chunk paths (driver-visible record) ----
    workloads = None
    if not args.no_workloads:
        del q_p, k_p, v_p, o1_h, l1_h, o2_h, l2_h
        workloads = {}
        for name in synth.WORKLOADS:
            rec = workload_record(name, dev, peak_burst, args.steps)
            for path in ("fused", "chunk_merge", "chunk_merge_bf16_partials", "ring_accumulate",
                         "stale_kv_patch"):
                rec[path]["ms"] = max_over_ranks(dist, rec[path]["ms"])
            workloads[name] = rec
    hbm = float(peaks["hbm_gbs"])
    fused_tflops = w.flops / (fused_ms * 1e-3) / 1e12
    chunk_tflops = w.flops / (chunk_ms * 1e-3) / 1e12
    merge_bytes = p * B * H * N * (D * 4 + 4) + B * H * N * (D * 4 + 4)
    merge_gbs = merge_bytes / (merge_ms * 1e-3) / 1e9
    traffic = profiled_traffic(w.name)

    # Roofline fraction of every attention path against the measured bf16 burst peak (each is
    # timed over well under a second at the maximum SM clock, the burst figure's conditions; the
    # sustained figure, measured over seconds under the power cap, is reported beside it) and of
    # the HBM-bound kernels (against the measured copy).
    def tf_frac(tflops):
        return {"tflops": tflops, "frac_of_burst_peak": tflops / peak_burst,
                "frac_of_sustained_peak": tflops / peak_sust}

    line = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            tf, secs, rows, threads = oracle_sample_tflops(w, q_h, k_h, v_h,
                                                           target_s=args.cpu_baseline_s)
            cpu = {"value": tf, "unit": UNIT, "cores": threads, "kind": "oracle",
                   "sample": f"{B * H} heads x {rows} query rows against all {N} keys "
                             f"({secs:.1f} s of fp64 oracle)"}
            # The same oracle on one core, over a smaller sample.
            tf1, secs1, rows1, _ = oracle_sample_tflops(
                w, q_h, k_h, v_h, target_s=min(4.0, args.cpu_baseline_s / 3), threads=1)
            cpu["single_core"] = {"value": tf1, "cores": 1,
                                  "sample": f"{B * H} heads x {rows1} query rows "
                                            f"({secs1:.1f} s)"}
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 Q/K/V shaped like Wan2.2 TI2V-5B attention)",
            "config": workload_config(w),
            "fraction_of_peak": fused_tflops / peak_burst,
            "step_distribution_ms": {
                "fused": pct(fused_all), "chunk_merge": pct(chunk_all)},
            "small_workload": None if not small else {
                "l2_flushed_ms_per_step": ms_step, "warm_ms_per_step": warm_ms,
                "cuda_graph_ms_per_step": graph_ms, "cuda_graph_error": graph_err},
            "paths": {
                "fused": {"ms": fused_ms, **tf_frac(fused_tflops)},
                "chunk_merge": {"ms": chunk_ms, **tf_frac(chunk_tflops),
                                "ratio_to_fused": chunk_ms / fused_ms,
                                "merge_ms": merge_ms, "merge_gbs": merge_gbs,
                                "merge_frac_of_hbm": merge_gbs / hbm},
                "chunk_merge_bf16_partials": {"ms": chunk16_ms,
                                              **tf_frac(w.flops / (chunk16_ms * 1e-3) / 1e12),
                                              "ratio_to_fused": chunk16_ms / fused_ms},
                "fused_without_lse": {"ms": no_lse_ms,
                                      **tf_frac(w.flops / (no_lse_ms * 1e-3) / 1e12),
                                      "o_bitwise_equal": no_lse_same},
                "chunk_merge_per_rank_launches": {
                    "ms": per_rank_ms, **tf_frac(w.flops / (per_rank_ms * 1e-3) / 1e12),
                    "ratio_to_fused": per_rank_ms / fused_ms, "launches": p + 1},
                "ring_accumulate": {"ms": ring_ms,
                                    **tf_frac(w.flops / (ring_ms * 1e-3) / 1e12),
                                    "ratio_to_fused": ring_ms / fused_ms,
                                    "max_abs_vs_fused": ring_diff},
                "fused_bsnd_layout": {"ms": bsnd_ms, **tf_frac(w.flops / (bsnd_ms * 1e-3) / 1e12),
                                      "max_abs_vs_bhnd": bsnd_diff},
                "bsnd_to_bhnd_transpose": {"ms": transpose_ms,
                                           "gbs": transpose_bytes / (transpose_ms * 1e-3) / 1e9,
                                           "frac_of_hbm": transpose_bytes / (transpose_ms * 1e-3)
                                           / 1e9 / hbm},
                "stale_kv_patch": {"ms": stale_ms, "queries": m, "keys": N, "kv_splits": s_split,
                                   **tf_frac(stale_flops / (stale_ms * 1e-3) / 1e12),
                                   "unsplit_ms": stale_ms_unsplit,
                                   "unsplit_tflops": stale_flops / (stale_ms_unsplit * 1e-3)
                                   / 1e12},
                "cross_attention_512_text_keys": {"ms": cross_ms, "out_dtype": "f32",
                                                  **tf_frac(cross_flops / (cross_ms * 1e-3) / 1e12)},
                "cross_attention_512_text_keys_bf16_out": {
                    "ms": cross16_ms, "out_dtype": "bf16",
                    **tf_frac(cross_flops / (cross16_ms * 1e-3) / 1e12)},
                "fused_vs_chunk_max_abs": diff,
            },
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel<128,fp32>",
                         "achieved": fused_tflops, "peak": peak_burst, "unit": "TFLOP/s",
                         "frac": fused_tflops / peak_burst,
                         "peak_kind": f"{peak_src} bf16 burst (the timed region is under a "
                                      f"second; its sampled clocks are below)",
                         "frac_of_sustained_peak": fused_tflops / peak_sust,
                         # The burst peak scaled by the median SM clock sampled inside the
                         # timed region: the power cap lowers the clock under sustained load.
                         "frac_at_sampled_clock": (
                             fused_tflops / (peak_burst * clocks["sm_mhz"] / clocks["sm_max_mhz"])
                             if clocks.get("sm_mhz") and clocks.get("sm_max_mhz") else None),
                         "traffic": traffic,
                         "algorithmic_bytes": 3 * B * H * N * D * 2 + B * H * N * (D * 4 + 4)},
            "e2e": {"value": e2e_value, "unit": UNIT, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, **e2e_check},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "workloads": workloads,
        }
    if dist is not None:
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


def time_launches(fn, dev, reps, warmup, flush=None):
    """Mean device time (ms) of fn over `reps` launches after `warmup`, CUDA events on the current
    stream; with `flush` (a buffer larger than L2) written before every timed launch, each launch
    is timed on its own."""
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(dev)
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps
    total = 0.0
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        total += a.elapsed_time(b)
    return total / reps


def workload_record(name, dev, peak_burst, steps):
    """The fused pass and the p-chunk paths of one workload (its own inputs, timed outside the
    step): TFLOP/s, fraction of the measured bf16 burst peak, and each chunk path's time against
    the fused pass.  Inputs below L2 are timed with L2 flushed before every launch."""
    from diffusion_transformer_long_gb300 import ditattn as da

    w = synth.WORKLOADS[name]
    q, k, v = (t.to(dev) for t in synth.make_qkv(w))
    B, H, N, D, p = w.B, w.H, w.N, w.D, w.p
    out = torch.empty((B, H, N, D), device=dev, dtype=torch.float32)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    parts = torch.empty((p, B, H, N, D), device=dev, dtype=torch.float32)
    parts16 = torch.empty((p, B, H, N, D), device=dev, dtype=torch.bfloat16)
    lses = torch.empty((p, B, H, N), device=dev, dtype=torch.float32)
    out_c, lse_c = torch.empty_like(out), torch.empty_like(lse)
    small = 3 * B * H * N * D * 2 <= L2_BYTES
    flush = torch.empty(int(256e6) // 4, device=dev, dtype=torch.float32) if small else None
    reps = max(3, steps // (4 if N > 50000 else 1))
    starts = synth.chunk_starts(w.chunks)

    def fused():
        da.attn_fwd(q, k, v, out=out, lse=lse, scale=w.scale)

    def chunks32():
        da.attn_chunks_fwd(q, k, v, w.chunks, partials=parts, lses=lses, scale=w.scale)
        da.attn_lse_merge(parts, lses, out=out_c, lse=lse_c)

    def chunks16():
        da.attn_chunks_fwd(q, k, v, w.chunks, partials=parts16, lses=lses, scale=w.scale)
        da.attn_lse_merge(parts16, lses, out=out_c, lse=lse_c)

    def ring():
        for c, (s0, n) in enumerate(zip(starts, w.chunks)):
            kc, vc = k[:, :, s0:s0 + n], v[:, :, s0:s0 + n]
            if c == 0:
                da.attn_chunk_fwd(q, kc, vc, out=out_c, lse=lse_c, scale=w.scale)
            else:
                da.attn_chunk_fwd_accumulate(q, kc, vc, out_c, lse_c, scale=w.scale)

    # One stale-KV patch (displaced patch parallelism): the first chunk's rows as the patch, with
    # the library's split-KV suggestion and unsplit.
    m = w.chunks[0]
    kb, vb = k.clone(), v.clone()
    q_patch = q[:, :, :m].contiguous()
    k_new, v_new = k[:, :, :m].contiguous(), v[:, :, :m].contiguous()
    o_patch = torch.empty((B, H, m, D), device=dev, dtype=torch.float32)
    l_patch = torch.empty((B, H, m), device=dev, dtype=torch.float32)
    s_split, ws = da.splitkv_plan(B, H, m, N, D, dev)

    def patch(splits):
        return lambda: da.stale_kv_attention(q_patch, k_new, v_new, kb, vb, 0, out=o_patch,
                                             lse=l_patch, scale=w.scale, splits=splits,
                                             workspace=ws if splits > 1 else None)

    t = {}
    for key, fn in (("fused", fused), ("chunk_merge", chunks32), ("chunk_merge_bf16_partials",
                                                                   chunks16), ("ring_accumulate", ring),
                    ("stale_kv_patch", patch(s_split)), ("stale_kv_patch_unsplit", patch(1))):
        t[key] = time_launches(fn, dev, reps, 3, flush)
    da.check(dev)
    tf = w.flops / (t["fused"] * 1e-3) / 1e12
    rec = {"shape": f"B={B} H={H} N={N} D={D}", "p": p, "chunks": list(w.chunks),
           "timing": "L2 flushed before every launch" if small else "back to back (inputs > L2)",
           "reps": reps,
           "fused": {"ms": t["fused"], "tflops": tf, "frac_of_burst_peak": tf / peak_burst}}
    for key in ("chunk_merge", "chunk_merge_bf16_partials", "ring_accumulate"):
        rec[key] = {"ms": t[key], "ratio_to_fused": t[key] / t["fused"]}
    rec["stale_kv_patch"] = {"queries": m, "keys": N, "kv_splits": s_split,
                             "ms": t["stale_kv_patch"], "unsplit_ms": t["stale_kv_patch_unsplit"]}
    del q, k, v, out, lse, parts, parts16, lses, out_c, lse_c, flush, kb, vb, q_patch, k_new, v_new
    del o_patch, l_patch, ws
    torch.cuda.empty_cache()
    return rec


def run_profile_case(args):
    """Runs ONE path of the step (--warmup + --steps launches, untimed, no JSON) on the
    workload's inputs and nothing else: the small, short command an ncu capture wraps."""
    from diffusion_transformer_long_gb300 import ditattn as da

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    q, k, v = (t.to(dev) for t in synth.make_qkv(w))
    B, H, N, D, p = w.B, w.H, w.N, w.D, w.p
    out = torch.empty((B, H, N, D), device=dev, dtype=torch.float32)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    s0, n0 = synth.chunk_starts(w.chunks)[1], w.chunks[1]
    if args.profile_case == "merge":
        parts = torch.randn((p, B, H, N, D), device=dev)
        lses = torch.randn((p, B, H, N), device=dev)
    if args.profile_case == "chunks":
        parts = torch.empty((p, B, H, N, D), device=dev)
        lses = torch.empty((p, B, H, N), device=dev)
    if args.profile_case == "transpose":
        src = da.bhnd_to_bsnd(q)
        dst = torch.empty_like(q)
    torch.cuda.synchronize(dev)
    for _ in range(args.warmup + args.steps):
        if args.profile_case == "fused":
            da.attn_fwd(q, k, v, out=out, lse=lse, scale=w.scale)
        elif args.profile_case == "chunks":
            da.attn_chunks_fwd(q, k, v, w.chunks, partials=parts, lses=lses, scale=w.scale)
        elif args.profile_case == "chunk":
            da.attn_chunk_fwd(q, k[:, :, s0:s0 + n0], v[:, :, s0:s0 + n0], out=out, lse=lse,
                              scale=w.scale)
        elif args.profile_case == "accumulate":
            da.attn_chunk_fwd_accumulate(q, k[:, :, s0:s0 + n0], v[:, :, s0:s0 + n0], out, lse,
                                         scale=w.scale)
        elif args.profile_case == "merge":
            da.attn_lse_merge(parts, lses, out=out, lse=lse)
        elif args.profile_case == "transpose":
            da.bsnd_to_bhnd(src, out=dst)
        elif args.profile_case == "cross":
            da.attn_chunk_fwd(q, k[:, :, :512], v[:, :, :512], out=out, lse=lse, scale=w.scale)
    torch.cuda.synchronize(dev)
    da.check(dev)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="wan22", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-baseline-s", type=float, default=15.0)
    ap.add_argument("--ref-step-s", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload record (every config's fused and chunk paths)")
    ap.add_argument("--profile-case", choices=["fused", "chunks", "chunk", "accumulate", "merge",
                                               "transpose", "cross"],
                    help="run only this path, untimed (for ncu captures); prints nothing")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    if args.profile_case:
        return run_profile_case(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
