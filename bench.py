#!/usr/bin/env python
"""Benchmark of the NF4 + LoRA linear layer on B300.

Headline: forward + backward (to dX, dA, dB) TFLOP/s of the 7B-attention-shaped projection
(W 4096 x 4096 as NF4 with double-quantized scales, X 4096 tokens x 4096 bf16, LoRA r=16,
alpha=32), inputs resident in HBM, L2 flushed between steps, per-step CUDA events.
Alongside: the dominant kernel's roofline (live CUDA-event timing through the library's
profiling hook), an end-to-end number through the public API with host buffers, the HBM-bound
kernels (dequantize, quantize, decode M = 1/4/16) in GB/s, SM clocks sampled during the
timed region, and the CPU oracle timed on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica (the layer needs no exchange
for a fixed batch); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
METRIC = "NF4+LoRA linear fwd+bwd TFLOP/s and dequant GB/s on 1 B300, % of roofline"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def traffic_records():
    """ncu DRAM bytes per launch committed under profiles/, keyed by kernel, valid only
    while the kernel's source file is unchanged (sha256 of the file)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    out = {}
    if not os.path.exists(path):
        return out
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        name, src, sha, nbytes, workload = line.split(None, 4)
        fp = os.path.join(ROOT, src)
        if os.path.exists(fp) and hashlib.sha256(open(fp, "rb").read()).hexdigest() == sha:
            out[(name, workload.strip())] = float(nbytes)
    return out


# ------------------------------------------------------------------ clocks sampler
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples (the JSON line carries their summary); QLORA_CLOCKS_DIR keeps them
        import tempfile
        out_dir = os.environ.get("QLORA_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ helpers
def make_l2_flush(dev):
    """Cold-L2 reset between timed calls: write 256 MiB (twice the 126 MB L2), then read
    another 256 MiB, so the L2 ends up holding clean lines of unrelated data.  Without the
    read the timed kernel's first misses would also pay for writing the flush's dirty lines
    back to HBM (~6 us per 117 MB streamed, measured on B300)."""
    import torch
    wbuf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(32 << 20, dtype=torch.int64, device=dev)
    sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush():
        wbuf.zero_()
        torch.sum(rbuf, (0,), out=sink)
    return flush


def bf16_dev(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over the ranks (the timed region's wall time: the slowest replica)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle sample
def oracle_sample(p, X, Wd, A, B, dY, target_s: float = 12.0):
    """The oracle (fp64 CPU loops) on a bounded sample of the workload: Y and dX for a
    subset of token rows plus U, V, dA, dB over all rows.  Returns (TFLOP/s, desc, cores)."""
    import oracle
    M, N, K, r = p.M, p.N, p.K, p.r

    def run(nrows):
        rows = np.linspace(0, M - 1, nrows).astype(np.int64)
        t0 = time.perf_counter()
        oracle.lora_fwd(X, Wd, A, B, p.scale, rows)
        oracle.lora_dx(dY, Wd, A, B, p.scale, rows)
        t1 = time.perf_counter()
        return t1 - t0

    run(2)  # thread-pool start-up outside the calibration
    t_rows = run(64) / 64
    t0 = time.perf_counter()
    oracle.lora_dadb(dY, X, A, B, p.scale)
    t_full = time.perf_counter() - t0

    def rows_for(per_row):
        return int(max(8, min(M, (target_s - t_full) / max(per_row, 1e-9))))

    nrows = rows_for(t_rows)
    t_rows_total = run(nrows)
    if t_rows_total + t_full < 0.6 * target_s and nrows < M:  # calibration ran slow: re-size once
        nrows = rows_for(t_rows_total / nrows)
        t_rows_total = run(nrows)
    flops = (2.0 * nrows * (N * K + r * K + r * N) * 2          # Y rows (with U), dX rows (with V)
             + 2.0 * (M * K * r + M * N * r + r * K * M + N * r * M))  # U, V, dA, dB over all M
    secs = t_rows_total + t_full
    desc = (f"oracle fp64 loops: Y and dX for {nrows} of {M} token rows, U/V/dA/dB over all "
            f"{M} rows ({flops / 1e9:.1f} GFLOP in {secs:.1f} s)")
    return flops / secs / 1e12, desc, oracle.num_threads(), secs


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from bit_nf4_quantized_37_b300 import workloads as wl
    import oracle
    p = wl.config2()
    W = p.W()
    q = oracle.quantize(W)
    Wd = oracle.dequantize(q).reshape(p.N, p.K)
    X, A, B, dY = p.X(), p.A(), p.B(), p.dY()
    vals = []
    descs = []
    cores = oracle.num_threads()
    per_step_s = max(3.0, 60.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup + args.steps):
        v, d, cores, secs = oracle_sample(p, X, Wd, A, B, dY, target_s=per_step_s)
        if i >= args.warmup:
            vals.append(v)
            descs.append(d)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(p),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": descs[-1]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(p):
    return {"workload": f"7B attention projection: W {p.N}x{p.K} NF4 (block 64, double-quant 256),"
                        f" X {p.M}x{p.K} bf16, LoRA r={p.r} alpha={p.alpha:g}, fwd + bwd (dX, dA, dB)",
            "M": p.M, "N": p.N, "K": p.K, "r": p.r, "alpha": p.alpha,
            "l2": "flushed between timed steps (256 MiB write, then 256 MiB read of another "
                  "buffer: cold L2 without dirty lines)",
            "parallelism": "replicas"}


# ------------------------------------------------------------------ our arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--eager", action="store_true", help="no CUDA graph for the timed step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    world, rank, local = dist_setup(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    import bit_nf4_quantized_37_b300 as qn
    from bit_nf4_quantized_37_b300 import build, workloads as wl
    build.build()
    qn.lib()
    peaks, peak_src = load_peaks()
    traffic = traffic_records()

    p = wl.config2()
    W = p.W()
    Xh, Ah, Bh, dYh = p.X(), p.A(), p.B(), p.dY()
    q = qn.nf4_quantize(torch.from_numpy(W).to(dev))
    X, A, B, dY = (bf16_dev(t, dev) for t in (Xh, Ah, Bh, dYh))
    l2_flush = make_l2_flush(dev)
    s = p.scale

    def step():
        Y, U = qn.qlora_linear_fwd(X, q, A, B, s)
        dX, dA, dB = qn.qlora_linear_bwd(dY, X, q, A, B, s, U)
        return Y, dX, dA, dB

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # The timed step is one CUDA-graph replay of forward + backward (the library's launches
    # captured once).  Per-kernel device times come from a second graph of the same step
    # captured with the library's per-kernel CUDA events, replayed for the same number of
    # steps right after the timed ones (event nodes between kernels would cut the
    # programmatic-launch overlap of the timed graph).  --eager times the calls as issued
    # from Python instead, with the events in the same calls.
    graph = graph_prof = None
    if not args.eager:
        qn.profile_start()  # fill the event pool before capture
        step()
        torch.cuda.synchronize()
        qn.profile_stop()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            step()
        graph_prof = torch.cuda.CUDAGraph()
        qn.profile_start()  # its records (the captured event nodes) stay live until the end
        with torch.cuda.graph(graph_prof, capture_error_mode="thread_local"):
            step()
        for _ in range(args.warmup):
            graph.replay()
            graph_prof.replay()
        torch.cuda.synchronize()

    clocks = Clocks(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    if graph is None:
        qn.profile_start()
    for i in range(args.steps):
        l2_flush()
        ev[i][0].record()
        if graph is None:
            step()
        else:
            graph.replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    if graph is not None:  # the per-kernel profile: same steps, same flushes
        for i in range(args.steps):
            l2_flush()
            graph_prof.replay()
        torch.cuda.synchronize()
    prof = qn.profile_stop()
    clk = clocks.stop() if clocks else None
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world)
    flops_step = p.fwd_bwd_flops()
    value = flops_step * args.steps * world / (total_ms / 1e3) / 1e12
    # launches recorded per captured step (graph) or over all steps (eager)
    launches = sum(v[0] for v in prof.values()) * (args.steps if graph is not None else 1)

    # dominant kernel and its roofline (algorithmic FLOPs per launch / mean launch time)
    dom = max(prof.items(), key=lambda kv: kv[1][1])
    dom_name, (dom_n, dom_ms) = dom
    per_launch_flops = {
        "fused_fwd_gemm": 2.0 * p.M * p.N * p.K + 2.0 * p.M * p.N * p.r,
        "fused_dx_gemm": 2.0 * p.M * p.N * p.K + 2.0 * p.M * p.K * p.r,
    }
    rl = None
    if dom_name in per_launch_flops:
        ach = per_launch_flops[dom_name] / (dom_ms / dom_n / 1e3) / 1e12
        tr = traffic.get((dom_name, "config2"))
        rl = {"bound": "tensor", "kernel": dom_name, "achieved": ach, "peak": peaks["bf16_tflops"],
              "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "traffic": tr,
              "peak_source": f"{peak_src} bf16 burst",
              "mean_launch_ms": dom_ms / dom_n}
    kernels = {k: {"launches": n, "ms_per_launch": ms / n, "share": ms / sum(v[1] for v in prof.values())}
               for k, (n, ms) in sorted(prof.items(), key=lambda kv: -kv[1][1])}
    other = {}
    for k in ("fused_fwd_gemm", "fused_dx_gemm"):
        if k in prof:
            n, ms = prof[k]
            a = per_launch_flops[k] / (ms / n / 1e3) / 1e12
            other[k] = {"achieved_tflops": a, "frac_of_bf16_burst": a / peaks["bf16_tflops"],
                        "frac_of_bf16_sustained": a / peaks["bf16_tflops_sustained"]}

    # end to end through the public API with host buffers (pinned), copies inside the region
    Xp = torch.from_numpy(Xh.view(np.int16)).view(torch.bfloat16).pin_memory()
    dYp = torch.from_numpy(dYh.view(np.int16)).view(torch.bfloat16).pin_memory()
    Yp = torch.empty(p.M, p.N, dtype=torch.bfloat16).pin_memory()
    dXp = torch.empty(p.M, p.K, dtype=torch.bfloat16).pin_memory()
    dAp = torch.empty(p.r, p.K, dtype=torch.float32).pin_memory()
    dBp = torch.empty(p.N, p.r, dtype=torch.float32).pin_memory()
    # Steps are pipelined the way a caller streaming batches would run them: step i + 1's
    # inputs go up on one copy stream and step i's results come down on another while step i
    # computes on the current stream (the two directions of the host link run at once). The
    # device inputs are double-buffered; events order every reuse of a buffer.
    Xd = [torch.empty_like(X) for _ in range(2)]
    dYd = [torch.empty_like(dY) for _ in range(2)]
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        b = i & 1
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(in_free[b])  # step i - 2 has finished with this buffer
            Xd[b].copy_(Xp, non_blocking=True)
            dYd[b].copy_(dYp, non_blocking=True)
            in_ready[b].record(up)

    def e2e_steps(n, start):
        up.wait_event(start)
        upload(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                upload(i + 1)
            comp.wait_event(in_ready[b])
            Y, U = qn.qlora_linear_fwd(Xd[b], q, A, B, s)
            dX, dA, dB = qn.qlora_linear_bwd(dYd[b], Xd[b], q, A, B, s, U)
            in_free[b].record(comp)
            done[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(done[b])
                for host, dev_t in ((Yp, Y), (dXp, dX), (dAp, dA), (dBp, dB)):
                    host.copy_(dev_t, non_blocking=True)
                    dev_t.record_stream(down)  # not reused before its copy has run
        comp.wait_stream(down)

    w0 = torch.cuda.Event()
    w0.record(comp)
    e2e_steps(3, w0)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    e2e_steps(args.steps, e0)
    e1.record(comp)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_val = flops_step * args.steps * world / (e2e_ms / 1e3) / 1e12
    h2d = Xp.numel() * 2 + dYp.numel() * 2
    d2h = Yp.numel() * 2 + dXp.numel() * 2 + dAp.numel() * 4 + dBp.numel() * 4

    secondary = {} if args.no_secondary else measure_secondary(qn, wl, dev, peaks, traffic,
                                                               l2_flush)
    if not args.no_secondary:
        with_cpu = rank == 0 and not args.no_cpu
        secondary.update(measure_merge_and_error(qn, wl, p, q, A, B, dev, peaks, l2_flush))
        secondary.update(measure_f16(qn, p, q, X, A, B, dY, peaks, l2_flush))
        secondary["config3_mlp_M2048"] = measure_config3(qn, wl, dev, peaks, l2_flush, with_cpu)
        secondary["config5_llama7b_stack"] = measure_config5(qn, wl, dev, peaks, l2_flush, with_cpu)
        if with_cpu:
            add_cpu_secondary(secondary, wl)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded normal weights / activations, random-init adapters)",
        "config": config_block(p),
        "roofline": rl,
        "gemm_rooflines": other,
        "kernels": kernels,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "timed_step": "eager calls" if graph is None else "CUDA graph replay of fwd + bwd",
        "clocks": clk,
        "secondary": secondary,
    }
    if rank == 0 and not args.no_cpu:
        import oracle
        Wd = oracle.dequantize(oracle.quantize(W)).reshape(p.N, p.K)
        v, desc, cores, _ = oracle_sample(p, Xh, Wd, Ah, Bh, dYh)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def graph_timed_ms(fn, l2_flush, reps: int = 10) -> float:
    """Device time of one call: reps x (L2 flush + call) as one CUDA graph minus the same
    graph of flushes alone."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()

    def capture(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            body()
        return g

    def replay_ms(g):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g.replay()
        torch.cuda.synchronize()
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    def calls():
        for _ in range(reps):
            l2_flush()
            fn()

    def flushes():
        for _ in range(reps):
            l2_flush()

    return (replay_ms(capture(calls)) - replay_ms(capture(flushes))) / reps


def measure_merge_and_error(qn, wl, p, q, A, B, dev, peaks, l2_flush):
    """Adapter merge W' + s B A (bf16 out) on the 4096^2 layer, the loss of requantizing the
    merged weights, and the NF4-vs-INT4 squared errors on normal and Student-t(3) weights."""
    import torch
    hbm = peaks["hbm_gbs"]
    out = {}
    Wm = torch.empty(p.N, p.K, dtype=torch.bfloat16, device=dev)
    ms = graph_timed_ms(lambda: qn.nf4_merge_lora(q, A, B, p.scale, out=Wm), l2_flush)
    nbytes = q.storage_bytes() + 2 * p.r * (p.N + p.K) + 2 * p.N * p.K
    _, m32 = qn.nf4_merge_lora(q, A, B, p.scale, bf16=False, f32=True)
    base = qn.nf4_dequantize(q).float()
    requant = qn.nf4_dequantize(qn.nf4_quantize(m32)).float()
    delta = torch.linalg.vector_norm(m32 - base).item()
    loss = torch.linalg.vector_norm(requant - m32).item()
    out["merge_4096x4096_r16"] = {"GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm,
                                  "ms": ms, "bytes": nbytes,
                                  "requant_error_over_adapter_update": loss / delta}
    for kind in ("normal", "student_t3"):
        if kind == "normal":
            W = torch.from_numpy(p.W()).to(dev)
        else:
            W = torch.from_numpy(wl.student_t_weight((p.N, p.K), seed=43, df=3.0,
                                                     sigma=0.02)).to(dev)
        st = qn.nf4_int4_error_stats(W).cpu().tolist()
        ms = graph_timed_ms(lambda: qn.nf4_int4_error_stats(W), l2_flush)
        out[f"nf4_vs_int4_{kind}_4096x4096"] = {
            "nf4_rel_mse": st[1] / st[0], "int4_rel_mse": st[2] / st[0],
            "nf4_over_int4": st[1] / st[2], "ms": ms,
            "GB/s": 4 * W.numel() / ms / 1e6}
    return out


def measure_f16(qn, p, q, X, A, B, dY, peaks, l2_flush):
    """The fp16 compute type on the same 4096^2 layer: forward + backward with X, A, B and dY
    converted to fp16, against the bf16 burst peak (the tensor cores' dense fp16 and bf16
    rates are equal)."""
    import torch
    Xh, Ah, Bh, dYh = (t.to(torch.float16) for t in (X, A, B, dY))

    def step():
        Y, U = qn.qlora_linear_fwd_f16(Xh, q, Ah, Bh, p.scale)
        qn.qlora_linear_bwd_f16(dYh, Xh, q, Ah, Bh, p.scale, U)

    ms = graph_timed_ms(step, l2_flush)
    tf = p.fwd_bwd_flops() / ms / 1e9
    return {"fwd_bwd_f16_4096x4096x4096_r16": {
        "TFLOP/s": tf, "frac_tensor": tf / peaks["bf16_tflops"], "ms": ms}}


def profiled(qn, fn, l2_flush, reps: int = 10):
    """Whole-call device time (graph_timed_ms) and the library's per-kernel mean device times
    from a second graph of the same calls with the profiling events."""
    import torch
    ms = graph_timed_ms(fn, l2_flush, reps)
    qn.profile_start()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        for _ in range(reps):
            l2_flush()
            fn()
    g.replay()
    torch.cuda.synchronize()
    prof = qn.profile_stop()
    return ms, {k: v[1] / reps for k, v in prof.items()}


def fused_fracs(p, kms, peaks):
    """TFLOP/s and fraction of the bf16 burst peak of the two fused GEMMs of one fwd + bwd."""
    out = {}
    flops = {"fused_fwd_gemm": 2.0 * p.M * p.N * p.K + 2.0 * p.M * p.N * p.r,
             "fused_dx_gemm": 2.0 * p.M * p.N * p.K + 2.0 * p.M * p.K * p.r}
    for k, f in flops.items():
        if k in kms and kms[k] > 0:
            a = f / kms[k] / 1e9
            out[k] = {"ms": kms[k], "TFLOP/s": a, "frac_bf16_burst": a / peaks["bf16_tflops"]}
    return out


def oracle_quantize_sample(W: np.ndarray, target_s: float = 3.0):
    """The oracle's quantize on leading rows of W (about target_s of CPU time): GB/s of
    algorithmic bytes (4 B read + 0.516 B written per weight) and the sample's text."""
    import oracle
    rows = max(1, min(W.shape[0], int(2e6 // W.shape[1])))
    t0 = time.perf_counter()
    oracle.quantize(W[:rows])
    dt = time.perf_counter() - t0
    rows = max(1, min(W.shape[0], int(rows * target_s / max(dt, 1e-6))))
    t0 = time.perf_counter()
    oracle.quantize(W[:rows])
    dt = time.perf_counter() - t0
    n = rows * W.shape[1]
    return {"GB/s": n * 4.51587 / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"quantize of {rows} x {W.shape[1]} weights in {dt:.1f} s (one thread: the "
                      "oracle's quantize has no parallel loop)"}


def measure_config3(qn, wl, dev, peaks, l2_flush, with_cpu: bool):
    """The 7B MLP projections (gate / up 11008 x 4096, down 4096 x 11008, 0.1% Student-t
    outliers), M = 2048 tokens, r = 16: fwd + bwd of each, TFLOP/s against the bf16 burst."""
    import torch
    out = {}
    tot_ms = tot_flops = 0.0
    cpu_s = cpu_flops = 0.0
    cpu_desc = []
    cores = None
    for p in wl.config3():
        W = p.W()
        q = qn.nf4_quantize(torch.from_numpy(W).to(dev))
        Xh, Ah, Bh, dYh = p.X(), p.A(), p.B(), p.dY()
        X, A, B, dY = (bf16_dev(t, dev) for t in (Xh, Ah, Bh, dYh))

        def step():
            Y, U = qn.qlora_linear_fwd(X, q, A, B, p.scale)
            qn.qlora_linear_bwd(dY, X, q, A, B, p.scale, U)

        ms, kms = profiled(qn, step, l2_flush)
        f = p.fwd_bwd_flops()
        tf = f / ms / 1e9
        out[p.name] = {"ms": ms, "TFLOP/s": tf, "frac_bf16_burst": tf / peaks["bf16_tflops"],
                       "gemms": fused_fracs(p, kms, peaks), "kernels_ms": kms}
        tot_ms += ms
        tot_flops += f
        if with_cpu:
            import oracle
            Wd = oracle.dequantize(oracle.quantize(W)).reshape(p.N, p.K)
            v, desc, cores, secs = oracle_sample(p, Xh, Wd, Ah, Bh, dYh, target_s=6.0)
            cpu_s += secs
            cpu_flops += v * 1e12 * secs
            cpu_desc.append(desc)
        del q, X, A, B, dY
    tf = tot_flops / tot_ms / 1e9
    out["total_3_projections"] = {"ms": tot_ms, "TFLOP/s": tf,
                                  "frac_bf16_burst": tf / peaks["bf16_tflops"],
                                  "target_ms_at_60pct": tot_flops / (0.6 * peaks["bf16_tflops"]) / 1e9}
    if with_cpu:
        out["cpu_oracle"] = {"value": cpu_flops / cpu_s / 1e12, "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": "; ".join(cpu_desc)}
    return out


def measure_config5(qn, wl, dev, peaks, l2_flush, with_cpu: bool):
    """The 32-layer Llama-7B-shaped stack, all-linear LoRA r = 16: nf4_quantize of all 224
    weight matrices (6.48 G weights, fp32 resident on the device), then forward + backward of
    every projection of every layer at M = 512 tokens (the seeded inputs of layer 0's
    projections, shared by the layers), each timed as one CUDA graph of the whole stack."""
    import torch
    from concurrent.futures import ThreadPoolExecutor
    hbm = peaks["hbm_gbs"]
    out = {}
    Ws, qs = [], []
    with ThreadPoolExecutor(8) as gen:
        for layer in range(32):
            projs = wl.config5(layer=layer)
            for p, W in zip(projs, gen.map(lambda pp: pp.W(), projs)):
                Ws.append(torch.from_numpy(W).to(dev))
                qs.append(qn.NF4Tensor.empty(p.N, p.K, dev))
    numel = sum(w.numel() for w in Ws)
    nbytes = sum(4 * w.numel() + q.storage_bytes() for w, q in zip(Ws, qs))
    ws = torch.empty(max(qn.nf4_quantize_workspace_bytes(w.numel()) for w in Ws),
                     dtype=torch.uint8, device=dev)

    def quantize_all():
        for w, q in zip(Ws, qs):
            qn.nf4_quantize(w, q, workspace=ws)

    ms = graph_timed_ms(quantize_all, l2_flush, reps=3)
    out["quantize_stack_224_matrices"] = {
        "GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm, "ms": ms,
        "bytes": nbytes, "weights": numel}
    if with_cpu:
        out["quantize_stack_224_matrices"]["cpu_oracle"] = oracle_quantize_sample(
            Ws[6].cpu().numpy(), target_s=3.0)
    del Ws, ws
    torch.cuda.empty_cache()

    projs0 = wl.config5(layer=0)
    ins = {}
    for p in projs0:
        ins[p.name.split("-")[-1]] = tuple(bf16_dev(t, dev) for t in (p.X(), p.A(), p.B(), p.dY()))
    scale = projs0[0].scale

    def layer_calls(layer):
        for i, p in enumerate(projs0):
            X, A, B, dY = ins[p.name.split("-")[-1]]
            q = qs[7 * layer + i]
            Y, U = qn.qlora_linear_fwd(X, q, A, B, scale)
            qn.qlora_linear_bwd(dY, X, q, A, B, scale, U)

    layer_flops = sum(p.fwd_bwd_flops() for p in projs0)
    per_proj = {}
    for i, p in enumerate(projs0):
        X, A, B, dY = ins[p.name.split("-")[-1]]
        q = qs[i]

        def step(q=q, X=X, A=A, B=B, dY=dY):
            Y, U = qn.qlora_linear_fwd(X, q, A, B, scale)
            qn.qlora_linear_bwd(dY, X, q, A, B, scale, U)

        pms, kms = profiled(qn, step, l2_flush)
        tf = p.fwd_bwd_flops() / pms / 1e9
        per_proj[p.name.split("-")[-1]] = {"ms": pms, "TFLOP/s": tf,
                                           "frac_bf16_burst": tf / peaks["bf16_tflops"],
                                           "gemms": fused_fracs(p, kms, peaks)}
    out["layer_projections_M512"] = per_proj
    sms = graph_timed_ms(lambda: [layer_calls(l) for l in range(32)], l2_flush, reps=2)
    tf = 32 * layer_flops / sms / 1e9
    out["stack_fwd_bwd_M512"] = {"ms": sms, "TFLOP/s": tf, "frac_bf16_burst": tf / peaks["bf16_tflops"],
                                 "flops": 32 * layer_flops,
                                 "note": "32 layers x 7 projections, forward then backward each, "
                                         "one L2 flush per stack pass"}
    if with_cpu:
        import oracle
        p = projs0[6]  # the down projection, the largest contraction
        Xh, Ah, Bh, dYh = p.X(), p.A(), p.B(), p.dY()
        Wd = oracle.dequantize(oracle.quantize(p.W())).reshape(p.N, p.K)
        v, desc, cores, _ = oracle_sample(p, Xh, Wd, Ah, Bh, dYh, target_s=5.0)
        out["stack_fwd_bwd_M512"]["cpu_oracle"] = {
            "value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": "layer 0 down projection: " + desc}
    del qs
    torch.cuda.empty_cache()
    return out


def measure_secondary(qn, wl, dev, peaks, traffic, l2_flush, reps: int = 10):
    """HBM-bound paths on the decode-shaped 28672 x 8192 weight: dequantize, quantize and the
    M = 1 / 4 / 16 decode forward, each in GB/s of algorithmic bytes against the HBM peak."""
    import torch
    out = {}
    p4 = wl.config4(1)
    W = torch.from_numpy(p4.W()).to(dev)
    numel = W.numel()
    q = qn.nf4_quantize(W)
    meta = q.storage_bytes()
    Wd = torch.empty(p4.N, p4.K, dtype=torch.bfloat16, device=dev)

    def capture(body):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            body()
        return graph

    def replay_ms(graph):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        graph.replay()  # warm
        torch.cuda.synchronize()
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    def timed(fn, names):
        # Whole-call device time: reps x (L2 flush + call) as one CUDA graph, minus the same
        # graph of flushes alone (no event nodes between the library's launches, so its
        # programmatic-launch overlaps stay).  Per-kernel times: a third graph of the same
        # sequence with the library's per-kernel events.
        for _ in range(3):
            fn()
        torch.cuda.synchronize()

        def calls():
            for _ in range(reps):
                l2_flush()
                fn()

        def flushes():
            for _ in range(reps):
                l2_flush()

        ms = (replay_ms(capture(calls)) - replay_ms(capture(flushes))) / reps
        qn.profile_start()
        g_prof = capture(calls)
        g_prof.replay()
        torch.cuda.synchronize()
        prof = qn.profile_stop()
        return ms, prof

    hbm = peaks["hbm_gbs"]
    ms, _ = timed(lambda: qn.nf4_dequantize(q, Wd), ["nf4_dequant"])
    nbytes = meta + 2 * numel
    out["dequantize_28672x8192"] = {"GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm,
                                    "ms": ms, "bytes": nbytes,
                                    "traffic": traffic.get(("nf4_dequant", "config4"))}
    Wh = torch.empty(p4.N, p4.K, dtype=torch.float16, device=dev)
    ms, _ = timed(lambda: qn.nf4_dequantize_f16(q, Wh), ["nf4_dequant"])
    out["dequantize_f16_28672x8192"] = {"GB/s": nbytes / ms / 1e6,
                                        "frac_hbm": nbytes / ms / 1e6 / hbm, "ms": ms,
                                        "bytes": nbytes}
    del Wh
    qq = qn.NF4Tensor.empty(p4.N, p4.K, dev)
    ms, prof = timed(lambda: qn.nf4_quantize(W, qq),
                     ["nf4_quant_blocks", "nf4_absmax_mean", "nf4_double_quant"])
    nbytes = 4 * numel + meta
    out["quantize_28672x8192"] = {"GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm,
                                  "ms": ms, "bytes": nbytes,
                                  "kernels_ms": {k: v[1] / reps for k, v in prof.items()}}
    del W
    for M in (1, 4, 16):
        p = wl.config4(M)
        X = bf16_dev(p.X(), dev)
        A = bf16_dev(p.A(), dev)
        B = bf16_dev(p.B(), dev)
        Y = torch.empty(M, p.N, dtype=torch.bfloat16, device=dev)
        fn = lambda: qn.qlora_linear_fwd(X, q, A, B, p.scale, save_u=False, out=Y)  # noqa: E731
        ms_all, prof = timed(fn, ["decode_u", "decode_gemv"])
        ms_gemv = prof["decode_gemv"][1] / reps
        nbytes = meta + 2 * M * p.K + 2 * M * p.N + 2 * p.r * (p.K + p.N)
        out[f"decode_fwd_M{M}"] = {
            "GB/s": nbytes / ms_all / 1e6, "frac_hbm": nbytes / ms_all / 1e6 / hbm,
            "ms": ms_all, "bytes": nbytes,
            "gemv_kernel_GB/s": meta / ms_gemv / 1e6,
            "gemv_kernel_frac_hbm": meta / ms_gemv / 1e6 / hbm,
            "gemv_traffic": traffic.get(("decode_gemv", "config4")) if M == 1 else None,
            "kernels_ms": {k: v[1] / reps for k, v in prof.items()}}
    # the fp16 compute type at M = 1
    p = wl.config4(1)
    X, A, B = (bf16_dev(t, dev).to(torch.float16) for t in (p.X(), p.A(), p.B()))
    Y = torch.empty(1, p.N, dtype=torch.float16, device=dev)
    fn = lambda: qn.qlora_linear_fwd_f16(X, q, A, B, p.scale, save_u=False, out=Y)  # noqa: E731
    ms_all, prof = timed(fn, ["decode_u", "decode_gemv"])
    nbytes = meta + 2 * p.K + 2 * p.N + 2 * p.r * (p.K + p.N)
    out["decode_fwd_f16_M1"] = {
        "GB/s": nbytes / ms_all / 1e6, "frac_hbm": nbytes / ms_all / 1e6 / hbm, "ms": ms_all,
        "bytes": nbytes, "kernels_ms": {k: v[1] / reps for k, v in prof.items()}}
    # per-token adapters: 16 tokens over 4 adapters (r = 64) on the same base
    p = wl.config4(16)
    nad = 4
    X = bf16_dev(p.X(), dev)
    A_all = torch.stack([bf16_dev(wl.bf16_normal((p.r, p.K), seed=4100 + i, sigma=0.01), dev)
                         for i in range(nad)])
    B_all = torch.stack([bf16_dev(wl.bf16_normal((p.N, p.r), seed=4200 + i, sigma=0.01), dev)
                         for i in range(nad)])
    idx = torch.arange(16, dtype=torch.int32, device=dev) % nad
    scales = torch.full((nad,), p.scale, dtype=torch.float32, device=dev)
    Y = torch.empty(16, p.N, dtype=torch.bfloat16, device=dev)
    fn = lambda: qn.qlora_linear_fwd_multi(X, q, A_all, B_all, idx, scales, out=Y)  # noqa: E731
    ms_all, prof = timed(fn, ["multi_u", "multi_z", "decode_gemv"])
    nbytes = meta + 2 * 16 * p.K + 2 * 16 * p.N + nad * 2 * p.r * (p.K + p.N)
    out["decode_fwd_M16_4adapters"] = {
        "GB/s": nbytes / ms_all / 1e6, "frac_hbm": nbytes / ms_all / 1e6 / hbm, "ms": ms_all,
        "bytes": nbytes, "kernels_ms": {k: v[1] / reps for k, v in prof.items()}}
    return out


def add_cpu_secondary(secondary, wl):
    """The oracle beside the HBM-bound lines on the 28672 x 8192 weight: quantize and
    dequantize on leading rows, the decode forward (M = 1 / 4 / 16) in full."""
    import oracle
    p4 = wl.config4(1)
    W = p4.W()
    qline = secondary.get("quantize_28672x8192")
    if qline is not None:
        qline["cpu_oracle"] = oracle_quantize_sample(W, target_s=3.0)
    rows = 2048
    o = oracle.quantize(W[:rows])
    t0 = time.perf_counter()
    Wd_part = oracle.dequantize(o)
    dt = time.perf_counter() - t0
    n = rows * p4.K
    for key in ("dequantize_28672x8192", "dequantize_f16_28672x8192"):
        if key in secondary:
            secondary[key]["cpu_oracle"] = {
                "GB/s": n * 2.51587 / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"dequantize of {rows} x {p4.K} weights in {dt:.2f} s (one thread)"}
    del Wd_part
    Wd = oracle.dequantize(oracle.quantize(W)).reshape(p4.N, p4.K)
    for M in (1, 4, 16):
        key = f"decode_fwd_M{M}"
        if key not in secondary:
            continue
        pm = wl.config4(M)
        X, A, B = pm.X(), pm.A(), pm.B()
        t0 = time.perf_counter()
        oracle.lora_fwd(X, Wd, A, B, pm.scale)
        dt = time.perf_counter() - t0
        nbytes = secondary[key]["bytes"]
        secondary[key]["cpu_oracle"] = {
            "GB/s": nbytes / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"the whole forward (Y for all {M} tokens) over the dequantized weight in "
                      f"{dt:.2f} s; the same algorithmic bytes as the device line"}


if __name__ == "__main__":
    main()
