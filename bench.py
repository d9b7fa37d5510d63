#!/usr/bin/env python3
"""Decode-step benchmark: one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one decode step of the whole layer stack (every kernel of the plan) over one batch of
synthetic input resident in HBM.  The default workload is the 28-layer bf16 talker (h2048,
16/8 heads, d128, SwiGLU 6144) with 2048 prefilled positions; its 128-step position range
2048..2175 is replayed cyclically (the stream is truncated back to 2048 after every 128 steps),
so every timed step is a genuine step of that workload.  Its per-step working set (3.3 GB of
weights and KV) is far larger than the 129 MB L2, so no L2 flush is needed between steps.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the path has no
exchange step); the timed region is bracketed by barriers, the time is the max over ranks and
the value is the aggregate steps/s of all ranks.

--impl reference times the CPU oracle (the plain sequential C restatement) on the host cores
with the same workload, metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tts_autoregressive_decode_gb300 import workloads as W  # noqa: E402

METRIC = "decode steps/sec and achieved HBM GB/s (% of GB300 peak) per token, 1 GPU"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes per launch of the dominant kernel from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), with the hash of the kernel source it was taken on.  A changed kernel
# reports null until it is captured again.
NCU_TRAFFIC = {
    # gate/up GEMV (k_gemv_rows<bf16, m1, NJ1>, N = 12288, K = 2048): one launch captured with
    # ncu (dram__bytes_read.sum, dram__bytes_write.sum) on the 2-layer case of the same shapes; a
    # launch does the same work at any layer count
    W.TALKER_H2048_L28.name: {"bytes_per_launch": 50_385_408, "source_sha": "6b44da6d6704a6bc"},
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1280)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=W.TALKER_H2048_L28.name,
                   choices=sorted(W.WORKLOADS))
    p.add_argument("--layers", type=int, default=0,
                   help="keep only the first N layers (small cases for profiler captures)")
    p.add_argument("--kernel-rounds", type=int, default=20)
    p.add_argument("--prefill-rows", type=int, default=64,
                   help="rows of the timed prefill block (talker workloads; 0: skip)")
    p.add_argument("--plan", choices=["kernels", "persistent"], default="kernels",
                   help="step plan: the chain of kernels (default) or the persistent kernel")
    p.add_argument("--tensor-gemv", action="store_true",
                   help="GEMVs of 3..8 rows (8-stream steps, prefill blocks) on the tensor cores")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--streams8", type=int, default=1,
                   help="also time the 8-stream 28-layer workload (1, default) or not (0)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured hbm_gbs (MEASURED_PEAKS.json, STREAM-style copy)"
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


# ------------------------------------------------------------------------------ bytes

def vector_bytes(w: W.Workload) -> int:
    h, d = w.hidden, w.head_dim
    per = (2 * h + 2 * d) if w.kind == "talker" else (6 if w.layer_scale else 4) * h
    tail = h if w.kind == "talker" else (3 * h if w.head else 0)  # final norm / out_norm + EOS
    return 4 * (w.layers * per + tail)


def kv_bytes(w: W.Workload, positions) -> int:
    """K and V bytes a step reads: talker pos+1 keys per stream and layer; codec: the ring."""
    if w.kind == "talker":
        return sum(2 * (p + 1) * w.kvw * 4 * w.layers for p in positions)
    return len(positions) * w.layers * (2 * w.ring * w.hidden * 4 + 4 * w.ring)


def step_bytes(w: W.Workload, positions) -> int:
    return w.matrix_bytes() + vector_bytes(w) + kv_bytes(w, positions)


def dominant_kernel(w: W.Workload, m: int):
    """(stage, name, algorithmic bytes per launch) of the plan's largest kernel."""
    es = 2 if w.weight_dtype == "bf16" else 4
    h, I = w.hidden, w.inter
    if w.kind == "talker":
        return (3, "norm + gate/up GEMV + SwiGLU (k_gemv_rows)",
                2 * I * h * es + 4 * (m * h + h + m * I))
    return (3, "LayerNorm + lin1 GEMV + GELU (k_gemv_rows)", I * h * es + 4 * (m * h + 2 * h + m * I))


# the sources the gate/up GEMV (k_gemv_rows) is compiled from
GEMV_SOURCES = ("gemv.cu", "gemv_rows.cuh", "common.cuh", "kernels.h")


def kernel_source_sha(files=GEMV_SOURCES) -> str:
    """Hash of the dominant kernel's source files: a stored ncu traffic figure is only reported
    for the sources it was measured on."""
    d = os.path.join(ROOT, "tts_autoregressive_decode_gb300", "csrc")
    h = hashlib.sha256()
    for f in files:
        h.update(f.encode())
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------ oracle timing

def oracle_rate(syn, seconds: float, threads: int, max_steps: int = 64, layers=None):
    """Steps/s of the CPU oracle on the workload's first steps (a bounded sample)."""
    import oracle

    w = syn.workload
    if layers is not None and layers < w.layers:
        import dataclasses
        sub = dataclasses.replace(syn, workload=dataclasses.replace(w, layers=layers),
                                  layers=syn.layers[:layers],
                                  prefill_k=[None if k is None else k[:layers] for k in syn.prefill_k],
                                  prefill_v=[None if v is None else v[:layers] for v in syn.prefill_v])
        syn = sub
    orc = oracle.OracleModel(syn, threads=threads)
    m = w.streams
    t0 = time.perf_counter()
    n = 0
    x = syn.x0 if w.feedback else None
    while n < max_steps and (n == 0 or time.perf_counter() - t0 < seconds):
        t = n % w.steps
        if n and t == 0:
            for s in range(m):
                orc.prefill_kv(s, syn.prefill_k[s], syn.prefill_v[s]) if syn.lengths[s] else orc.reset(s)
        xin = x if w.feedback else syn.inputs[t]
        y = orc.step(xin, [orc.length(s) for s in range(m)])
        if w.feedback:
            x = (y.astype(np.float32) + syn.e).astype(np.float32)
        n += 1
    dt = time.perf_counter() - t0
    orc.close()
    return n, dt


# ------------------------------------------------------------------------------ arms

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(pg, value: float, device) -> float:
    """The largest of the ranks' values, e.g. the slowest rank's timed span (the value itself
    with one rank).  `device` holds the reduction's tensor: "cuda" for NCCL, "cpu" for gloo."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, seconds: float) -> float:
    """Whole-job steps per second: each of `world` replicas ran `steps` steps in at most
    `seconds` (the max over ranks)."""
    return world * steps / seconds


def bench_config(w: W.Workload, lengths, world: int) -> dict:
    """The workload as both arms state it (the same dict, so the two lines compare)."""
    talker = w.kind == "talker"
    nb = step_bytes(w, lengths if talker else [0] * w.streams)
    return {"workload": w.name, "layers": w.layers, "hidden": w.hidden,
            "heads": f"{w.q_heads}/{w.kv_heads}", "head_dim": w.head_dim, "inter": w.inter,
            "weights": w.weight_dtype, "kv": "f32", "streams": w.streams,
            "positions": (f"{list(lengths)}..+{w.steps - 1}, replayed cyclically" if talker
                          else f"from {list(lengths)}, continuing"),
            "l2": ("no flush: per-step working set %.2f GB >> 129 MB L2" % (nb / 1e9)
                   if nb > 4 * 129e6 else
                   "per-step working set %.1f MB may be partly L2-resident" % (nb / 1e6)),
            "parallelism": f"replicas x{world}"}


def cpu_baselines(syn, seconds: float, one_core_seconds: float):
    """The oracle timed twice on the host: the sequential oracle on one core, and the
    row-parallel build of the same oracle on every core (bitwise the same results)."""
    w = syn.workload
    threads = os.cpu_count() or 1
    n, dt = oracle_rate(syn, seconds, threads)
    all_cores = {"value": n / dt, "unit": "steps/s", "cores": threads,
                 "sample": f"the first {n} steps of {w.name} (positions from the workload start), "
                           f"{dt:.1f} s on {threads} threads"}
    n1, dt1 = oracle_rate(syn, one_core_seconds, 1)
    one_core = {"value": n1 / dt1, "unit": "steps/s", "cores": 1,
                "sample": f"the first {n1} steps of {w.name}, {dt1:.1f} s on 1 thread"}
    return {"value": all_cores["value"], "unit": "steps/s", "cores": threads, "kind": "oracle",
            "sample": all_cores["sample"], "all_cores": all_cores, "one_core": one_core}


def run_reference(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    w = W.WORKLOADS[args.workload]
    syn = W.generate(w)
    threads = os.cpu_count() or 1
    # one full step first, to size the per-step sample so the whole run stays within minutes
    n1, dt1 = oracle_rate(syn, 0.0, threads, max_steps=1)
    budget = 150.0
    layers = w.layers
    if (args.steps + args.warmup) * dt1 > budget:
        layers = max(1, int(w.layers * budget / ((args.steps + args.warmup) * dt1)))
    _, _ = oracle_rate(syn, 1e9, threads, max_steps=args.warmup, layers=layers) if args.warmup else (0, 0)
    n, dt = oracle_rate(syn, 1e9, threads, max_steps=args.steps, layers=layers)
    per_step = dt / n * (w.layers / layers)       # full-stack equivalent seconds per step
    value = 1.0 / per_step
    # the sequential oracle on one core: one step of the same sample size
    n1, dt1 = oracle_rate(syn, 0.0, 1, max_steps=1, layers=layers)
    one_core = {"value": n1 / (dt1 * (w.layers / layers)), "unit": "steps/s", "cores": 1,
                "sample": f"{n1} step" + (f" on the first {layers} layers, scaled" if layers < w.layers
                                          else "") + ", 1 thread"}
    sample = (f"{n} steps of the {w.layers}-layer workload"
              + (f", each timed on its first {layers} layers and scaled by {w.layers}/{layers}"
                 if layers < w.layers else "")
              + f", positions from the workload start, {threads} threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": bench_config(w, syn.lengths, 1),
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": threads, "kind": "oracle",
                         "sample": sample, "one_core": one_core},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def time_streams8(args, stream, peak):
    """The 8-stream workload (28-layer bf16 talker, lengths U[512, 4096], 64 steps): K steps of
    its position range, replayed cyclically like the main workload, between CUDA events."""
    import torch

    from tts_autoregressive_decode_gb300.decoder import Decoder

    from tts_autoregressive_decode_gb300 import _lib

    w = W.TALKER_H2048_L28_M8
    syn = W.generate(w)
    dec = Decoder.from_synthetic(syn, flags=_lib.DEC_FLAG_TENSOR_GEMV if args.tensor_gemv else 0)
    m, base = w.streams, list(syn.lengths)
    X = torch.from_numpy(syn.inputs).cuda()
    out = torch.empty((m, w.hidden), dtype=torch.float32, device="cuda")
    del syn

    def one(i):
        t = i % w.steps
        if t == 0 and dec.length(0) != base[0]:
            for s_ in range(m):
                dec.truncate(s_, base[s_])
        dec.step(X[t], dec.lengths(m), out)

    for i in range(max(3, args.warmup)):
        one(i)
    dec.sync()
    for s_ in range(m):
        dec.truncate(s_, base[s_])
    dec.sync()
    steps = max(1, min(args.steps, 4 * w.steps))
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        one(i)
    e1.record(stream)
    torch.cuda.synchronize()
    dec.sync()
    ms = e0.elapsed_time(e1) / steps
    per = [step_bytes(w, [b + (i % w.steps) for b in base]) for i in range(w.steps)]
    nb = sum(per[i % w.steps] for i in range(steps)) / steps
    gbs = nb / (ms * 1e-3) / 1e9
    kpl = dec.kernels_per_step(m)
    dec.close()
    return {"workload": w.name, "streams": m, "lengths": base, "steps": steps,
            "ms_per_step": ms, "steps_per_s": 1e3 / ms, "tokens_per_s": m * 1e3 / ms,
            "bytes_per_step": nb, "achieved_hbm_gbs": gbs, "frac_of_peak": gbs / peak,
            "kernels_per_step": kpl,
            "note": "weights read once per step for all 8 rows, plus each stream's K/V"}


def run_ours(args):
    import torch

    from tts_autoregressive_decode_gb300 import native_build
    from tts_autoregressive_decode_gb300.decoder import Decoder

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    if rank == 0 or world == 1:
        native_build.build()
    if pg:
        pg.barrier()
    w = W.WORKLOADS[args.workload]
    if args.layers:
        import dataclasses
        w = dataclasses.replace(w, layers=min(args.layers, w.layers))
    talker = w.kind == "talker"
    syn = W.generate(w)
    if not talker:
        # the ring keeps positions growing: size the RoPE table for warm-up + timed + e2e steps
        syn.max_pos = max(syn.max_pos,
                          max(syn.lengths) + 2 * (args.warmup + args.steps) + 2 * w.steps + 8)
    from tts_autoregressive_decode_gb300 import _lib
    flags = (_lib.DEC_FLAG_PERSISTENT if args.plan == "persistent" else 0) | \
        (_lib.DEC_FLAG_TENSOR_GEMV if args.tensor_gemv else 0)
    dec = Decoder.from_synthetic(syn, flags=flags)
    m, h = w.streams, w.hidden
    base = list(syn.lengths)
    X = torch.from_numpy(syn.inputs).cuda()                  # [steps][m][h], resident in HBM
    out = torch.empty((m, h), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    set_len_kernels = [0]

    def positions(i):
        return [b + (i % w.steps) for b in base] if talker else [dec.length(s) for s in range(m)]

    def one_step(i, x=None):
        t = i % w.steps
        if talker and t == 0 and dec.length(0) != base[0]:
            for s in range(m):
                dec.truncate(s, base[s])
            set_len_kernels[0] += m
        dec.step(X[t] if x is None else x, dec.lengths(m), out)

    # ---- warm-up, then rewind to the workload's first position -----------------------------
    for i in range(args.warmup):
        one_step(i)
    dec.sync()
    if talker:
        for s in range(m):
            dec.truncate(s, base[s])
    dec.sync()
    pos_before = dec.lengths(m)

    # ---- timed region: K steps, CUDA events on the launching stream -------------------------
    step_positions = [positions(i) if talker else None for i in range(min(args.steps, w.steps))]
    clocks = ClockSampler(local)
    clocks.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    set_len_kernels[0] = 0
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        one_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clk = clocks.stop()
    dec.sync()
    ms = max_over_ranks(pg, e0.elapsed_time(e1), "cuda")
    launches = args.steps * dec.kernels_per_step(m) + set_len_kernels[0]

    # bytes: mean over the steps actually timed (the talker's range cycles)
    if talker:
        per_cycle = [step_bytes(w, p) for p in step_positions]
        nb = sum(per_cycle[i % len(per_cycle)] for i in range(args.steps)) / args.steps
    else:
        nb = step_bytes(w, [0] * m)
    ms_step = ms / args.steps
    value = job_throughput(world, args.steps, ms / 1e3)
    peak, peak_src = peaks()
    step_gbs = nb / (ms_step * 1e-3) / 1e9

    # ---- the dominant kernel ----------------------------------------------------------------
    kpl = dec.kernels_per_step(m)
    k_alone_ms = None
    if kpl == 1:
        # the persistent step kernel is the whole step: its launches are the timed region's
        kname = ("persistent streamed step kernel (k_stream_step: every layer's GEMVs, "
                 "attention, merge and the output rows)")
        kbytes = nb
        k_ms = ms_step
    else:
        # one launch per layer captured in a CUDA graph (no host launch cost in the timing),
        # replayed between CUDA events on the replay stream: chained as programmatic dependents
        # (the step's launch configuration) and, for reference, each launch alone
        if talker:
            for s in range(m):
                dec.truncate(s, base[s])
        dec.sync()
        stage, kname, kbytes = dominant_kernel(w, m)

        def time_graph(chained):
            cap = torch.cuda.Stream()
            graph = torch.cuda.CUDAGraph()
            dec.set_stream(cap)
            with torch.cuda.graph(graph, stream=cap):
                for l in range(w.layers):
                    dec.launch_stage(l, stage, m, chained=chained and l > 0)
            dec.set_stream(None)
            graph.replay()
            torch.cuda.synchronize()
            durs = []
            for _ in range(args.kernel_rounds):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                graph.replay()
                b.record(stream)
                torch.cuda.synchronize()
                durs.append(a.elapsed_time(b) / w.layers)
            del graph
            return statistics.median(durs)

        k_ms = time_graph(True)
        k_alone_ms = time_graph(False)
    k_gbs = kbytes / (k_ms * 1e-3) / 1e9
    sha = kernel_source_sha()
    tr = NCU_TRAFFIC.get(w.name)
    traffic = tr["bytes_per_launch"] if tr and tr.get("source_sha") == sha else None

    # ---- batched causal prefill (talker): a 64-row block at the workload's first position -------
    prefill = None
    if talker and args.prefill_rows > 0 and base[0] + args.prefill_rows <= syn.max_pos:
        n = args.prefill_rows
        xp = torch.randn((n, h), generator=torch.Generator().manual_seed(7)).cuda()
        yp = torch.empty_like(xp)
        times = []
        for rep in range(4):
            dec.truncate(0, base[0])
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dec.prefill(0, xp, yp)
            b.record(stream)
            torch.cuda.synchronize()
            if rep:
                times.append(a.elapsed_time(b))
        dec.truncate(0, base[0])
        pms = statistics.median(times)
        rows = dec.prefill_rows()
        blocks = (n + rows - 1) // rows
        pbytes = blocks * (w.matrix_bytes() + vector_bytes(w)) + kv_bytes(w, [base[0] + i for i in range(n)])
        prefill = {"rows": n, "block_rows": rows, "ms": pms, "tokens_per_s": n / (pms * 1e-3),
                   "achieved_hbm_gbs": pbytes / (pms * 1e-3) / 1e9,
                   "bytes": pbytes, "position": base[0],
                   "note": "weights read once per block of block_rows rows"}

    # ---- the flow head on the backbone's hidden state (FlowLM-shaped workloads) ------------------
    flow = None
    if w.head and W.FLOW_D512.cond == w.hidden:
        from tts_autoregressive_decode_gb300.decoder import FlowHead
        fs = W.FLOW_D512
        fw = W.generate_flow(fs, calls=1)
        head = FlowHead(fs, fw)
        noise = torch.from_numpy(fw["noise"][0]).cuda()
        lat = torch.empty_like(noise)
        for _ in range(10):
            head.step(out[0], noise, lat)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(200):
            head.step(out[0], noise, lat)
        b.record(stream)
        torch.cuda.synchronize()
        fus = a.elapsed_time(b) / 200 * 1e3
        D_, L_, C_, B_ = fs.dim, fs.latent, fs.cond, fs.blocks
        fbytes = 4 * (D_ * L_ + D_ * C_ + (3 * B_ + 2) * D_ * D_ + 2 * B_ * D_ * D_ + L_ * D_)
        flow = {"shape": fs.name, "us_per_call": fus, "kernels": head.kernels_per_step(),
                "weight_bytes": fbytes, "achieved_hbm_gbs": fbytes / (fus * 1e-6) / 1e9,
                "note": "one LSD step conditioned in place on the step's output row"}
        head.close()

    # ---- 8 concurrent streams of the 28-layer talker (its own decoder, timed the same way) ------
    streams8 = None
    if args.streams8 and w.name == W.TALKER_H2048_L28.name and not args.layers:
        streams8 = time_streams8(args, stream, peak)

    # ---- end to end through the C ABI with host buffers ----------------------------------------
    e2e = None
    if not args.no_e2e:
        if talker:
            for s in range(m):
                dec.truncate(s, base[s])
        xh = torch.from_numpy(syn.inputs.copy()).pin_memory()
        oh = torch.empty((m, h), dtype=torch.float32).pin_memory()
        import ctypes as C
        dec.sync()
        t0 = time.perf_counter()
        for i in range(args.steps):
            t = i % w.steps
            if talker and t == 0 and dec.length(0) != base[0]:
                for s in range(m):
                    dec.truncate(s, base[s])
            p = (C.c_int32 * m)(*dec.lengths(m))
            dec.step_host_ptr(m, xh[t].data_ptr(), p, oh.data_ptr())
        dt = max_over_ranks(pg, time.perf_counter() - t0, "cuda")
        e2e = {"value": job_throughput(world, args.steps, dt), "unit": "steps/s",
               "h2d_bytes_per_step": m * h * 4, "d2h_bytes_per_step": m * h * 4 + 4}

    # ---- the oracle on the host cores (rank 0, one GPU only) -----------------------------------
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baselines(syn, args.cpu_seconds, args.cpu_seconds)

    if rank != 0:
        return
    cfg = bench_config(w, base, world)
    plan = ("one CUDA graph per step holding one cooperative persistent kernel" if kpl == 1
            else f"one CUDA graph per step, {kpl} PDL-chained kernels")
    if args.tensor_gemv:
        plan += "; GEMVs of 3..8 rows (prefill blocks, 8-stream steps) on the tensor cores"
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": cfg, "plan": plan,
        "tokens_per_s": value * m,
        "achieved_hbm_gbs": step_gbs, "hbm_frac_of_peak": step_gbs / peak,
        "bytes_per_step": nb,
        "roofline": {"bound": "hbm", "achieved": k_gbs, "peak": peak, "unit": "GB/s",
                     "frac": k_gbs / peak, "traffic": traffic, "kernel": kname,
                     "bytes_per_launch": kbytes, "us_per_launch": k_ms * 1e3,
                     "launches": (f"{w.layers} launches of the kernel (one per layer's weights) "
                                  "chained as programmatic dependents, as in the step"
                                  if k_alone_ms is not None else "the step's single launch"),
                     "alone_us_per_launch": k_alone_ms * 1e3 if k_alone_ms is not None else None,
                     "peak_source": peak_src + (" (burst: the kernel's graph of one launch per layer, timed on its own)"
                                                if k_alone_ms is not None else " (burst)")},
        "step_roofline": {"bound": "hbm", "achieved": step_gbs, "peak": peak, "unit": "GB/s",
                          "frac": step_gbs / peak, "bytes_per_step": nb},
        "gpu_launches": launches,
        "e2e": e2e, "cpu_baseline": cpu, "clocks": clk, "prefill": prefill, "flow_head": flow,
        "streams8": streams8,
    }
    print(json.dumps(line))
    if pg:
        pg.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
