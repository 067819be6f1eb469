#!/usr/bin/env python
"""Benchmark of the BitDelta hot path on GB300.

Headline workload ("stack70b"): the seven linears (q, k, v, o, gate, up,
down) of 20 decoder layers of a 70B-shaped model (hidden 8192, FFN 28672,
8 key/value heads of 128) with a resident bf16 base (34.2 GB) and 14
fine-tuned variants stored as BitDelta signs + scales (Laplace(0, 1e-3)
deltas, 2.14 GB of bits each, all resident).  One step is one decode batch of
128 tokens whose variant ids follow a Zipf(1.1) mix: the tokens are grouped
by variant once, then every linear runs the fused multi-variant kernel
y = x (W_base + alpha_v sign(delta_v))^T on its own synthetic activations.
``value`` is tokens per second over all ranks (weak scaling: every rank is an
independent replica; the path has no data exchange).

The same run also times, on rank 0, the other steps of the path on their own
workloads ("rows"): compression of 14 variants of a 28672 x 8192 matrix, the
prefill linear (gate and up, 4 variants x 4096 tokens), the single
4096 x 4096 linear at 1..64 tokens, the 14-variant FFN up-projection
(14336 x 4096, 64 tokens), per-row scales, the materialised reconstruction
and the delta cache.

``--impl reference`` times the CPU oracle on a bounded sample of the same
workload instead (host cores only).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "BitDelta fused linear: % HBM roofline (decode), % TC peak (prefill), tok/s"
UNIT = "tok/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300's nominal HBM3e bandwidth (~8 TB/s): a second, fixed denominator beside
# the measured copy peak
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--path", default="auto", help="kernel path: auto|simt|decode_tc|decode_fold|prefill_tc")
    p.add_argument("--layers", type=int, default=20)
    p.add_argument("--tokens", type=int, default=128)
    p.add_argument("--variants", type=int, default=14)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-rows", action="store_true", help="skip the compress/prefill/single rows")
    p.add_argument("--only", choices=["compress", "prefill", "single", "ffn14", "alpha_rows", "reconstruct", "delta_cache"],
                   default=None,
                   help="run just one row (for profiling); prints only that row")
    p.add_argument("--compress-variants", type=int, default=14)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample-rows", type=int, default=8192,
                   help="rows per linear of one layer in the oracle's sample")
    return p.parse_args()


# -- helpers -------------------------------------------------------------------

def peaks():
    f = ROOT / "MEASURED_PEAKS.json"
    if f.exists():
        d = json.loads(f.read_text())
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "compress_28672x8192": ["bd_compress.cu", "bd_internal.cuh"],
    # the decode step's kernels (grouping, staging, the shared-accumulator linear), its
    # dispatch and the helpers they are built from
    "linear_stack70b": ["bd_linear.cu", "bd_paths.cuh", "bd_internal.cuh", "bd_decode_fold.cu",
                        "bd_tmap.cu", "bd_tc_common.cuh", "bd_sm100.cuh"],
}


def sources_digest(names) -> str:
    """sha256 (16 hex) over the named kernel sources that exist."""
    h = hashlib.sha256()
    for n in names:
        p = ROOT / "bit_delta_compressed_gb300" / "csrc" / n
        if p.exists():
            h.update(n.encode())
            h.update(p.read_bytes())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key: str):
    """DRAM bytes per launch from an ncu capture of the kernel's current
    sources: a line 'traffic <key> <bytes> sources <digest>' in profiles/*.md.
    None when absent or when the sources changed since the capture."""
    digest = sources_digest(KERNEL_SOURCES.get(kernel_key, []))
    stale = []
    for f in sorted((ROOT / "profiles").glob("*.md")):
        for line in f.read_text().splitlines():
            m = re.match(r"\s*traffic\s+(\S+)\s+([0-9.eE+]+)\s+sources\s+(\w+)", line)
            if m and m.group(1) == kernel_key:
                if m.group(3) == digest:
                    return float(m.group(2))
                stale.append("%s (%s)" % (f.name, m.group(3)))
    sys.stderr.write("bench: no ncu traffic figure for %s matches the current sources (digest %s; %s); "
                     "reporting traffic null\n" % (kernel_key, digest,
                                                   "stale: " + ", ".join(stale) if stale else "none recorded"))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# -- the workload ----------------------------------------------------------------

def max_over_ranks(value: float, world: int, device) -> float:
    """The slowest rank's value (every rank passes its own)."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Tokens per second over all ranks: every rank is an independent replica
    processing its own batch in the same step time (weak scaling)."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


def distinct_count(ids) -> int:
    return len(set(int(v) for v in ids))


def build_stack(args, torch, bd, wl, dev, seed):
    """Resident base weights, 14 variants' bits and scales, per-linear x."""
    g = wl.generator(seed, dev)
    V, M = args.variants, args.tokens
    ids_cpu = wl.variant_ids_zipf(M, V, 1.1, wl.generator(seed + 1))
    ids = ids_cpu.to(dev)
    linears = []
    for layer in range(args.layers):
        for name, N, K in wl.LAYER_LINEARS:
            wb = wl.base_weights(N, K, g, dev)
            alphas = torch.empty(V, dtype=torch.float32, device=dev)
            bits = []
            ws = bd.compress_workspace(N, K, dev)
            for v in range(V):
                wf = wl.finetuned_weights(wb, 1e-3, g)
                b = torch.empty((N, K // 32), dtype=torch.int32, device=dev)
                bd.compress(wf, wb, workspace=ws, alpha_out=alphas[v:v + 1], bits_out=b)
                bits.append(b)
                del wf
            x = wl.activations(M, K, g, dev)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            linears.append({"name": "%d.%s" % (layer, name), "N": N, "K": K, "wb": wb,
                            "alphas": alphas, "bits": bits, "ptrs": bd.bits_pointer_array(bits),
                            "x": x, "y": y})
    torch.cuda.synchronize()
    return ids, ids_cpu, linears


def linear_bytes(M, N, K, D, y_bytes=2):
    """Algorithmic HBM bytes of one fused linear launch: the bf16 base once,
    one bit per weight per distinct variant, activations in, outputs out."""
    return 2 * N * K + D * N * K // 8 + 2 * M * K + y_bytes * M * N


# -- CPU oracle sample -------------------------------------------------------------

def oracle_sample_time(args, wl, rows_per_linear, seed, nthreads=None):
    """Time the oracle on one layer's seven linears, ``rows_per_linear`` output
    rows each, all tokens, on ``nthreads`` host threads (default: all);
    returns (seconds, weights covered, threads)."""
    import numpy as np
    import torch
    import oracle
    o = oracle.get()
    g = wl.generator(seed + 7)
    V, M = args.variants, args.tokens
    ids = wl.variant_ids_zipf(M, V, 1.1, wl.generator(seed + 1)).numpy()
    cases = []
    for name, N, K in wl.LAYER_LINEARS:
        r = min(rows_per_linear, N)
        wb = wl.base_weights(r, K, g).view(torch.int16).numpy().view(np.uint16)
        bits = [torch.randint(-2 ** 31, 2 ** 31, (r, K // 32), generator=g, dtype=torch.int64)
                .to(torch.int32).numpy().view(np.uint32) for _ in range(V)]
        alphas = np.full(V, 1e-3, dtype=np.float32)
        x = wl.activations(M, K, g).view(torch.int16).numpy().view(np.uint16)
        cases.append((x, wb, alphas, bits, r * K))
    t0 = time.perf_counter()
    for x, wb, alphas, bits, _ in cases:
        o.linear(x, ids, wb, alphas, bits, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, sum(c[4] for c in cases), oracle.host_threads() if nthreads is None else int(nthreads)


def cpu_value(args, wl, seconds, weights_done):
    total = args.layers * sum(n * k for _, n, k in wl.LAYER_LINEARS)
    step_s = seconds * total / weights_done
    return args.tokens / step_s


# -- arms --------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    import workloads as wl
    for _ in range(args.warmup):
        oracle_sample_time(args, wl, max(8, args.cpu_sample_rows // 64), args.seed)
    times = []
    weights = threads = 0
    for _ in range(args.steps):
        dt, weights, threads = oracle_sample_time(args, wl, max(8, args.cpu_sample_rows // 64), args.seed)
        times.append(dt)
    sec = sum(times) / len(times)
    value = cpu_value(args, wl, sec, weights)
    step_ms = args.tokens / value * 1e3
    sample = ("oracle fp64 linear on layer 0's seven linears, %d output rows each, all %d tokens, "
              "14 variants; step time extrapolated by weight count to %d layers"
              % (max(8, args.cpu_sample_rows // 64), args.tokens, args.layers))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": stack_config(args, reference_distinct(args, wl)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def reference_distinct(args, wl):
    """Distinct variants of rank 0's batch (the same ids the GPU arm draws)."""
    return distinct_count(wl.variant_ids_zipf(args.tokens, args.variants, 1.1,
                                              wl.generator(args.seed + 1)).tolist())


def stack_config(args, D):
    return {"workload": "stack70b", "layers": args.layers, "linears_per_layer": 7,
            "hidden": 8192, "ffn": 28672, "kv_dim": 1024, "tokens": args.tokens,
            "variants": args.variants, "variant_mix": "zipf(1.1)", "distinct_variants": D,
            "laplace_b": 1e-3, "y_dtype": "bf16", "path": args.path,
            "l2": "inputs larger than L2 (64 GB of weights and bits resident)"}


def run_ours(args, rank, world, local_rank):
    import torch
    import bit_delta_compressed_gb300 as bd
    import workloads as wl

    bd.get_lib()          # fails loudly if the library is missing
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    pk, pk_src = peaks()
    seed = args.seed + 1000 * rank

    ids, ids_cpu, linears = build_stack(args, torch, bd, wl, dev, seed)
    V, M = args.variants, args.tokens
    D = distinct_count(ids_cpu.tolist())
    ws_bytes = max(int(bd.get_lib().bitdelta_linear_workspace(M, L["N"], L["K"], V)) for L in linears)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    n_lin = len(linears)

    def new_event():
        return torch.cuda.Event(enable_timing=True)
    # one event pair around every fused-linear launch of every timed step
    ev = [[(new_event(), new_event()) for _ in range(n_lin)] for _ in range(args.steps)]

    def step(events=None):
        bd.group(ids, V, ws)
        for i, L in enumerate(linears):
            if events is not None:
                events[i][0].record(stream)
            bd.linear_grouped(L["x"], L["wb"], L["alphas"], L["ptrs"], V, L["y"], ws, path=args.path)
            if events is not None:
                events[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = bd.device_status(ws)
    if st != 0:
        raise RuntimeError("device status after warm-up: " + bd.status_string(st))

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    sampler = ClockSampler(gpu_uuid(torch, dev)) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t0, t1 = new_event(), new_event()
    launches0 = int(bd.get_lib().bitdelta_launch_count())
    torch.cuda.profiler.start()       # bounds an ncu launch list to the timed region
    t0.record(stream)
    for s_i in range(args.steps):
        step(ev[s_i])
    t1.record(stream)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    launches = int(bd.get_lib().bitdelta_launch_count()) - launches0
    barrier()
    clocks = sampler.stop() if sampler else None
    ms_per_step = max_over_ranks(t0.elapsed_time(t1) / args.steps, world, dev)
    value = whole_job_rate(M, world, ms_per_step)

    # roofline of the dominant kernel: algorithmic bytes per launch over the
    # average launch duration inside the timed region
    launch_ms = sum(a.elapsed_time(b) for row in ev for a, b in row) / (args.steps * n_lin)
    alg = sum(linear_bytes(M, L["N"], L["K"], D) for L in linears) / n_lin
    achieved = alg / (launch_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": profiled_traffic("linear_stack70b"),
            "nominal_peak": NOMINAL_HBM_GBS, "frac_nominal": achieved / NOMINAL_HBM_GBS,
            "kernel": "fused multi-variant linear (%s path)" % args.path,
            "alg_bytes_per_launch": alg, "avg_launch_us": launch_ms * 1e3,
            "peak_source": ("measured: MEASURED_PEAKS.json hbm_gbs (copy)" if pk_src == "measured"
                            else "fallback 6.8 TB/s")}

    e2e = measure_e2e(args, torch, bd, linears, ids, ws, V, stream)
    chained = measure_chained(args, torch, bd, linears, ids, ws, V, stream)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; random-init 70B-shaped weights, Laplace deltas)",
            "config": stack_config(args, D), "roofline": roof, "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks, "chained": chained}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, w_done, threads = oracle_sample_time(args, wl, args.cpu_sample_rows, args.seed)
        line["cpu_baseline"] = {
            "value": cpu_value(args, wl, dt, w_done), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "fp64 oracle linear on one layer's seven linears, %d output rows each, all %d "
                      "tokens, 14 variants (%.1f s); extrapolated by weight count to %d layers"
                      % (args.cpu_sample_rows, M, dt, args.layers)}
        st_rows = max(8, args.cpu_sample_rows // 16)
        dt1, w1, _ = oracle_sample_time(args, wl, st_rows, args.seed, nthreads=1)
        line["cpu_baseline"]["single_thread"] = {
            "value": cpu_value(args, wl, dt1, w1), "unit": UNIT, "cores": 1,
            "sample": "the same, %d output rows per linear (%.1f s)" % (st_rows, dt1)}
    del linears
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_rows:
        line["rows"] = run_rows(args, torch, bd, wl, dev, pk)
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_e2e(args, torch, bd, linears, ids, ws, V, stream):
    """Same metric through the public API with host buffers: per step the
    activations and ids go host->device from pinned memory and every y comes
    back device->host, inside the timed region.  The copies run on streams of
    their own, as a serving loop would issue them: linear i's input copy
    overlaps the compute of the linears before it and its output copy the
    compute of those after it.  Events order every buffer's reuse: a step's
    copy into x_i waits for the previous step's linear i, its linear i waits
    for the previous step's copy out of y_i, and the ids wait for the previous
    grouping."""
    hx = [L["x"].cpu().pin_memory() for L in linears]
    hy = [torch.empty(L["y"].shape, dtype=L["y"].dtype, pin_memory=True) for L in linears]
    hids = ids.cpu().pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hx) + hids.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in hy)
    n = len(linears)
    dev = ids.device
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    ev_in, ev_done, ev_out = [ev() for _ in range(n)], [ev() for _ in range(n)], [ev() for _ in range(n)]
    ev_ids, ev_group = ev(), ev()
    state = {"first": True}

    def e2e_step():
        first = state["first"]
        with torch.cuda.stream(s_in):
            if not first:
                s_in.wait_event(ev_group)
            ids.copy_(hids, non_blocking=True)
            ev_ids.record(s_in)
            for i, (L, h) in enumerate(zip(linears, hx)):
                if not first:
                    s_in.wait_event(ev_done[i])
                L["x"].copy_(h, non_blocking=True)
                ev_in[i].record(s_in)
        stream.wait_event(ev_ids)
        bd.group(ids, V, ws)
        ev_group.record(stream)
        for i, L in enumerate(linears):
            stream.wait_event(ev_in[i])
            if not first:
                stream.wait_event(ev_out[i])
            bd.linear_grouped(L["x"], L["wb"], L["alphas"], L["ptrs"], V, L["y"], ws, path=args.path)
            ev_done[i].record(stream)
        with torch.cuda.stream(s_out):
            for i, (L, h) in enumerate(zip(linears, hy)):
                s_out.wait_event(ev_done[i])
                h.copy_(L["y"], non_blocking=True)
                ev_out[i].record(s_out)
        state["first"] = False

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    n_steps = max(3, args.steps // 5)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    s_in.wait_event(a)
    s_out.wait_event(a)
    for _ in range(n_steps):
        e2e_step()
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n_steps
    return {"value": args.tokens / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "copies": "pinned host buffers; input and output copies on their own streams, "
                      "overlapping the compute of other linears"}


def measure_chained(args, torch, bd, linears, ids, ws, V, stream):
    """The same stack as real decoder layers: each layer's projections fed by
    the previous ones (q/k/v from the hidden state, o from q in place of the
    attention output, gate/up from the residual sum, down from silu(gate) * up,
    residual adds), the glue in torch; the batch grouped once per step."""
    from bit_delta_compressed_gb300 import layer
    per = len(layer.NAMES)
    layers = []
    for i in range(0, len(linears), per):
        chunk = linears[i:i + per]
        lin = {n: L for n, L in zip(layer.NAMES, chunk)}
        bufs = {n: L["y"] for n, L in zip(layer.NAMES, chunk)}
        layers.append((lin, bufs))
    h0 = linears[0]["x"]

    def chained_step():
        bd.group(ids, V, ws)
        h = h0
        for lin, bufs in layers:
            h = layer.chained_layer(bd, lin, h, V, ws, bufs, path=args.path)
        return h
    for _ in range(2):
        chained_step()
    torch.cuda.synchronize()
    n = max(3, args.steps // 5)
    ms = time_events(torch, chained_step, n, stream)
    return {"value": args.tokens / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "dataflow": "q,k,v <- h; o <- q (attention output stand-in); h1 = h + o; "
                        "gate, up <- h1; down <- silu(gate) * up; h2 = h1 + down (glue in torch)"}


def time_graph(torch, fn, iters, stream):
    """Time per replay of ``fn`` captured in a CUDA graph: the same launches
    without the per-call host work.  Returns (ms, None), or (None, reason)
    when capture fails."""
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
    except Exception as e:          # reported in the row; the eager figures stand
        torch.cuda.synchronize()
        return None, "%s: %s" % (type(e).__name__, str(e).splitlines()[0] if str(e) else "")
    graph.replay()
    torch.cuda.synchronize()
    ms = time_events(torch, graph.replay, iters, stream)
    del graph
    return ms, None


def time_events(torch, fn, iters, stream):
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(iters):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def run_rows(args, torch, bd, wl, dev, pk,
             which=("compress", "prefill", "single", "ffn14", "alpha_rows", "reconstruct", "delta_cache")):
    """Compress, prefill, the single-linear decode, the per-row-scale linear
    and the materialised reconstruction on their own workloads."""
    rows = {}
    g = wl.generator(args.seed + 50, dev)
    if "compress" in which:
        rows["compress"] = row_compress(args, torch, bd, wl, dev, pk, g)
        torch.cuda.empty_cache()
    if "prefill" in which:
        rows["prefill"] = row_prefill(args, torch, bd, wl, dev, pk, g)
        torch.cuda.empty_cache()
    if "single" in which:
        rows["single4096"] = row_single(args, torch, bd, wl, dev, pk, g)
        torch.cuda.empty_cache()
    if "ffn14" in which:
        rows["ffn14"] = row_ffn14(args, torch, bd, wl, dev, pk, g)
        torch.cuda.empty_cache()
    if "alpha_rows" in which:
        rows["alpha_rows"] = row_alpha_rows(args, torch, bd, wl, dev, pk, g)
        torch.cuda.empty_cache()
    if "reconstruct" in which:
        rows["reconstruct"] = row_reconstruct(args, torch, bd, wl, dev, pk, g)
        torch.cuda.empty_cache()
    if "delta_cache" in which:
        rows["delta_cache"] = row_delta_cache(args, torch, dev)
    return rows


def row_compress(args, torch, bd, wl, dev, pk, g):
    """14 variants of one 28672 x 8192 bf16 matrix (inputs 6.6 GB)."""
    stream = torch.cuda.current_stream()
    N, K, V = 28672, 8192, args.compress_variants
    wb = wl.base_weights(N, K, g, dev)
    wfs = [wl.finetuned_weights(wb, 1e-3, g) for _ in range(V)]
    alphas = torch.empty(V, dtype=torch.float32, device=dev)
    bits = [torch.empty((N, K // 32), dtype=torch.int32, device=dev) for _ in range(V)]
    cws = bd.compress_workspace(N, K, dev)

    def compress_all():
        for v in range(V):
            bd.compress(wfs[v], wb, workspace=cws, alpha_out=alphas[v:v + 1], bits_out=bits[v])
    for _ in range(3):
        compress_all()
    ms = time_events(torch, compress_all, 5, stream)
    per = 2 * 2 * N * K + N * K // 8
    ach = V * per / (ms / 1e3) / 1e9
    return {"workload": "%d variants of 28672x8192 bf16" % V, "ms": ms, "launches": V,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / pk["hbm_gbs"], "alg_bytes_per_launch": per,
                         "traffic": profiled_traffic("compress_28672x8192")}}


def row_prefill(args, torch, bd, wl, dev, pk, g):
    """gate and up (28672 x 8192), 4 variants x 4096 tokens grouped."""
    stream = torch.cuda.current_stream()
    N, K = 28672, 8192
    Vp, per = 4, 4096
    ids = wl.variant_ids_blocks([per] * Vp).to(dev)
    Mp = ids.numel()
    mats = []
    for _ in range(2):
        w = wl.base_weights(N, K, g, dev)
        b = [torch.randint(-2 ** 31, 2 ** 31, (N, K // 32), generator=g, device=dev,
                           dtype=torch.int64).to(torch.int32) for _ in range(Vp)]
        mats.append((w, b, bd.bits_pointer_array(b)))
    al = torch.full((Vp,), 1e-3, device=dev)
    x = wl.activations(Mp, K, g, dev)
    y = torch.empty((Mp, N), dtype=torch.bfloat16, device=dev)
    wsp = bd.linear_workspace(Mp, N, K, Vp, dev)
    bd.group(ids, Vp, wsp)
    path = pick_path(bd, "prefill_tc" if args.path == "auto" else args.path,
                     lambda p: bd.linear_grouped(x, mats[0][0], al, mats[0][2], Vp, y, wsp, path=p))

    def prefill():
        bd.group(ids, Vp, wsp)
        for w, b, p in mats:
            bd.linear_grouped(x, w, al, p, Vp, y, wsp, path=path)
    prefill()
    torch.cuda.synchronize()
    ms = time_events(torch, prefill, 3, stream)
    flops = 2 * 2 * Mp * N * K
    tf = flops / (ms / 1e3) / 1e12
    # the page's reading of prefill: rebuild each variant's W_eff (this
    # library's reconstruct kernel), then a library GEMM (torch.matmul, cuBLAS)
    w_eff = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    y2 = torch.empty((Mp, N), dtype=torch.bfloat16, device=dev)
    bits_of = [b for _, b, _ in mats]

    def materialise_then_gemm():
        for (w, b, _) in mats:
            for v in range(Vp):
                bd.reconstruct(w, al[v:v + 1], b[v], out=w_eff)
                torch.matmul(x[v * per:(v + 1) * per], w_eff.t(), out=y2[v * per:(v + 1) * per])
    materialise_then_gemm()
    torch.cuda.synchronize()
    ms_mat = time_events(torch, materialise_then_gemm, 3, stream)
    del w_eff, y2, bits_of
    return {"workload": "gate+up 28672x8192, 4 variants x 4096 tokens", "ms": ms, "path": path,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": tf / pk["bf16_tflops"], "traffic": None},
            "materialise_then_gemm_ms": ms_mat}


def row_single(args, torch, bd, wl, dev, pk, g):
    """Single 4096 x 4096 linear, 1 variant, M in {1, 8, 32, 64}; 16 weight
    copies rotate so that every call reads from HBM (> 2x L2).  Timed twice:
    eager calls (host work per call included: at these sizes the host can
    take longer than the device) and the same calls replayed from a CUDA
    graph (device time; the roofline fraction of the launches)."""
    stream = torch.cuda.current_stream()
    N = K = 4096
    copies = 16
    ws_list = []
    for _ in range(copies):
        w = wl.base_weights(N, K, g, dev)
        b = torch.randint(-2 ** 31, 2 ** 31, (N, K // 32), generator=g, device=dev,
                          dtype=torch.int64).to(torch.int32)
        ws_list.append((w, b, bd.bits_pointer_array([b])))
    al1 = torch.full((1,), 5e-4, device=dev)
    single = {}
    for M in (1, 8, 32, 64):
        x = wl.activations(M, K, g, dev)
        ids1 = torch.zeros(M, dtype=torch.int32, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        wsm = bd.linear_workspace(M, N, K, 1, dev)
        bd.group(ids1, 1, wsm)

        def run_all():
            for w, b, p in ws_list:
                bd.linear_grouped(x, w, al1, p, 1, y, wsm, path=args.path)
        run_all()
        ms = time_events(torch, run_all, 10, stream) / copies
        byt = linear_bytes(M, N, K, 1)
        single["M=%d" % M] = launch_figures(torch, run_all, ms, copies, byt, pk, stream)
    return single


def launch_figures(torch, fn, eager_ms, calls, byt, pk, stream):
    """Eager and graph-replayed time per call of ``fn`` (``calls`` linears),
    with the achieved bandwidth of each."""
    out = {"eager_us": eager_ms * 1e3, "eager_gbs": byt / (eager_ms / 1e3) / 1e9}
    out["eager_frac"] = out["eager_gbs"] / pk["hbm_gbs"]
    gms, err = time_graph(torch, fn, 10, stream)
    if gms is None:
        out["graph"] = "capture failed: " + err
        return out
    gms /= calls
    out["graph_us"] = gms * 1e3
    out["graph_gbs"] = byt / (gms / 1e3) / 1e9
    out["graph_frac"] = out["graph_gbs"] / pk["hbm_gbs"]
    return out


def row_ffn14(args, torch, bd, wl, dev, pk, g):
    """Multi-tenant FFN up-projection 14336 x 4096, 14 variants (Laplace
    scales uniform in [2e-4, 2e-3]), 64 tokens with uniform ids, through the
    automatic path; 3 weight sets rotate (> 4x L2)."""
    stream = torch.cuda.current_stream()
    N, K, V, M = 14336, 4096, 14, 64
    sets = 3
    alphas = torch.tensor(wl.scales_uniform(V, 2e-4, 2e-3, wl.generator(args.seed + 21)),
                          dtype=torch.float32, device=dev)
    ids = wl.variant_ids_uniform(M, V, wl.generator(args.seed + 22)).to(dev)
    D = int(torch.unique(ids[ids >= 0]).numel())
    mats = []
    for _ in range(sets):
        w = wl.base_weights(N, K, g, dev)
        b = [torch.randint(-2 ** 31, 2 ** 31, (N, K // 32), generator=g, device=dev,
                           dtype=torch.int64).to(torch.int32) for _ in range(V)]
        mats.append((w, b, bd.bits_pointer_array(b)))
    x = wl.activations(M, K, g, dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = bd.linear_workspace(M, N, K, V, dev)
    bd.group(ids, V, ws)

    def run_all():
        for w, b, p in mats:
            bd.linear_grouped(x, w, alphas, p, V, y, ws, path=args.path)
    run_all()
    ms = time_events(torch, run_all, 10, stream) / sets
    out = {"shape": [N, K], "variants": V, "tokens": M, "distinct": D,
           "algorithmic_bytes": linear_bytes(M, N, K, D)}
    out.update(launch_figures(torch, run_all, ms, sets, out["algorithmic_bytes"], pk, stream))
    return out


def row_alpha_rows(args, torch, bd, wl, dev, pk, g):
    """One scale per (variant, output row): the gate shape (28672 x 8192), 14
    variants, 128 tokens with Zipf(1.1) ids, through ``bitdelta_linear_rows``
    (grouping included in every call, as for a single linear), beside the
    per-matrix call with the same ids and path.  4 weight sets rotate (> 2x L2)."""
    stream = torch.cuda.current_stream()
    N, K, V, M = 28672, 8192, 14, 128
    sets = 4
    ids = wl.variant_ids_zipf(M, V, 1.1, wl.generator(args.seed + 7)).to(dev)
    D = int(torch.unique(ids[ids >= 0]).numel())
    mats = []
    for _ in range(sets):
        w = wl.base_weights(N, K, g, dev)
        b = [torch.randint(-2 ** 31, 2 ** 31, (N, K // 32), generator=g, device=dev,
                           dtype=torch.int64).to(torch.int32) for _ in range(V)]
        ar = (5e-4 + 1.5e-3 * torch.rand((V, N), generator=g, device=dev)).contiguous()
        mats.append((w, b, bd.bits_pointer_array(b), ar, ar[:, 0].contiguous()))
    x = wl.activations(M, K, g, dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = bd.linear_workspace(M, N, K, V, dev)
    path = "auto" if args.path == "auto" else args.path

    def run_rows_all():
        for w, b, p, ar, _ in mats:
            bd.linear_rows(x, ids, w, ar, b, out=y, out_dtype=torch.bfloat16, workspace=ws, path=path,
                           bits_ptrs=p)

    def run_matrix_all():
        for w, b, p, _, a1 in mats:
            bd.linear(x, ids, w, a1, b, out=y, out_dtype=torch.bfloat16, workspace=ws, path=path,
                      bits_ptrs=p)
    run_rows_all()
    run_matrix_all()
    torch.cuda.synchronize()
    ms_r = time_events(torch, run_rows_all, 5, stream) / sets
    ms_m = time_events(torch, run_matrix_all, 5, stream) / sets
    byt = linear_bytes(M, N, K, D) + D * N * 4
    ach = byt / (ms_r / 1e3) / 1e9
    return {"workload": "gate 28672x8192, 14 variants (Zipf 1.1), 128 tokens, per-row scales",
            "us": ms_r * 1e3, "per_matrix_us": ms_m * 1e3, "path": path, "distinct_variants": D,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / pk["hbm_gbs"], "alg_bytes_per_launch": byt, "traffic": None}}


def row_reconstruct(args, torch, bd, wl, dev, pk, g):
    """Materialised W_eff: 14 variants of one 28672 x 8192 matrix rebuilt in
    bf16 (HBM roofline, 4.125 bytes per weight); then the gate decode workload
    (14 Zipf variants, 128 tokens) as "reconstruct, then a library GEMM"
    (torch.matmul per present variant and one for base-model tokens) beside
    the fused linear on the same inputs."""
    stream = torch.cuda.current_stream()
    N, K, V, M = 28672, 8192, 14, 128
    wb = wl.base_weights(N, K, g, dev)
    bits = [torch.randint(-2 ** 31, 2 ** 31, (N, K // 32), generator=g, device=dev,
                          dtype=torch.int64).to(torch.int32) for _ in range(V)]
    alphas = 1e-3 * (1 + torch.rand(V, generator=g, device=dev))
    w_eff = torch.empty((N, K), dtype=torch.bfloat16, device=dev)

    def rec_all():
        for v in range(V):
            bd.reconstruct(wb, alphas[v:v + 1], bits[v], out=w_eff)
    rec_all()
    ms_rec = time_events(torch, rec_all, 5, stream)
    per = 2 * N * K + N * K // 8 + 2 * N * K
    ach = V * per / (ms_rec / 1e3) / 1e9
    ids = wl.variant_ids_zipf(M, V, 1.1, wl.generator(args.seed + 7)).to(dev)
    x = wl.activations(M, K, g, dev)
    groups = [(v, torch.nonzero(ids == v).flatten()) for v in range(V)]
    groups = [(v, idx) for v, idx in groups if idx.numel() > 0]
    base_idx = torch.nonzero(ids < 0).flatten()
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    def materialise_then_gemm():
        for v, idx in groups:
            bd.reconstruct(wb, alphas[v:v + 1], bits[v], out=w_eff)
            y[idx] = torch.matmul(x[idx], w_eff.t())
        if base_idx.numel():
            y[base_idx] = torch.matmul(x[base_idx], wb.t())
    ws = bd.linear_workspace(M, N, K, V, dev)
    ptrs = bd.bits_pointer_array(bits)
    y2 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    def fused():
        bd.linear(x, ids, wb, alphas, bits, out=y2, out_dtype=torch.bfloat16, workspace=ws, bits_ptrs=ptrs)
    materialise_then_gemm()
    fused()
    torch.cuda.synchronize()
    ms_mat = time_events(torch, materialise_then_gemm, 3, stream)
    ms_fused = time_events(torch, fused, 5, stream)
    return {"workload": "14 variants of 28672x8192; gate decode 128 tokens, 14 Zipf variants",
            "ms": ms_rec, "launches": V,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / pk["hbm_gbs"], "alg_bytes_per_launch": per, "traffic": None},
            "decode_gate_materialise_then_gemm_ms": ms_mat, "decode_gate_fused_ms": ms_fused,
            "fused_speedup": ms_mat / ms_fused, "distinct_variants": len(groups)}


def row_delta_cache(args, torch, dev):
    """Delta-cache loads: three variants of 1 GiB of packed bits each (pinned
    host memory) through a 2 GiB device cache without a hot set (every
    variant evictable), so every other acquire loads one variant and evicts
    another; bytes moved host -> device per second on the cache's copy
    stream."""
    from bit_delta_compressed_gb300.cache import DeltaCache
    nbits = 1 << 30
    cache = DeltaCache(2 * nbits + (1 << 20), dev, pinned_top_k=0)
    for i in range(3):
        bits = torch.empty(nbits // 4, dtype=torch.int32).pin_memory()
        bits.fill_(i)
        cache.register("v%d" % i, [torch.full((1024,), 1e-3).pin_memory()], [bits])
    order = ["v0", "v1", "v2", "v0", "v1", "v2"]
    cache.release(cache.acquire("v0"))
    cache.release(cache.acquire("v1"))
    torch.cuda.synchronize()
    before = cache.bytes_loaded
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(cache.copy_stream)
    for name in order[2:]:
        cache.release(cache.acquire(name))
    t1.record(cache.copy_stream)
    torch.cuda.synchronize()
    moved = cache.bytes_loaded - before
    ms = t0.elapsed_time(t1)
    hot = delta_cache_hot_set(torch, dev)
    return {"hot_set": hot,
            "workload": "3 variants x 1 GiB of bits through a 2 GiB device cache (LRU x rate, no hot set)",
            "loads": len(order) - 2, "bytes": moved, "ms": ms, "gbs": moved / (ms / 1e3) / 1e9}


def delta_cache_hot_set(torch, dev):
    """The page's residency policy on a request stream: 14 variants of 32 MiB
    of bits, a device cache with room for 8, 400 acquires whose variants
    follow a Zipf(1.1) mix (a fake clock advancing 10 ms per request).  Loads
    and hit rate with the six most requested variants kept resident, beside
    the same stream through plain rate-weighted LRU."""
    from bit_delta_compressed_gb300.cache import DeltaCache
    import workloads as wl
    V, nbits, reqs = 14, 32 << 20, 400
    order = wl.variant_ids_zipf(reqs, V, 1.1, wl.generator(77)).tolist()
    host = [torch.full((nbits // 4,), v, dtype=torch.int32).pin_memory() for v in range(V)]
    scales = [torch.full((64,), 1e-3).pin_memory() for _ in range(V)]
    out = {}
    for k in (6, 0):
        t = [0.0]
        cache = DeltaCache(8 * (nbits + 256) + 4096, dev, pinned_top_k=k, clock=lambda: t[0])
        for v in range(V):
            cache.register("v%d" % v, [scales[v]], [host[v]])
        for v in order:
            t[0] += 0.01
            cache.release(cache.acquire("v%d" % v))
        torch.cuda.synchronize()
        loads = sum(st.loads for st in cache.stats.values())
        out["top%d" % k] = {"loads": loads, "hit_rate": 1.0 - loads / reqs,
                            "resident": cache.resident_names()}
        del cache
    torch.cuda.empty_cache()
    out["workload"] = "14 variants x 32 MiB, room for 8, 400 Zipf(1.1) requests"
    return out


def pick_path(bd, preferred, call):
    """``preferred`` if the library takes it for this shape, else "auto"."""
    try:
        call(preferred)
        return preferred
    except bd.BitDeltaError as e:
        if e.code != bd.BD_ERR_UNSUPPORTED:
            raise
        return "auto"


def run_only(args):
    import torch
    import bit_delta_compressed_gb300 as bd
    import workloads as wl
    bd.get_lib()
    dev = torch.device("cuda", 0)
    pk, _ = peaks()
    rows = run_rows(args, torch, bd, wl, dev, pk, which=(args.only,))
    print(json.dumps({"rows": rows}), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    if args.only:
        run_only(args)
        return
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    if len(sys.argv) > 1 and sys.argv[1] == "--digest":
        print(sources_digest(KERNEL_SOURCES[sys.argv[2]]))
    else:
        main()
