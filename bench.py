#!/usr/bin/env python
"""Benchmark of the weight-only quantized matmul (W4A16 decode by default).

One step = one wq_matmul (the whole hot path: weight stream, in-register
dequant, tensor-core MMA, group rescale, epilogue) over one batch of
synthetic input with the weights resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--m M] [--no-sweep]

Prints ONE JSON line (rank 0).  Timing: W untimed steps plus a short hold of
the same launches, then exactly K steps replayed from CUDA graphs on the
launching stream, bracketed by a barrier and torch.cuda.synchronize(), timed
with CUDA events; the weights, scales, zeros, x and y rotate over buffer sets
whose total footprint exceeds 3x the L2 size, so every step streams its
weights from HBM.  For N > 1 (torchrun) every rank runs an independent
replica (the path needs no exchange) and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A16 effective weight GB/s and TFLOP/s at M=1..1024; % of HBM / bf16 MMA roofline"
UNIT = "GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="int4_asym_sweep")
    ap.add_argument("--m", type=int, default=16)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--hold-s", type=float, default=0.6, help="seconds of identical launches before the timed region")
    ap.add_argument("--kernel-only", action="store_true",
                    help="only the timed kernel launches (no e2e, sweep, CPU baseline or clocks): for profilers")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """C/CUDA source with comments and blank space removed: edits to comments
    or layout leave the compiled kernels, and so a capture of them, unchanged."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def sources_sha() -> str:
    """Hash of the kernel sources' code, to tie an ncu capture to the kernels it measured."""
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "weight_only_quantized_wq_gb300", "csrc", "*"))):
        h.update(os.path.basename(f).encode() + b"\0" + _code_only(open(f, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def traffic_for(key: str):
    """DRAM bytes per launch from a committed ncu summary, only if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(key)
    if not d or d.get("sources_sha") != sources_sha():
        return None
    return d.get("bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[2 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ GPU timing
def make_sets(p, torch, wq, l2_bytes):
    """Rotating device copies of one problem, total footprint >= 3x L2."""
    per = p.total_bytes()
    nset = max(2, -(-3 * l2_bytes // per))
    nset = min(nset, 64)
    base_packed = wq.wq_pack(p.qweight.cuda(), p.K, p.N, p.w_bit)
    sets = []
    for i in range(nset):
        sets.append({
            "x": p.x.cuda(),
            "packed": base_packed if i == 0 else base_packed.clone(),
            "scales": p.scales.cuda(),
            "zeros": None if p.zeros is None else p.zeros.cuda(),
            "out": torch.empty((p.M, p.N), dtype=torch.float32, device="cuda"),
        })
    ws = wq.binding.workspace_for(p.M, p.N, p.K, p.w_bit, p.group_size, "cuda")
    return sets, ws


def call(p, s, wq, ws):
    wq.wq_matmul(s["x"], s["packed"], s["scales"], s["zeros"], p.M, p.N, p.K, p.w_bit, p.group_size,
                 out=s["out"], workspace=ws)


def capture(p, sets, ws, n, start, torch, wq):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            call(p, sets[(start + i) % len(sets)], wq, ws)
    return g


def time_graphs(p, sets, ws, steps, warmup, torch, wq, hold_s=0.0, dist=None):
    """Warm-up, an optional hold, then exactly `steps` launches from graphs; returns seconds."""
    call(p, sets[0], wq, ws)  # first call sets kernel attributes outside capture
    torch.cuda.synchronize()
    chunk = min(steps, 100)
    g = capture(p, sets, ws, chunk, 0, torch, wq)
    rem = steps % chunk
    g_rem = capture(p, sets, ws, rem, 0, torch, wq) if rem else None
    gw = capture(p, sets, ws, max(1, warmup), 0, torch, wq)
    gw.replay()
    torch.cuda.synchronize()
    if hold_s > 0:
        t0 = time.time()
        while time.time() - t0 < hold_s:
            g.replay()
            torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps // chunk):
        g.replay()
    if g_rem is not None:
        g_rem.replay()
    e1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1) / 1e3


def uses_prefill(p) -> bool:
    """The library takes its tensor-core path for 65+ tokens of int4 codes whose
    group size is a multiple of 64 and whose scales have the x dtype."""
    return p.M >= 65 and p.w_bit == 4 and p.group_size % 64 == 0 and p.x_dtype == p.s_dtype


def kernel_name(p) -> str:
    if uses_prefill(p):
        return "prefill_kernel (tcgen05)"
    return "decode_kernel" if p.M <= 64 else "decode_kernel (64-row slices)"


def launches_per_call(p) -> int:
    return 1 if uses_prefill(p) else -(-p.M // 64)


def time_e2e(p, sets, ws, steps, warmup, torch, wq):
    """Public API with host buffers, as a serving loop runs it: every step copies
    its x from pinned host memory (H2D stream), calls wq_matmul (the launching
    stream) and copies its y back to pinned host memory (D2H stream).  Events
    order each step's copies around its call, and a buffer set is reused only
    after its previous y has reached the host, so the copies of one step overlap
    the kernels of its neighbours.  CUDA events on the launching stream bracket
    all steps (it waits for the last D2H copy before the closing event)."""
    n = len(sets)
    xh = [s["x"].cpu().pin_memory() for s in sets]
    yh = [torch.empty((p.M, p.N), dtype=torch.float32).pin_memory() for _ in range(n)]
    main = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    x_in = [torch.cuda.Event() for _ in range(n)]
    y_out = [torch.cuda.Event() for _ in range(n)]
    y_home = [torch.cuda.Event() for _ in range(n)]  # the set's last y is in host memory
    used = [False] * n

    def step(i):
        k = i % n
        s = sets[k]
        with torch.cuda.stream(h2d_s):
            if used[k]:
                h2d_s.wait_event(y_home[k])
            s["x"].copy_(xh[k], non_blocking=True)
            x_in[k].record(h2d_s)
        main.wait_event(x_in[k])
        call(p, s, wq, ws)
        y_out[k].record(main)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(y_out[k])
            yh[k].copy_(s["out"], non_blocking=True)
            y_home[k].record(d2h_s)
        used[k] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    h2d_s.wait_event(e0)  # the first copy starts inside the timed region
    for i in range(steps):
        step(i)
    main.wait_stream(d2h_s)
    e1.record(main)
    torch.cuda.synchronize()
    h2d = p.x.numel() * p.x.element_size()
    return e0.elapsed_time(e1) / 1e3, h2d, p.M * p.N * 4


def roofline_entry(p, sec_per_launch, pk, src):
    if p.M >= 256:
        achieved = p.flops / sec_per_launch / 1e12
        peak = pk["bf16_tflops"]
        return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "peak_source": src + " bf16 burst"}
    achieved = p.total_bytes() / sec_per_launch / 1e9
    peak = pk["hbm_gbs"]
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": src + " copy bandwidth"}


def sweep(torch, wq, syn, l2, pk, src):
    out = []
    c5 = syn.int4_asym_sweep(4096)
    problems = [syn.int4_asym_tiny(), syn.int8_per_channel(), syn.int4_sym_decode(), syn.int2_asym()]
    problems += [c5.rows(m) for m in syn.C5_MS]
    for p in problems:
        sets, ws = make_sets(p, torch, wq, l2)
        n = 50 if p.M <= 256 else 10
        sec = time_graphs(p, sets, ws, n, 5, torch, wq) / n
        e = {"workload": p.name, "M": p.M, "kernel": kernel_name(p), "us": round(sec * 1e6, 2),
             "weight_GBps": round(p.weight_bytes() / sec / 1e9, 1),
             "total_GBps": round(p.total_bytes() / sec / 1e9, 1),
             "TFLOPs": round(p.flops / sec / 1e12, 2),
             "roofline": roofline_entry(p, sec / launches_per_call(p) * launches_per_call(p), pk, src)}
        out.append(e)
        del sets
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ oracle (CPU)
def oracle_step(p, ncols, threads):
    """The CPU oracle over the first `ncols` columns of the workload (all rows)."""
    import concurrent.futures as cf
    import oracle
    blk = max(16, ncols // (threads * 2) // 16 * 16)
    edges = list(range(0, ncols, blk)) + [ncols]

    def part(i):
        n0, n1 = edges[i], edges[i + 1]
        if p.w_bit == 8:
            return oracle.matmul_int8(p.x, p.x_dtype == "bf16", p.qweight, p.scales, p.M, p.N, p.K, n0=n0, n1=n1)
        return oracle.matmul_grouped(p.x, p.x_dtype == "bf16", p.qweight.numpy(), p.scales, p.s_dtype == "bf16",
                                     None if p.zeros is None else p.zeros.numpy(), p.M, p.N, p.K, p.w_bit,
                                     p.group_size, n0=n0, n1=n1)

    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(part, range(len(edges) - 1)))


def sample_cols(p, target_cols_frac=1.0):
    return max(16, int(p.N * target_cols_frac) // 16 * 16)


def cpu_measure(p, steps, warmup, min_seconds=0.0):
    """Time the oracle on a column sample; returns (GB/s of weight bytes covered,
    cores, sample text, seconds per step).  At least `steps` steps, and more
    (up to 200) until `min_seconds` of CPU work have been timed."""
    threads = os.cpu_count() or 1
    ncols = sample_cols(p)
    for _ in range(warmup):
        oracle_step(p, ncols, threads)
    t0 = time.perf_counter()
    done = 0
    while done < steps or (time.perf_counter() - t0 < min_seconds and done < 200):
        oracle_step(p, ncols, threads)
        done += 1
    dt = (time.perf_counter() - t0) / done
    wbytes = p.weight_bytes() * ncols / p.N
    sample = "all %d rows x first %d of %d columns (K=%d) per step, %d steps (%.1f s)" % (
        p.M, ncols, p.N, p.K, done, dt * done)
    return wbytes / dt / 1e9, threads, sample, dt


def max_over_ranks(sec, dist, torch, device="cuda"):
    """The job's time: the slowest rank's (every rank times the same number of steps)."""
    if dist is None:
        return sec
    t = torch.tensor([sec], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(world, weight_bytes, steps, sec):
    """Whole-job throughput: the weight bytes every rank streamed over the job's time."""
    return world * weight_bytes * steps / sec / 1e9


def get_problem(args):
    from weight_only_quantized_wq_gb300 import synthetic as syn
    f = syn.WORKLOADS[args.workload]
    return f(args.m) if args.workload == "int4_asym_sweep" else f()


def config_of(p, extra=None):
    c = {"workload": p.name, "M": p.M, "K": p.K, "N": p.N, "w_bit": p.w_bit, "group_size": p.group_size,
         "x_dtype": p.x_dtype, "scale_dtype": p.s_dtype, "accumulate": "fp32", "output": "fp32"}
    c.update(extra or {})
    return c


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        import oracle
        oracle.build()
        p = get_problem(args)
        steps = max(1, min(args.steps, 20))
        warm = max(0, min(args.warmup, 3))
        gbps, cores, sample, dt = cpu_measure(p, steps, warm)
        line = {"impl": "reference", "metric": METRIC, "value": round(gbps, 3), "unit": UNIT, "n_gpus": args.gpus,
                "steps": steps, "warmup": warm, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config_of(p), "cpu_baseline": {"kind": "oracle", "value": round(gbps, 3), "unit": UNIT,
                                                         "cores": cores, "sample": sample},
                "e2e": {"value": round(gbps, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    dist = None
    if world > 1:
        import torch.distributed as td
        torch.cuda.set_device(local)
        td.init_process_group("nccl", init_method="env://")
        dist = td
    import weight_only_quantized_wq_gb300 as wq
    from weight_only_quantized_wq_gb300 import build as wqbuild
    from weight_only_quantized_wq_gb300 import synthetic as syn
    if rank == 0:
        wqbuild.build()
    if dist is not None:
        dist.barrier()
    wq.binding.lib()
    torch.cuda.set_device(local)
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    pk, pk_src = peaks()

    p = get_problem(args)
    sets, ws = make_sets(p, torch, wq, l2)
    clocks = ClockSampler(local)
    if not args.kernel_only:
        clocks.start()
    sec = time_graphs(p, sets, ws, args.steps, args.warmup, torch, wq, hold_s=0 if args.kernel_only else args.hold_s,
                      dist=dist)
    clk = None if args.kernel_only else clocks.stop()
    sec = max_over_ranks(sec, dist, torch)
    per_step = sec / args.steps
    value = job_gbps(world, p.weight_bytes(), args.steps, sec)
    lpc = launches_per_call(p)
    roof = roofline_entry(p, per_step, pk, pk_src)
    key = "%s|M=%d" % (args.workload, p.M)
    roof["traffic"] = traffic_for(key)
    roof["kernel"] = kernel_name(p)
    roof["launch_us"] = round(per_step / lpc * 1e6, 3)

    if args.kernel_only:
        e2e_sec, h2d, d2h = sec, 0, 0
    else:
        e2e_sec, h2d, d2h = time_e2e(p, sets, ws, args.steps, args.warmup, torch, wq)
    e2e_sec = max_over_ranks(e2e_sec, dist, torch)
    e2e_val = job_gbps(world, p.weight_bytes(), args.steps, e2e_sec)

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(p, {"parallelism": "replicas" if world > 1 else "single GPU",
                                    "l2": "rotating %d buffer sets, %.0f MB total > 3x L2 (%.0f MB)" % (
                                        len(sets), len(sets) * p.total_bytes() / 1e6, l2 / 1e6),
                                    "tflops": round(p.flops * args.steps / sec / 1e12, 3)}),
            "roofline": roof,
            "e2e": {"value": round(e2e_val, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * lpc,
            "clocks": clk}
    if rank == 0:
        del sets
        torch.cuda.empty_cache()
        if not args.no_sweep and not args.kernel_only:
            line["sweep"] = sweep(torch, wq, syn, l2, pk, pk_src)
        if not args.kernel_only:
            gbps, cores, sample, _ = cpu_measure(p, 1, 1, min_seconds=10.0)
            line["cpu_baseline"] = {"value": round(gbps, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": sample}
        print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
