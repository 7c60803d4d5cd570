#!/usr/bin/env python
"""Benchmark of the weight-only quantized matmul (W4A16 decode by default).

One step = one wq_matmul (the whole hot path: weight stream, in-register
dequant, tensor-core MMA, group rescale, epilogue) over one batch of
synthetic input with the weights resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--m M] [--out-dtype f32|f16|bf16] [--no-sweep]

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
    ap.add_argument("--out-dtype", choices=["f32", "f16", "bf16"], default="f32")
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
class Bench:
    """One workload on the GPU: rotating device copies of its inputs (total
    footprint >= 3x L2, so every step streams its weights from HBM), and the
    library call a step makes.  Grouped / int8 problems go through
    wq_matmul_ex (out_dtype fp32, fp16 or bf16), ternary ones through
    wq_t2_matmul."""

    def __init__(self, p, torch, wq, l2_bytes, out_dtype="f32"):
        self.p, self.torch, self.wq = p, torch, wq
        self.ternary = not hasattr(p, "w_bit")
        self.odt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[out_dtype]
        self.out_dtype = out_dtype
        per = p.total_bytes()
        nset = min(64, max(2, -(-3 * l2_bytes // per)))
        if self.ternary:
            base = wq.wq_t2_pack(p.packed.cuda(), p.K, p.N)
        else:
            base = wq.wq_pack(p.qweight.cuda(), p.K, p.N, p.w_bit)
        self.sets = []
        for i in range(nset):
            st = {"x": p.x.cuda(), "packed": base if i == 0 else base.clone()}
            if self.ternary:
                st["out"] = torch.empty((p.M, p.N), dtype=torch.int32, device="cuda")
            else:
                st["scales"] = p.scales.cuda()
                st["zeros"] = None if p.zeros is None else p.zeros.cuda()
                st["out"] = torch.empty((p.M, p.N), dtype=self.odt, device="cuda")
            self.sets.append(st)
        if self.ternary:
            need = wq.wq_t2_workspace_bytes(p.M, p.N, p.K)
            self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
        else:
            self.ws = wq.binding.workspace_for(p.M, p.N, p.K, p.w_bit, p.group_size, "cuda")

    def call(self, i):
        p, s = self.p, self.sets[i % len(self.sets)]
        if self.ternary:
            self.wq.wq_t2_matmul(s["x"], s["packed"], p.M, p.N, p.K, out=s["out"], workspace=self.ws)
        else:
            self.wq.wq_matmul_ex(s["x"], s["packed"], s["scales"], s["zeros"], p.M, p.N, p.K, p.w_bit,
                                 p.group_size, out=s["out"], out_dtype=self.odt, workspace=self.ws)

    def path(self) -> int:
        if self.ternary:
            return 0
        return self.wq.wq_matmul_path(self.p.M, self.p.N, self.p.K, self.p.w_bit, self.p.group_size,
                                      self.p.x.dtype, self.p.scales.dtype)

    def kernel_name(self) -> str:
        k = self.wq.binding.PATHS[self.path()]
        if self.path() == 0 and self.p.M > 64:
            k += " (64-row slices)"
        return k

    def launches_per_call(self) -> int:
        if self.path() != 0:
            return 1
        return -(-self.p.M // 64) + (1 if self.ternary else 0)

    def out_bytes(self) -> int:
        return self.p.M * self.p.N * self.sets[0]["out"].element_size()

    def total_bytes(self) -> int:
        """Algorithmic bytes of one call with this output type."""
        return self.p.total_bytes() - self.p.M * self.p.N * 4 + self.out_bytes()


def capture(b, n, torch, start=0):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            b.call(start + i)
    return g


def replay_timed(graphs, torch, dist=None):
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for g in graphs:
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1) / 1e3


def time_graphs(b, steps, warmup, torch, hold_s=0.0, dist=None):
    """Warm-up, an optional hold, then exactly `steps` calls replayed from CUDA
    graphs on the launching stream; returns seconds."""
    b.call(0)  # the first call sets kernel attributes and plans outside capture
    torch.cuda.synchronize()
    chunk = min(steps, 100)
    g = capture(b, chunk, torch)
    rem = steps % chunk
    g_rem = capture(b, rem, torch) if rem else None
    gw = capture(b, max(1, warmup), torch)
    gw.replay()
    torch.cuda.synchronize()
    if hold_s > 0:
        t0 = time.time()
        while time.time() - t0 < hold_s:
            g.replay()
            torch.cuda.synchronize()
    return replay_timed([g] * (steps // chunk) + ([g_rem] if g_rem is not None else []), torch, dist)


def time_e2e(b, steps, warmup, torch, graph=True):
    """The public API with host buffers, as a serving loop runs it: every step
    copies its x from pinned host memory (H2D stream), makes the library call
    (the launching stream) and copies its y back to pinned host memory (D2H
    stream).  Events order each step's copies around its call, and a buffer
    set is reused only after its previous y has reached the host, so the copies
    of one step overlap the kernels of its neighbours.  graph=True captures the
    steps in CUDA graphs (as a serving loop that replays its decode step does;
    the copies stay inside every step), graph=False issues them from Python.
    CUDA events on the launching stream bracket all steps."""
    p = b.p
    n = len(b.sets)
    xh = [s["x"].cpu().pin_memory() for s in b.sets]
    yh = [torch.empty_like(s["out"], device="cpu").pin_memory() for s in b.sets]
    main = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    x_in = [torch.cuda.Event() for _ in range(n)]
    y_out = [torch.cuda.Event() for _ in range(n)]
    y_home = [torch.cuda.Event() for _ in range(n)]  # the set's last y is in host memory
    used = [False] * n

    def step(i):
        k = i % n
        s = b.sets[k]
        cur = torch.cuda.current_stream()
        h2d_s.wait_stream(cur) if not used[k] else None
        with torch.cuda.stream(h2d_s):
            if used[k]:
                h2d_s.wait_event(y_home[k])
            s["x"].copy_(xh[k], non_blocking=True)
            x_in[k].record(h2d_s)
        cur.wait_event(x_in[k])
        b.call(k)
        y_out[k].record(cur)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(y_out[k])
            yh[k].copy_(s["out"], non_blocking=True)
            y_home[k].record(d2h_s)
        used[k] = True

    h2d = p.x.numel() * p.x.element_size()
    d2h = b.out_bytes()
    if not graph:
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
        return e0.elapsed_time(e1) / 1e3, h2d, d2h

    def capture_steps(cnt):
        for k in range(n):
            used[k] = False
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cur = torch.cuda.current_stream()
            for i in range(cnt):
                step(i)
            cur.wait_stream(h2d_s)
            cur.wait_stream(d2h_s)
        return g

    b.call(0)
    torch.cuda.synchronize()
    chunk = min(steps, 100)
    g = capture_steps(chunk)
    rem = steps % chunk
    g_rem = capture_steps(rem) if rem else None
    gw = capture_steps(max(1, min(warmup, chunk)))
    gw.replay()
    torch.cuda.synchronize()
    sec = replay_timed([g] * (steps // chunk) + ([g_rem] if g_rem is not None else []), torch)
    return sec, h2d, d2h


# ------------------------------------------------------------------ read-only floor
_floor_lib = None


def floor_us(nbytes, l2, torch, sms):
    """Best time (us) of the read-only streaming kernel (libwqfloor.so) reading
    nbytes once, over rotating buffers > 3x L2, replayed from CUDA graphs, over
    a few launch shapes: the practical floor of any kernel that must read
    those bytes once."""
    global _floor_lib
    import ctypes
    from weight_only_quantized_wq_gb300 import build as wqbuild
    if _floor_lib is None:
        _floor_lib = ctypes.CDLL(wqbuild.build_floor())
        _floor_lib.wq_floor_read.restype = ctypes.c_int
        _floor_lib.wq_floor_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_void_p]
    nb = (nbytes + 15) // 16 * 16
    nbuf = min(64, max(2, -(-3 * l2 // nb)))
    bufs = [torch.empty(nb, dtype=torch.uint8, device="cuda").fill_(i) for i in range(nbuf)]
    best = None
    for blocks in (sms * 2, sms * 4, sms * 8, sms * 16):
        for threads in (256, 512, 1024):
            sink = torch.zeros(blocks, dtype=torch.int32, device="cuda")
            st = torch.cuda.current_stream().cuda_stream

            def launch(i):
                rc = _floor_lib.wq_floor_read(bufs[i % nbuf].data_ptr(), nb, sink.data_ptr(), blocks, threads, st)
                assert rc == 0, rc
            launch(0)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                st = torch.cuda.current_stream().cuda_stream
                for i in range(50):
                    launch(i)
            g.replay()
            torch.cuda.synchronize()
            sec = min(replay_timed([g], torch) for _ in range(3)) / 50
            best = sec if best is None or sec < best else best
    del bufs
    torch.cuda.empty_cache()
    return best * 1e6


def roofline_entry(b, sec_per_call, pk, src, floor=None):
    """Bound from the algorithmic bytes and FLOP against the measured peaks:
    whichever takes longer at its peak decides the bound."""
    p = b.p
    nbytes, flops = b.total_bytes(), p.flops
    tensor = flops / (pk["bf16_tflops"] * 1e12) > nbytes / (pk["hbm_gbs"] * 1e9)
    if tensor:
        achieved = flops / sec_per_call / 1e12
        peak = pk["bf16_tflops"]
        e = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
             "frac": round(achieved / peak, 4), "peak_source": src + " bf16 burst"}
    else:
        achieved = nbytes / sec_per_call / 1e9
        peak = pk["hbm_gbs"]
        e = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
             "frac": round(achieved / peak, 4), "peak_source": src + " copy bandwidth",
             "frac_weights_of_8000GBps": round(p.weight_bytes() / sec_per_call / 8e12, 4)}
        if floor is not None:
            e["floor_us"] = round(floor, 2)
            e["frac_of_floor"] = round(floor / (sec_per_call * 1e6), 4)
    return e


def sweep(torch, wq, syn, l2, pk, src, sms):
    out = []
    c5 = syn.int4_asym_sweep(4096)
    runs = [(syn.int4_asym_tiny(), "f32", "int4_asym_tiny|M=1"), (syn.int8_per_channel(), "f32", "int8_per_channel|M=16"),
            (syn.int4_sym_decode(), "f32", "int4_sym_decode|M=1"), (syn.int2_asym(), "f32", "int2_asym|M=8")]
    runs += [(c5.rows(m), "f32", "int4_asym_sweep|M=%d" % m) for m in syn.C5_MS]
    runs += [(c5.rows(16), "bf16", "int4_asym_sweep|M=16|out=bf16"),
             (c5.rows(1024), "bf16", "int4_asym_sweep|M=1024|out=bf16"),
             (syn.ternary_decode(), "s32", "ternary_decode|M=16"),
             (syn.int4_asym_short_k(128), "f32", "int4_asym_short_k|M=128"),
             (syn.int4_asym_short_k(1024), "f32", "int4_asym_short_k|M=1024")]
    for p, odt, key in runs:
        b = Bench(p, torch, wq, l2, out_dtype="f32" if odt == "s32" else odt)
        n = 50 if p.M <= 256 else 10
        sec = time_graphs(b, n, 5, torch) / n
        e = {"workload": p.name, "M": p.M, "out": odt, "kernel": b.kernel_name(), "us": round(sec * 1e6, 2),
             "weight_GBps": round(p.weight_bytes() / sec / 1e9, 1),
             "total_GBps": round(b.total_bytes() / sec / 1e9, 1),
             "TFLOPs": round(p.flops / sec / 1e12, 2)}
        fl = floor_us(b.total_bytes(), l2, torch, sms) if p.M <= 64 else None
        e["roofline"] = roofline_entry(b, sec, pk, src, fl)
        e["roofline"]["traffic"] = traffic_for(key)
        out.append(e)
        del b
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ oracle (CPU)
def oracle_part(p, n0, n1):
    import oracle
    if not hasattr(p, "w_bit"):
        return oracle.t2_matmul(p.x, p.packed[:, n0:n1].contiguous(), p.M, n1 - n0, p.K)
    if p.w_bit == 8:
        return oracle.matmul_int8(p.x, p.x_dtype == "bf16", p.qweight, p.scales, p.M, p.N, p.K, n0=n0, n1=n1)
    return oracle.matmul_grouped(p.x, p.x_dtype == "bf16", p.qweight.numpy(), p.scales, p.s_dtype == "bf16",
                                 None if p.zeros is None else p.zeros.numpy(), p.M, p.N, p.K, p.w_bit,
                                 p.group_size, n0=n0, n1=n1)


def oracle_step(p, ncols, threads):
    """The CPU oracle over the first `ncols` columns of the workload (all rows),
    split into column blocks over `threads` threads (its C code releases the GIL)."""
    import concurrent.futures as cf
    blk = max(16, ncols // (threads * 2) // 16 * 16)
    edges = list(range(0, ncols, blk)) + [ncols]
    if threads == 1:
        for i in range(len(edges) - 1):
            oracle_part(p, edges[i], edges[i + 1])
        return
    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda i: oracle_part(p, edges[i], edges[i + 1]), range(len(edges) - 1)))


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        fields = {}
        for line in out.splitlines():
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
        name = fields.get("Model name") or fields.get("Vendor ID") or "unknown"
        return "%s (%s cores)" % (name, fields.get("CPU(s)", "?"))
    except (OSError, subprocess.TimeoutExpired):
        return "unknown"


def cpu_measure(p, steps, warmup, min_seconds=0.0, threads=None, ncols=None):
    """Time the oracle on a column sample; returns (GB/s of weight bytes covered,
    threads, sample text, seconds per step).  At least `steps` steps, and more
    (up to 200) until `min_seconds` of CPU work have been timed."""
    threads = threads or os.cpu_count() or 1
    ncols = ncols or p.N
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


def cpu_baseline(p):
    """The oracle on every host core (about 10 s), and on one core over a
    column slice (about 3 s)."""
    gbps, cores, sample, _ = cpu_measure(p, 1, 1, min_seconds=10.0)
    one_cols = max(16, p.N // 16 // 16 * 16)
    g1, _, s1, _ = cpu_measure(p, 1, 0, min_seconds=3.0, threads=1, ncols=one_cols)
    return {"value": round(gbps, 3), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
            "cpu_model": cpu_model(), "single_thread_value": round(g1, 4), "single_thread_sample": s1}


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
    return f(args.m) if args.workload in ("int4_asym_sweep", "int4_asym_short_k") else f()


def config_of(p, extra=None, out="fp32"):
    if not hasattr(p, "w_bit"):
        c = {"workload": p.name, "M": p.M, "K": p.K, "N": p.N, "w_bit": 2, "scheme": "ternary planar (Liger)",
             "x_dtype": "int8", "accumulate": "exact integer", "output": "int32"}
    else:
        c = {"workload": p.name, "M": p.M, "K": p.K, "N": p.N, "w_bit": p.w_bit, "group_size": p.group_size,
             "x_dtype": p.x_dtype, "scale_dtype": p.s_dtype, "accumulate": "fp32", "output": out}
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
        steps, warm = max(1, args.steps), max(0, args.warmup)
        # Exactly the requested steps, each a column sample of the workload sized
        # so that the whole run takes about two minutes of host time.
        threads = os.cpu_count() or 1
        t0 = time.perf_counter()
        oracle_step(p, p.N, threads)
        full = time.perf_counter() - t0
        per_step = 120.0 / (steps + warm)
        ncols = max(16, min(p.N, int(p.N * per_step / full) // 16 * 16))
        gbps, cores, sample, dt = cpu_measure(p, steps, warm, ncols=ncols)
        line = {"impl": "reference", "metric": METRIC, "value": round(gbps, 3), "unit": UNIT, "n_gpus": args.gpus,
                "steps": steps, "warmup": warm, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config_of(p), "cpu_baseline": {"kind": "oracle", "value": round(gbps, 3), "unit": UNIT,
                                                         "cores": cores, "sample": sample,
                                                         "cpu_model": cpu_model()},
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
        wqbuild.build_floor()
    if dist is not None:
        dist.barrier()
    wq.binding.lib()
    torch.cuda.set_device(local)
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    sms = props.multi_processor_count
    pk, pk_src = peaks()

    p = get_problem(args)
    b = Bench(p, torch, wq, l2, out_dtype=args.out_dtype)
    clocks = ClockSampler(local)
    if not args.kernel_only:
        clocks.start()
    sec = time_graphs(b, args.steps, args.warmup, torch, hold_s=0 if args.kernel_only else args.hold_s, dist=dist)
    clk = None if args.kernel_only else clocks.stop()
    sec = max_over_ranks(sec, dist, torch)
    per_step = sec / args.steps
    value = job_gbps(world, p.weight_bytes(), args.steps, sec)
    lpc = b.launches_per_call()
    fl = None
    if not args.kernel_only and rank == 0 and p.M <= 64:
        fl = floor_us(b.total_bytes(), l2, torch, sms)
    roof = roofline_entry(b, per_step, pk, pk_src, fl)
    key = "%s|M=%d" % (args.workload, p.M) + ("" if args.out_dtype == "f32" else "|out=" + args.out_dtype)
    roof["traffic"] = traffic_for(key)
    roof["kernel"] = b.kernel_name()
    roof["launch_us"] = round(per_step / lpc * 1e6, 3)

    if args.kernel_only:
        e2e_sec, h2d, d2h, eager_sec = sec, 0, 0, None
    else:
        e2e_sec, h2d, d2h = time_e2e(b, args.steps, args.warmup, torch, graph=True)
        eager_sec, _, _ = time_e2e(b, min(args.steps, 500), args.warmup, torch, graph=False)
        eager_sec = eager_sec * args.steps / min(args.steps, 500)
    e2e_sec = max_over_ranks(e2e_sec, dist, torch)
    e2e_val = job_gbps(world, p.weight_bytes(), args.steps, e2e_sec)
    e2e = {"value": round(e2e_val, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if eager_sec is not None:
        e2e["mode"] = "steps replayed from CUDA graphs (H2D copy, call, D2H copy in every step)"
        e2e["eager_value"] = round(job_gbps(world, p.weight_bytes(), args.steps, max_over_ranks(eager_sec, dist,
                                                                                             torch)), 1)
        e2e["eager_mode"] = "the same steps issued from Python every step (host-bound)"

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if hasattr(p, "w_bit") else "int8",
            "data": "synthetic",
            "config": config_of(p, out={"f32": "fp32", "f16": "fp16", "bf16": "bf16"}[args.out_dtype]),
            "timing": {"parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "rotating %d buffer sets, %.0f MB total > 3x L2 (%.0f MB)" % (
                           len(b.sets), len(b.sets) * b.total_bytes() / 1e6, l2 / 1e6),
                       "tflops": round(p.flops * args.steps / sec / 1e12, 3)},
            "roofline": roof,
            "e2e": e2e,
            "gpu_launches": args.steps * lpc,
            "clocks": clk}
    if rank == 0:
        del b
        torch.cuda.empty_cache()
        if not args.no_sweep and not args.kernel_only:
            line["sweep"] = sweep(torch, wq, syn, l2, pk, pk_src, sms)
        if not args.kernel_only:
            line["cpu_baseline"] = cpu_baseline(p)
        print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
