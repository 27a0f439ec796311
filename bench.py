"""Benchmark of the FP8 linear-layer hot path on GB300.

One step = the per-token FP8 cast of X (1x128 groups, UE8M0 scales packed
four exponents per int32 word, written M-major) followed by the block-scaled
GEMM D = X W^T (bf16 out), over the
large cast+GEMM workload: X bf16 [16384, 7168] randn, W bf16 [18432, 7168]
randn * 0.02 cast once to E4M3 with 128x128 UE8M0 block scales (outside the
timed region, as a weight cast runs once per weight update). Inputs are
synthetic and seeded; they are larger than L2, so no flush is needed.

Prints one JSON line (rank 0). Keys: metric/value/unit (GEMM TFLOP/s of the
whole step), ms_per_step, timed_region (the block of K steps is repeated R
times so the timed region lasts at least --min-timed-s under the clock
sampler; value and ms_per_step cover all R*K steps), roofline (dominant
kernel: the GEMM, against the dense FP8 peak = 2x the measured bf16 peak, with
p10/median/p90 of its launches, a clock-normalised fraction and the ncu
tensor-pipe counter of its committed capture), cast (GB/s of the cast kernel
against measured HBM bandwidth), cast_sweep (the pages' per-token cast sweep:
tokens 1 ... 16384 at hidden 4096, groups 32/128, three scale formats, bf16
and fp32 input, eager and CUDA-graph, cold L2, plus one hot-L2 point),
workloads (the smaller configurations, each eager and CUDA-graph with
median/p10/p90: tiny fwd with fp32 scales, forward GEMMs at M = 64/128/4096
with packed and fp32 scales, the Linear fwd+dgrad+wgrad step with packed and
fp32 scales, the fused cast, the grouped GEMM, the low-latency cast, small-M
GEMMs back to back), e2e (host buffers, copies inside the timed region),
cpu_baseline (the CPU oracle on a bounded sample of this workload),
cpu_baselines (the oracle timed in full on the smaller configurations and the
cast single-threaded and on all cores), clocks (nvidia-smi samples inside the
timed region), gpu_launches. e2e runs the library's host-buffer call, which
overlaps the copies of one row chunk with the kernels of the next.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica (rows are independent:
weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "large_cast_gemm_16384x18432x7168_ue8m0"
METRIC = "block-scaled FP8 GEMM TFLOP/s (% FP8 peak); per-token cast GB/s (% HBM)"
UNIT = "TFLOP/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--m", type=int, default=16384)
    ap.add_argument("--n", type=int, default=18432)
    ap.add_argument("--k", type=int, default=7168)
    ap.add_argument("--fmt", choices=["ue8m0", "packed", "fp32"], default="packed")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads (small-M GEMMs, Linear step, low-latency cast)")
    ap.add_argument("--only-workloads", action="store_true",
                    help="run only the other workloads and print them as one JSON line")
    ap.add_argument("--reps", type=int, default=100, help="timed repetitions per other workload")
    ap.add_argument("--min-timed-s", type=float, default=0.5,
                    help="the block of K timed steps is repeated until the timed region lasts this long")
    ap.add_argument("--e2e-chunk", type=int, default=1024, help="rows per step of the host-buffer pipeline")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU-oracle sample time")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sus": p.get("bf16_tflops_sustained"),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples, each stamped with the host
    time it arrived, so that only the samples inside the timed region count."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.stamps = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.stamps.append(time.perf_counter())
            self.lines.append(line.strip())

    def stop(self, window=None):
        """Median SM clock, max clock and active throttle reasons of the
        samples (those stamped inside `window` = (t0, t1) when given)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        lines = self.lines
        if window is not None and len(self.stamps) == len(self.lines):
            lines = [ln for t, ln in zip(self.stamps, self.lines) if window[0] <= t <= window[1]]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


def recorded_counters(kernel_file: str):
    """The committed ncu counters of the GEMM kernel's launch (dict), or None
    when the kernel sources changed since they were taken."""
    import hashlib
    rec = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(rec):
        return None
    with open(rec) as fh:
        data = json.load(fh)
    h = hashlib.sha256()
    for f in data.get("sources", []):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    entry = data.get("kernels", {}).get(kernel_file)
    if not entry or data.get("sources_sha256") != h.hexdigest():
        return None
    return entry


def recorded_traffic(kernel_file: str):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu record
    and the workload they were taken on, or (None, None) when the kernel
    sources changed since the counters were taken."""
    entry = recorded_counters(kernel_file)
    if entry is None:
        return None, None
    return entry.get("dram_bytes_per_launch"), entry.get("workload")


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ timing helpers
def stats_us(ts_ms):
    """Median, p10 and p90 (us) of per-repetition times given in ms, and the
    mean of the middle 80 %. CUDA event readings on this GPU come in steps of
    about 2.05 us, so a short kernel's median sits on one of the two steps
    around its duration; the trimmed mean, averaging over where each launch
    fell between steps, is the closer figure there."""
    xs = sorted(ts_ms)
    n = len(xs)

    def q(f):
        return xs[min(n - 1, max(0, int(round(f * (n - 1)))))]

    cut = n // 10
    mid = xs[cut:n - cut] if n - 2 * cut > 0 else xs
    return {"us": round(statistics.median(xs) * 1e3, 2), "p10": round(q(0.1) * 1e3, 2),
            "p90": round(q(0.9) * 1e3, 2), "mean_mid80": round(statistics.fmean(mid) * 1e3, 2), "n": n}


class L2Flush:
    """Leaves L2 holding none of the timed kernel's data, outside the timed
    region: a 256 MB write (L2 is 129 MB), then a 256 MB read of another
    buffer. The read evicts the write's dirty lines, so the timed kernel does
    not pay for writing them back to HBM. With the write alone it did: 10-25 %
    of the time of a 60-120 MB cast or GEMM."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.r = torch.ones(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        self.r.sum(dtype=torch.int32)


def time_eager(fn, reps, flush=None, warm=10):
    """Per-repetition device times (ms) of fn with CUDA events on the current
    stream, L2 flushed (L2Flush, outside the events) before each."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return ts


def capture(fn, per):
    """A CUDA graph of `per` back-to-back calls of fn."""
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            for _ in range(per):
                fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def time_graph(fn, reps, flush=None, per=1):
    """Per-call device times (ms) of fn replayed from a CUDA graph of `per`
    calls: each repetition flushes L2 (outside the events) and times one
    replay, divided by `per`."""
    g = capture(fn, per)
    return [t / per for t in time_eager(g.replay, reps, flush, warm=3)]


def eager_and_graph(fn, reps, flush):
    """Both timings of one workload, L2 flushed before each repetition."""
    return {"eager_cold_l2": stats_us(time_eager(fn, reps, flush)),
            "graph_cold_l2": stats_us(time_graph(fn, reps, flush))}


# ------------------------------------------------------------------ CPU oracle
def _bits(t):
    import numpy as np
    import torch
    return t.view(torch.int16).numpy().view(np.uint16)


class CpuOracleSample:
    """The CPU oracle on a bounded sample of the workload: the per-token cast
    of a slice of X's rows and the fp64 GEMM of those rows against all of W.
    W's block cast (once per weight update) is prepared before any timing,
    as on the GPU."""

    def __init__(self, n, k, fmt_code):
        import oracle
        from quantised_linear_layers_gb300 import synthetic as syn

        oracle.build()
        self.o = oracle
        self.n, self.k = n, k
        self.fmt = oracle.SF_FP32 if fmt_code == 0 else oracle.SF_UE8M0
        self.threads = oracle.num_threads()
        w = syn.randn((n, k), seed=syn.SEED_W, mul=0.02)
        self.wq, self.ws = oracle.cast_per_block(_bits(w), self.fmt)
        self.rows = max(self.threads, 8)
        x = syn.randn((self.rows, k), seed=syn.SEED_X)
        self.xb = _bits(x)

    def once(self) -> float:
        t0 = time.perf_counter()
        xq, xs = self.o.cast_per_token(self.xb, 128, self.fmt)
        self.o.gemm(xq, xs, self.wq, self.ws, self.fmt, out="bf16")
        return time.perf_counter() - t0

    def run(self, target_s: float):
        """Repeat the sample for about target_s seconds; returns (TFLOP/s, s, rows)."""
        t = self.once()
        reps, total = 1, t
        while total < target_s and reps < 256:
            total += self.once()
            reps += 1
        rows = self.rows * reps
        return 2.0 * rows * self.n * self.k / total / 1e12, total, rows


def cpu_baselines():
    """The CPU oracle timed in full on the smaller configurations, on this
    host's cores (OpenMP, all cores unless stated):

    - tiny forward, LHS [128, 512], RHS [256, 512], fp32 scales: both casts and
      the GEMM;
    - forward GEMMs X [M, 7168] x W [4096, 7168]^T at M = 64, 128, 4096
      (operands cast before timing);
    - the Linear step X [4096, 7168], dY [4096, 4096], W [4096, 7168]: the
      three GEMMs (fwd, dgrad against W^T's block cast, fp32 wgrad with
      K = tokens), operands cast before timing;
    - the per-token cast, hidden 4096, group 32, packed UE8M0 (the pages'
      cast point) at 1 ... 16384 tokens (16384 timed on 4096 rows and scaled),
      single-threaded and on all cores."""
    import oracle
    from quantised_linear_layers_gb300 import synthetic as syn

    oracle.build()
    o = oracle
    cores = o.num_threads()
    out = {"cores": cores, "kind": "oracle"}

    def timed(f):
        t0 = time.perf_counter()
        r = f()
        return time.perf_counter() - t0, r

    # tiny forward, fp32 scales
    x = _bits(syn.randn((128, 512), seed=syn.SEED_X))
    w = _bits(syn.randn((256, 512), seed=syn.SEED_W))

    def tiny():
        xq, xs = o.cast_per_token(x, 128, o.SF_FP32)
        wq, ws = o.cast_per_block(w, o.SF_FP32)
        return o.gemm(xq, xs, wq, ws, o.SF_FP32, out="bf16")

    t, _ = timed(tiny)
    out["tiny_fwd_128x256x512_fp32"] = {"s": round(t, 4), "tflops": round(2 * 128 * 256 * 512 / t / 1e12, 6)}

    # forward GEMMs, hidden 7168
    wf = _bits(syn.randn((4096, 7168), seed=syn.SEED_W, mul=0.02))
    wq, ws = o.cast_per_block(wf, o.SF_UE8M0)
    rows = []
    for m in (64, 128, 4096):
        xq, xs = o.cast_per_token(_bits(syn.randn((m, 7168), seed=syn.SEED_X)), 128, o.SF_UE8M0)
        t, _ = timed(lambda: o.gemm(xq, xs, wq, ws, o.SF_UE8M0, out="bf16"))
        rows.append({"m": m, "s": round(t, 3), "tflops": round(2 * m * 4096 * 7168 / t / 1e12, 4)})
    out["gemm_fwd_n4096_k7168"] = rows

    # the Linear step's three GEMMs
    xl = syn.randn((4096, 7168), seed=syn.SEED_X)
    dy = syn.randn((4096, 4096), seed=syn.SEED_DY)
    xq, xs = o.cast_per_token(_bits(xl), 128, o.SF_UE8M0)
    dq, ds = o.cast_per_token(_bits(dy), 128, o.SF_UE8M0)
    wtq, wts = o.cast_per_block(np_t(wf), o.SF_UE8M0)
    dtq, dts = o.cast_per_token(np_t(_bits(dy)), 128, o.SF_UE8M0)
    xtq, xts = o.cast_per_token(np_t(_bits(xl)), 128, o.SF_UE8M0)
    t_f, _ = timed(lambda: o.gemm(xq, xs, wq, ws, o.SF_UE8M0, out="bf16"))
    t_d, _ = timed(lambda: o.gemm(dq, ds, wtq, wts, o.SF_UE8M0, out="bf16"))
    t_w, _ = timed(lambda: o.gemm(dtq, dts, xtq, xts, o.SF_UE8M0, b_per_row=True, out="f32"))
    fl = 2 * 4096 * 4096 * 7168
    out["linear_step_4096x4096x7168"] = {"s_fwd": round(t_f, 2), "s_dgrad": round(t_d, 2), "s_wgrad": round(t_w, 2),
                                         "tflops": round(3 * fl / (t_f + t_d + t_w) / 1e12, 4)}

    # the per-token cast at the pages' point, single-threaded and all cores
    rows = []
    for tok in (1, 64, 512, 4096, 16384):
        r = min(tok, 4096)
        xc = _bits(syn.randn_row_exp(r, 4096))
        byts = r * 4096 * 3 + r * 32 * 4
        ent = {"tokens": tok, "rows_timed": r}
        for th, key in ((1, "single"), (cores, "all")):
            o.set_num_threads(th)
            t, _ = timed(lambda: o.cast_per_token(xc, 32, o.SF_PACKED_UE8M0))
            ent[f"us_{key}"] = round(t * 1e6 * tok / r, 1)
            ent[f"gbs_{key}"] = round(byts / t / 1e9, 3)
        o.set_num_threads(cores)
        rows.append(ent)
    out["cast_h4096_g32_packed"] = rows
    return out


def np_t(a):
    """Transposed numpy view (the oracle reads strided inputs)."""
    return a.T


# ------------------------------------------------------------------ our arm
def run_ours(args, world, rank, local):
    import torch

    from quantised_linear_layers_gb300 import build as qbuild
    qbuild.build()
    from quantised_linear_layers_gb300 import ops
    from quantised_linear_layers_gb300 import synthetic as syn

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    ops.load_library()
    m, n, k = args.m, args.n, args.k
    fmt = {"fp32": ops.SF_FP32, "ue8m0": ops.SF_UE8M0, "packed": ops.SF_PACKED_UE8M0}[args.fmt]
    pk = peaks()
    fp8_peak = 2.0 * pk["bf16"]
    fp8_peak_sus = 2.0 * pk["bf16_sus"] if pk["bf16_sus"] else None

    if args.only_workloads:
        wl, _ = run_workloads(dev, pk, args.reps)
        if rank == 0:
            print(json.dumps({"workloads": wl}), flush=True)
        return

    x = syn.randn((m, k), seed=syn.SEED_X + 1000 * rank, device=str(dev))
    w = syn.randn((n, k), seed=syn.SEED_W, mul=0.02, device=str(dev))
    wq, ws = ops.fp8_cast_per_block(w, fmt)
    del w
    xq = torch.empty((m, k), dtype=torch.float8_e4m3fn, device=dev)
    xs = ops.empty_sf(m, ops.sf_shape(k, 128, fmt), fmt, dev, mn_major=True)
    d = torch.empty((m, n), dtype=torch.bfloat16, device=dev)

    def step():
        ops.fp8_cast_per_token(x, 128, fmt, out=xq, out_sf=xs)
        ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, fmt, out=d)

    t0 = time.perf_counter()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    warm_s = (time.perf_counter() - t0) / max(args.warmup, 3)
    assert ops.device_status() == 0

    # The K steps are timed as a block; the block is repeated R times so that
    # the timed region lasts at least --min-timed-s under the clock sampler.
    K = args.steps
    R = max(1, int(-(-args.min_timed_s // max(warm_s * K, 1e-6))))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K * R)]
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_host0 = time.perf_counter()
    for i in range(K * R):
        ev[i][0].record()
        ops.fp8_cast_per_token(x, 128, fmt, out=xq, out_sf=xs)
        ev[i][1].record()
        ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, fmt, out=d)
        ev[i][2].record()
    torch.cuda.synchronize()
    t_host1 = time.perf_counter()
    barrier(world)
    clocks = sampler.stop(window=(t_host0, t_host1))
    if clocks is not None:
        clocks["window_ms"] = round((t_host1 - t_host0) * 1e3, 1)
    steps_timed = K * R
    total_ms = ev[0][0].elapsed_time(ev[steps_timed - 1][2])
    cast_ts = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps_timed)]
    gemm_ts = [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps_timed)]
    cast_ms = sum(cast_ts) / steps_timed
    gemm_ms = sum(gemm_ts) / steps_timed
    assert ops.device_status() == 0
    total_ms = max_over_ranks(world, total_ms)
    ms_step = total_ms / steps_timed
    flops_step = 2.0 * m * n * k
    value = flops_step * world * steps_timed / (total_ms / 1e3) / 1e12

    sf_bytes = m * ops.sf_shape(k, 128, fmt) * 4
    cast_bytes = m * k * 2 + m * k + sf_bytes
    gemm_tflops = flops_step / (gemm_ms / 1e3) / 1e12
    cast_gbs = cast_bytes / (cast_ms / 1e3) / 1e9
    del xq, xs, d

    sweep = None
    if not args.no_sweep:
        sweep = run_cast_sweep(dev, pk, args.reps)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        # end to end through the library's host-buffer call: X from pinned host
        # memory in, D to pinned host memory out, every step; the copies of one
        # row chunk overlap the kernels of the next (ql_cast_gemm_host)
        xh = torch.empty((m, k), dtype=torch.bfloat16, pin_memory=True)
        xh.copy_(x.cpu())
        dh = torch.empty((m, n), dtype=torch.bfloat16, pin_memory=True)
        ke = min(K, 5)
        chunk = args.e2e_chunk
        wsp = torch.empty(ops.cast_gemm_host_workspace_size(n, k, chunk, fmt), dtype=torch.uint8, device=dev)

        def e2e_step():
            ops.cast_gemm_host(xh, wq, ws, fmt, dh, chunk, wsp)

        e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(ke):
            e2e_step()
        torch.cuda.synchronize()
        te = max_over_ranks(world, time.perf_counter() - t0)
        e2e = {"value": round(flops_step * world * ke / te / 1e12, 2), "unit": UNIT,
               "h2d_bytes_per_step": m * k * 2, "d2h_bytes_per_step": m * n * 2, "steps": ke,
               "call": "ql_cast_gemm_host", "chunk_rows": chunk,
               "ms_per_step": round(te / ke * 1e3, 3)}
        del wsp, xh, dh
    del x, wq, ws

    workloads = None
    if not args.no_workloads:
        workloads, _ = run_workloads(dev, pk, args.reps)

    cpu, cpu_more = None, None
    if rank == 0 and world == 1 and not args.no_cpu:
        sample = CpuOracleSample(n, k, fmt)
        v, secs, rows = sample.run(args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": sample.threads, "kind": "oracle",
               "sample": f"{rows} rows of X: per-token cast + fp64 GEMM against all {n} rows of W "
                         f"(k={k}), {secs:.1f} s; W's block cast done before timing"}
        del sample
        cpu_more = cpu_baselines()

    pair = fmt != ops.SF_FP32 and ((m + 255) // 256) * ((n + 223) // 224) >= ops.get_num_sms() // 2
    kernel = "gemm_mx2_kernel" if pair else ("gemm_mx_kernel" if fmt != ops.SF_FP32 else "gemm_fp8_kernel")
    traffic, traffic_workload = recorded_traffic(kernel)
    if traffic_workload is not None and traffic_workload != [m, n, k]:
        traffic = None
    counters = recorded_counters(kernel)
    tensor_pipe = None
    if counters is not None and counters.get("workload") == [m, n, k] and "tensor_pipe_active_pct_of_elapsed" in counters:
        tensor_pipe = {"active_pct_of_elapsed": counters["tensor_pipe_active_pct_of_elapsed"],
                       "sm_clock_hz_under_ncu": counters.get("sm_clock_hz_under_ncu"),
                       "source": "profiles/gemm_traffic.json (one ncu capture of this launch)"}
    sm_mhz = clocks["sm_mhz"] if clocks else None
    nominal_per_clk = 16384.0 * ops.get_num_sms()     # dense FP8 flop per SM clock x SMs
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic (seeded randn; W randn*0.02)",
            "timed_region": {"repeats_of_k_steps": R, "steps_timed": steps_timed,
                             "ms": round(total_ms, 2), "why": f"timed region >= {args.min_timed_s} s under the clock sampler"},
            "config": {"workload": WORKLOAD, "m": m, "n": n, "k": k, "x_dtype": "bf16", "out_dtype": "bf16",
                       "gran_k": 128, "scales": args.fmt, "l2": "inputs larger than L2 (no flush)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": round(gemm_tflops, 1),
                         "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                         "frac": round(gemm_tflops / fp8_peak, 4), "traffic": traffic,
                         "kernel": kernel, "peak_note": f"dense FP8 = 2 x {pk['source']} bf16 burst",
                         "frac_of_sustained": round(gemm_tflops / fp8_peak_sus, 4) if fp8_peak_sus else None,
                         "gemm_ms": {"p10": round(sorted(gemm_ts)[len(gemm_ts) // 10], 4),
                                     "median": round(statistics.median(gemm_ts), 4),
                                     "p90": round(sorted(gemm_ts)[(9 * len(gemm_ts)) // 10], 4)},
                         "clock_normalised": (
                             {"sm_mhz": sm_mhz,
                              "peak_at_clock_tflops": round(nominal_per_clk * sm_mhz * 1e6 / 1e12, 1),
                              "frac": round(gemm_tflops * 1e12 / (nominal_per_clk * sm_mhz * 1e6), 4),
                              "note": "achieved / (16384 dense FP8 flop per SM clock x SMs x median SM clock "
                                      "in the timed region)"} if sm_mhz else None),
                         "tensor_pipe": tensor_pipe},
            "gemm": {"ms": round(gemm_ms, 4), "tflops": round(gemm_tflops, 1)},
            "cast": {"ms": round(cast_ms, 4), "bytes": cast_bytes, "gbs": round(cast_gbs, 1),
                     "frac_hbm": round(cast_gbs / pk["hbm_gbs"], 4), "peak_gbs": pk["hbm_gbs"],
                     "us": stats_us(cast_ts)},
            "cast_sweep": sweep,
            "workloads": workloads,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "cpu_baselines": cpu_more,
            "clocks": clocks,
            "gpu_launches": 2 * steps_timed,
        }
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ cast sweep
def run_cast_sweep(dev, pk, reps):
    """The per-token cast sweep of the pages' results table: hidden 4096,
    tokens 1 / 64 / 512 / 4096 / 16384, group 32 and 128, fp32 / UE8M0 /
    packed-UE8M0 scales, bf16 and fp32 input (randn x 10^U(-3,3) per row).
    Each point: eager with L2 flushed before each repetition, and per cast
    inside a CUDA graph of back-to-back casts (L2 flushed before each replay),
    as GB/s of algorithmic bytes and as a fraction of measured HBM bandwidth.
    Plus one hot-L2 point: 4096 tokens, group 32, packed (input and output,
    50.9 MB, stay resident in the 129 MB L2 between repetitions)."""
    import torch

    from quantised_linear_layers_gb300 import ops
    from quantised_linear_layers_gb300 import synthetic as syn

    flush = L2Flush(dev)
    points = []
    for dt in (torch.bfloat16, torch.float32):
        for tok in (1, 64, 512, 4096, 16384):
            xin = syn.randn_row_exp(tok, 4096, dtype=dt, device=str(dev))
            for gran in (32, 128):
                for fmt in (ops.SF_FP32, ops.SF_UE8M0, ops.SF_PACKED_UE8M0):
                    q = torch.empty((tok, 4096), dtype=torch.float8_e4m3fn, device=dev)
                    sf = ops.empty_sf(tok, ops.sf_shape(4096, gran, fmt), fmt, dev)
                    f = lambda: ops.fp8_cast_per_token(xin, gran, fmt, out=q, out_sf=sf)
                    byts = tok * 4096 * (xin.element_size() + 1) + sf.numel() * 4
                    te = stats_us(time_eager(f, reps, flush))
                    per = 20 if tok <= 512 else 4
                    tg = stats_us(time_graph(f, max(10, reps // 4), flush, per=per))
                    points.append({
                        "tokens": tok, "x": "bf16" if dt == torch.bfloat16 else "f32", "gran": gran,
                        "scales": ("fp32", "ue8m0", "packed")[fmt], "bytes": byts,
                        "eager_cold_l2": te, "gbs": round(byts / te["us"] / 1e3, 1),
                        "frac_hbm": round(byts / te["us"] / 1e3 / pk["hbm_gbs"], 3),
                        "graph_per_cast": tg, "graph_casts": per})
            del xin
    # hot L2
    xin = syn.randn_row_exp(4096, 4096, device=str(dev))
    q = torch.empty((4096, 4096), dtype=torch.float8_e4m3fn, device=dev)
    sf = ops.empty_sf(4096, ops.sf_shape(4096, 32, 2), 2, dev)
    hot = stats_us(time_eager(lambda: ops.fp8_cast_per_token(xin, 32, 2, out=q, out_sf=sf), reps))
    byts = 4096 * 4096 * 3 + 4096 * 32 * 4
    return {"hidden": 4096, "l2": "flushed before each repetition (256 MB write, then 256 MB read)", "points": points,
            "hot_l2_4096_tokens_g32_packed": {"what": "input and output (50.9 MB) resident in L2", **hot,
                                               "gbs": round(byts / hot["us"] / 1e3, 1)},
            "pages_b200_us": {"1": [6.4, 1.2], "64": [6.3, 1.5], "512": [8.2, 2.0], "4096": [15.5, 6.3],
                              "16384": [38.7, 31.4], "note": "[Triton eager, Triton in a CUDA graph], "
                                                             "bf16, group 32, packed, on B200"}}


# ------------------------------------------------------------------ other workloads
def run_workloads(dev, pk, reps):
    """The smaller workloads of the method's pages, each timed with CUDA events
    (median, p10, p90 of `reps`, the L2 flushed before each repetition unless
    stated), eagerly and replayed from a CUDA graph:

    - tiny forward (LHS [128, 512], RHS [256, 512], fp32 scales): per-token
      cast, block cast and GEMM;
    - forward GEMM N=4096, K=7168 at M = 64, 128 (HBM-bound: W's bytes
      dominate) and 4096 (tensor-bound), with packed UE8M0 and with fp32
      scales, and at M = 64, 128 as 32 GEMMs back to back over 8 distinct
      weights;
    - the Linear layer's step, X [4096, 7168], dY [4096, 4096], W [4096, 7168]
      with packed UE8M0 and with fp32 scales: weight cast (W's 128x128 block
      cast, which also writes W^T's scale grid), forward (X cast along
      features and tokens in one pass + GEMM), backward (dY cast both ways in
      one pass + dgrad GEMM reading W's cast MN-major + fp32 wgrad GEMM on the
      token-axis casts); and its weight gradient with the operands cast from
      transposed views against cast in place and read MN-major;
    - the low-latency per-token cast (hidden 4096, group 32, packed UE8M0) at
      1, 64 and 512 tokens per cast inside a captured CUDA graph of 50 casts;
    - a GEMM whose output feeds the next FP8 layer: bf16 output plus the
      per-token cast, against the cast fused into the GEMM's epilogue;
    - the M-grouped contiguous GEMM of a mixture-of-experts layer: 8 experts
      of about 2048 tokens each, N=4096, K=7168.
    Returns (dict, number of this library's kernel launches timed).
    """
    import torch

    from quantised_linear_layers_gb300 import linear, ops
    from quantised_linear_layers_gb300 import synthetic as syn

    P, F = ops.SF_PACKED_UE8M0, ops.SF_FP32
    flush = L2Flush(dev)
    out, launches = {}, 0

    # tiny forward with fp32 scales
    xt = syn.randn((128, 512), seed=syn.SEED_X, device=str(dev))
    wt = syn.randn((256, 512), seed=syn.SEED_W, device=str(dev))
    txq = torch.empty((128, 512), dtype=torch.float8_e4m3fn, device=dev)
    txs = ops.empty_sf(128, 4, F, dev, mn_major=True)
    twq = torch.empty((256, 512), dtype=torch.float8_e4m3fn, device=dev)
    tws = torch.empty((2, 4), dtype=torch.float32, device=dev)
    td = torch.empty((128, 256), dtype=torch.bfloat16, device=dev)

    def tiny():
        ops.fp8_cast_per_token(xt, 128, F, out=txq, out_sf=txs)
        ops.fp8_cast_per_block(wt, F, out=twq, out_sf=tws)
        ops.gemm_fp8_nt_bf16(txq, txs, twq, tws, F, out=td)

    r = eager_and_graph(tiny, reps, flush)
    r["gemm_alone"] = eager_and_graph(lambda: ops.gemm_fp8_nt_bf16(txq, txs, twq, tws, F, out=td), reps, flush)
    r["flop"] = 2 * 128 * 256 * 512
    out["tiny_fwd_128x256x512_fp32"] = r
    launches += 2 * reps * 5

    w = syn.randn((4096, 7168), seed=syn.SEED_W, mul=0.02, device=str(dev))
    rows = []
    for fmt in (P, F):
        wq, ws = ops.fp8_cast_per_block(w, fmt)
        for m in (64, 128, 4096):
            x = syn.randn((m, 7168), seed=syn.SEED_X, device=str(dev))
            xq, xs = ops.fp8_cast_per_token(x, 128, fmt, sf_mn_major=True)
            d = torch.empty((m, 4096), dtype=torch.bfloat16, device=dev)
            r = eager_and_graph(lambda: ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, fmt, out=d), reps, flush)
            launches += 2 * reps
            sfb = 4 * (m + 4096 // 128) * ((7168 // 512) if fmt == P else (7168 // 128))
            byts = m * 7168 + 4096 * 7168 + m * 4096 * 2 + sfb
            fl = 2 * m * 4096 * 7168
            us = r["eager_cold_l2"]["us"]
            rows.append({"m": m, "n": 4096, "k": 7168, "scales": ("fp32", "ue8m0", "packed")[fmt], **r,
                         "tflops": round(fl / us / 1e6, 1), "gbs": round(byts / us / 1e3, 1),
                         "frac_hbm": round(byts / us / 1e3 / pk["hbm_gbs"], 3)})
        del wq, ws
    out["gemm_fwd_n4096_k7168_cold_l2"] = rows

    x = syn.randn((4096, 7168), seed=syn.SEED_X, device=str(dev))
    dy = syn.randn((4096, 4096), seed=syn.SEED_DY, device=str(dev))
    fl = 2 * 4096 * 4096 * 7168
    for fmt, key in ((P, "linear_step_4096x4096x7168_cold_l2"), (F, "linear_step_4096x4096x7168_fp32_cold_l2")):
        w8 = linear.FP8Weight(w, fmt)
        torch.cuda.synchronize()
        ev = []
        for i in range(10 + reps):
            flush()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record()
            w8.update(w)
            e[1].record()
            _, xc = linear.forward_saving(x, w8)
            e[2].record()
            linear.backward(dy, w8, xc)
            e[3].record()
            if i >= 10:
                ev.append(e)
                launches += 6
        torch.cuda.synchronize()
        part = [stats_us([e[j].elapsed_time(e[j + 1]) for e in ev]) for j in range(3)]
        step = stats_us([e[0].elapsed_time(e[3]) for e in ev])
        out[key] = {
            "weight_casts": part[0], "fwd": part[1], "bwd": part[2], "step": step,
            "tflops_step": round(3 * fl / step["us"] / 1e6, 1),
            "tflops_without_weight_casts": round(3 * fl / (step["us"] - part[0]["us"]) / 1e6, 1)}
        del w8
    # the step's casts alone, as GB/s of their algorithmic bytes: W's dual
    # block cast, X's and dY's dual per-token casts (one read, two E4M3 casts)
    casts = {}

    def _packed_words(rows, groups):
        return rows * ((groups + 3) // 4) * 4

    for name, f, byts in (
            ("w_block_dual_4096x7168", lambda: ops.fp8_cast_per_block_dual(w, P),
             4096 * 7168 * 3 + _packed_words(32, 56) + _packed_words(56, 32)),
            ("x_dual_4096x7168", lambda: ops.fp8_cast_per_token_dual(x, P),
             4096 * 7168 * 4 + _packed_words(4096, 56) + _packed_words(7168, 32)),
            ("dy_dual_4096x4096", lambda: ops.fp8_cast_per_token_dual(dy, P),
             4096 * 4096 * 4 + _packed_words(4096, 32) + _packed_words(4096, 32))):
        r = stats_us(time_eager(f, reps, flush))
        casts[name] = {**r, "bytes": byts, "gbs": round(byts / r["us"] / 1e3, 1),
                       "frac_hbm": round(byts / r["us"] / 1e3 / pk["hbm_gbs"], 3)}
        launches += reps
    out["linear_step_casts_cold_l2"] = casts
    # the weight gradient with transposed casts against MN-major operands
    t_tr = stats_us(time_eager(lambda: linear.wgrad(dy, x, P, mn_major=False), reps, flush))
    t_mn = stats_us(time_eager(lambda: linear.wgrad(dy, x, P, mn_major=True), reps, flush))
    launches += 6 * reps
    out["wgrad_transposed_vs_mn_major_4096x7168x4096"] = {"transposed_casts": t_tr, "mn_major": t_mn}
    del x, dy, w

    # GEMM whose output feeds the next FP8 layer: bf16 output then the
    # per-token cast, against the cast fused into the GEMM's epilogue
    # (Y = X W^T with X [4096, 4096], W [7168, 4096]; 1x128 packed output)
    xa = syn.randn((4096, 4096), seed=syn.SEED_X, device=str(dev))
    xaq, xas = ops.fp8_cast_per_token(xa, 128, P, sf_mn_major=True)
    wb = syn.randn((7168, 4096), seed=syn.SEED_W, mul=0.02, device=str(dev))
    wbq, wbs = ops.fp8_cast_per_block(wb, P)
    del xa, wb
    y = torch.empty((4096, 7168), dtype=torch.bfloat16, device=dev)
    yq = torch.empty((4096, 7168), dtype=torch.float8_e4m3fn, device=dev)
    ys = ops.empty_sf(4096, ops.sf_shape(7168, 128, P), P, dev, mn_major=True)

    def unfused():
        ops.gemm_fp8_nt_bf16(xaq, xas, wbq, wbs, P, out=y)
        ops.fp8_cast_per_token(y, 128, P, out=yq, out_sf=ys)

    def fused():
        ops.gemm_fp8_nt_fp8out(xaq, xas, wbq, wbs, P, 128, P, out=yq, out_sf=ys)

    t_un = stats_us(time_eager(unfused, reps, flush))
    t_fu = stats_us(time_eager(fused, reps, flush))
    launches += 3 * reps
    fl = 2 * 4096 * 7168 * 4096
    out["gemm_cast_fused_4096x7168x4096_cold_l2"] = {
        "gemm_bf16_then_cast": t_un, "fused": t_fu,
        "tflops_unfused": round(fl / t_un["us"] / 1e6, 1), "tflops_fused": round(fl / t_fu["us"] / 1e6, 1),
        "hbm_bytes_saved": 4096 * 7168 * 2 * 2}
    del xaq, xas, wbq, wbs, y, yq, ys

    rows = []
    G = 50
    for t in (1, 64, 512):
        xt = syn.randn_row_exp(t, 4096, device=str(dev))
        q = torch.empty((t, 4096), dtype=torch.float8_e4m3fn, device=dev)
        sf = ops.empty_sf(t, ops.sf_shape(4096, 32, P), P, dev)
        f = lambda: ops.fp8_cast_per_token(xt, 32, P, out=q, out_sf=sf)
        per = stats_us(time_graph(f, reps, None, per=G))
        launches += reps * G
        rows.append({"tokens": t, "bytes": t * 4096 * 3 + t * 32 * 4, "per_cast_in_graph_of_50": per})
    out["cast_low_latency_h4096_g32_packed"] = rows

    # M-grouped contiguous GEMM (mixture of experts): 8 experts of about 2048
    # tokens each (uneven), N = 4096, K = 7168, packed UE8M0 scales
    tokens = syn.tokens_per_expert(8, 2048, seed=17)
    idx, _ = syn.contiguous_layout(tokens, 128)
    mg = idx.numel()
    xg = syn.randn((mg, 7168), seed=syn.SEED_X, device=str(dev))
    xgq, xgs = ops.fp8_cast_per_token(xg, 128, P, sf_mn_major=True)
    del xg
    wg = torch.empty((8, 4096, 7168), dtype=torch.float8_e4m3fn, device=dev)
    wgs = torch.empty((8, 32, 14), dtype=torch.int32, device=dev)
    for e in range(8):
        we = syn.randn((4096, 7168), seed=100 + e, mul=0.02, device=str(dev))
        ops.fp8_cast_per_block(we, P, out=wg[e], out_sf=wgs[e])
    del we
    idx = idx.to(dev)
    dg = torch.empty((mg, 4096), dtype=torch.bfloat16, device=dev)
    r = stats_us(time_eager(lambda: ops.m_grouped_gemm_fp8_nt_bf16_contiguous(xgq, xgs, wg, wgs, idx, P, out=dg),
                            reps, flush))
    launches += reps
    fl = 2 * sum(tokens) * 4096 * 7168
    out["grouped_gemm_8experts_n4096_k7168_cold_l2"] = {
        "tokens": tokens, "m_aligned": mg, **r, "tflops_valid_rows": round(fl / r["us"] / 1e6, 1),
        "tflops_incl_padding": round(2 * mg * 4096 * 7168 / r["us"] / 1e6, 1)}
    del xgq, xgs, wg, wgs, dg

    # small M back to back, as in decoding: 32 GEMMs in a row over 8 distinct
    # weights (8 x 29.4 MB > L2), one event pair around the sequence; eager
    # launches and the sequence replayed from a CUDA graph
    wcopies = [ops.fp8_cast_per_block(syn.randn((4096, 7168), seed=200 + i, mul=0.02, device=str(dev)), P)
               for i in range(8)]
    rows = []
    for m in (64, 128):
        x = syn.randn((m, 7168), seed=syn.SEED_X, device=str(dev))
        xq, xs = ops.fp8_cast_per_token(x, 128, P, sf_mn_major=True)
        d = torch.empty((m, 4096), dtype=torch.bfloat16, device=dev)

        def seq():
            for _ in range(4):
                for wq_i, ws_i in wcopies:
                    ops.gemm_fp8_nt_bf16(xq, xs, wq_i, ws_i, P, out=d)

        n_rep = max(10, reps // 4)
        te = stats_us([t / 32 for t in time_eager(seq, n_rep)])
        tg = stats_us([t / 32 for t in time_eager(capture(seq, 1).replay, n_rep)])
        launches += 64 * n_rep
        byts = m * 7168 + 4096 * 7168 + m * 4096 * 2 + 4 * (m + 4096 // 128) * (7168 // 512)
        rows.append({"m": m, "eager_per_gemm": te, "graph_per_gemm": tg,
                     "gbs": round(byts / te["us"] / 1e3, 1), "frac_hbm": round(byts / te["us"] / 1e3 / pk["hbm_gbs"], 3),
                     "frac_hbm_graph": round(byts / tg["us"] / 1e3 / pk["hbm_gbs"], 3)})
    out["gemm_fwd_small_m_back_to_back_8_weights"] = rows
    del wcopies
    assert ops.device_status() == 0
    return out, launches


# ------------------------------------------------------------------ reference arm
def run_reference(args, world, rank):
    """The CPU oracle timed on the host cores, on a bounded sample per step:
    each step casts a slice of X's rows and multiplies it (fp64) against all of
    W. `ms_per_step` is that sampled step's measured time."""
    if rank != 0:
        return
    m, n, k = args.m, args.n, args.k
    fmt_code = {"fp32": 0, "ue8m0": 1, "packed": 2}[args.fmt]
    per_step = max(1.0, min(5.0, 120.0 / max(1, args.steps + args.warmup)))
    sample = CpuOracleSample(n, k, fmt_code)
    threads = sample.threads
    for _ in range(args.warmup):
        sample.once()
    vals, secs, rows_total = [], 0.0, 0
    for _ in range(args.steps):
        v, s, rows = sample.run(per_step)
        vals.append(v)
        secs += s
        rows_total += rows
    value = statistics.median(vals)
    ms_full = 2.0 * m * n * k / (value * 1e12) * 1e3 if value > 0 else None
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / max(1, args.steps) * 1e3, 1),
        "ms_per_step_note": "one sampled step (a slice of X's rows against all of W), measured",
        "ms_full_workload_extrapolated": ms_full,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded randn; W randn*0.02)",
        "config": {"workload": WORKLOAD, "m": m, "n": n, "k": k, "gran_k": 128, "scales": args.fmt},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"per step: a slice of X's rows cast + fp64 GEMM against all {n} rows of W; "
                                   f"{rows_total} rows over {secs:.1f} s"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
