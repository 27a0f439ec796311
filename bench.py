"""Benchmark of the FP8 linear-layer hot path on GB300.

One step = the per-token FP8 cast of X (1x128 groups, UE8M0 scales packed
four exponents per int32 word, written M-major) followed by the block-scaled
GEMM D = X W^T (bf16 out), over the
large cast+GEMM workload: X bf16 [16384, 7168] randn, W bf16 [18432, 7168]
randn * 0.02 cast once to E4M3 with 128x128 UE8M0 block scales (outside the
timed region, as a weight cast runs once per weight update). Inputs are
synthetic and seeded; they are larger than L2, so no flush is needed.

Prints one JSON line (rank 0). Keys: metric/value/unit (GEMM TFLOP/s of the
whole step), ms_per_step, roofline (dominant kernel: the GEMM, against the
dense FP8 peak = 2x the measured bf16 peak), cast (GB/s of the cast kernel
against measured HBM bandwidth), cast_sweep (the pages' per-token cast
point: 16384 tokens x 4096, group 32, packed UE8M0), workloads (the smaller
workloads, timed apart from the step: forward GEMMs at M = 64/128/4096, the
Linear layer's fwd+dgrad+wgrad step, the low-latency cast at 1-512 tokens
eager and inside a CUDA graph), e2e (host buffers,
copies inside the timed region), cpu_baseline (the CPU oracle on a bounded
sample), clocks (nvidia-smi during the timed region), gpu_launches. e2e runs
the library's host-buffer call, which overlaps the copies of one row chunk
with the kernels of the next.

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
    ap.add_argument("--reps", type=int, default=20, help="timed repetitions per other workload")
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
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

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
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
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


def recorded_traffic(kernel_file: str):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu record,
    or None when the kernel source changed since the counters were taken."""
    import hashlib
    rec = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(rec):
        return None, None
    with open(rec) as fh:
        data = json.load(fh)
    h = hashlib.sha256()
    for f in data.get("sources", []):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    entry = data.get("kernels", {}).get(kernel_file)
    if not entry or data.get("sources_sha256") != h.hexdigest():
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


# ------------------------------------------------------------------ CPU oracle
class CpuOracleSample:
    """The CPU oracle on a bounded sample of the workload: the per-token cast
    of a slice of X's rows and the fp64 GEMM of those rows against all of W.
    W's block cast (once per weight update) is prepared before any timing,
    as on the GPU."""

    def __init__(self, n, k, fmt_code):
        import numpy as np
        import torch

        import oracle
        from quantised_linear_layers_gb300 import synthetic as syn

        oracle.build()
        self.o = oracle
        self.n, self.k = n, k
        self.fmt = oracle.SF_FP32 if fmt_code == 0 else oracle.SF_UE8M0
        self.threads = oracle.num_threads()
        w = syn.randn((n, k), seed=syn.SEED_W, mul=0.02)
        self.wq, self.ws = oracle.cast_per_block(w.view(torch.int16).numpy().view(np.uint16), self.fmt)
        self.rows = max(self.threads, 8)
        x = syn.randn((self.rows, k), seed=syn.SEED_X)
        self.xb = x.view(torch.int16).numpy().view(np.uint16)

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

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert ops.device_status() == 0

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.5)
    for i in range(K):
        ev[i][0].record()
        ops.fp8_cast_per_token(x, 128, fmt, out=xq, out_sf=xs)
        ev[i][1].record()
        ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, fmt, out=d)
        ev[i][2].record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    total_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    cast_ms = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(K)) / K
    gemm_ms = sum(ev[i][1].elapsed_time(ev[i][2]) for i in range(K)) / K
    assert ops.device_status() == 0
    total_ms = max_over_ranks(world, total_ms)
    ms_step = total_ms / K
    flops_step = 2.0 * m * n * k
    value = flops_step * world * K / (total_ms / 1e3) / 1e12

    sf_bytes = m * ops.sf_shape(k, 128, fmt) * 4
    cast_bytes = m * k * 2 + m * k + sf_bytes
    gemm_tflops = flops_step / (gemm_ms / 1e3) / 1e12
    cast_gbs = cast_bytes / (cast_ms / 1e3) / 1e9

    # the pages' per-token cast point: 16384 x 4096 bf16, group 32, packed UE8M0
    sweep = None
    if not args.no_sweep:
        xs_in = syn.randn_row_exp(16384, 4096, device=str(dev))
        sq = torch.empty((16384, 4096), dtype=torch.float8_e4m3fn, device=dev)
        ssf = ops.empty_sf(16384, ops.sf_shape(4096, 32, 2), 2, dev)
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        for _ in range(5):
            ops.fp8_cast_per_token(xs_in, 32, 2, out=sq, out_sf=ssf)
        times_cold, times_hot = [], []
        for _ in range(20):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            ops.fp8_cast_per_token(xs_in, 32, 2, out=sq, out_sf=ssf)
            b.record()
            torch.cuda.synchronize()
            times_cold.append(a.elapsed_time(b))
        for _ in range(20):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            ops.fp8_cast_per_token(xs_in, 32, 2, out=sq, out_sf=ssf)
            b.record()
            torch.cuda.synchronize()
            times_hot.append(a.elapsed_time(b))
        sb = 16384 * 4096 * 2 + 16384 * 4096 + 16384 * 32 * 4
        tc = statistics.median(times_cold)
        th = statistics.median(times_hot)
        sweep = {"shape": [16384, 4096], "gran": 32, "scales": "packed_ue8m0", "bytes": sb,
                 "us_cold_l2": round(tc * 1e3, 2), "gbs_cold_l2": round(sb / (tc / 1e3) / 1e9, 1),
                 "frac_hbm_cold": round(sb / (tc / 1e3) / 1e9 / pk["hbm_gbs"], 3),
                 "us_hot_l2": round(th * 1e3, 2), "pages_b200_eager_us": 38.7}
        del xs_in, sq, ssf, flush

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
        del wsp

    workloads = None
    if not args.no_workloads:
        del x, xq, xs, d
        workloads, _ = run_workloads(dev, pk, args.reps)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        sample = CpuOracleSample(n, k, fmt)
        v, secs, rows = sample.run(args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": sample.threads, "kind": "oracle",
               "sample": f"{rows} rows of X: per-token cast + fp64 GEMM against all {n} rows of W "
                         f"(k={k}), {secs:.1f} s; W's block cast done before timing"}

    pair = fmt != ops.SF_FP32 and ((m + 255) // 256) * ((n + 255) // 256) >= ops.get_num_sms() // 2
    kernel = "gemm_mx2_kernel" if pair else ("gemm_mx_kernel" if fmt != ops.SF_FP32 else "gemm_fp8_kernel")
    traffic, traffic_workload = recorded_traffic(kernel)
    if traffic_workload is not None and traffic_workload != [m, n, k]:
        traffic = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic (seeded randn; W randn*0.02)",
            "config": {"workload": WORKLOAD, "m": m, "n": n, "k": k, "x_dtype": "bf16", "out_dtype": "bf16",
                       "gran_k": 128, "scales": args.fmt, "l2": "inputs larger than L2 (no flush)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": round(gemm_tflops, 1),
                         "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                         "frac": round(gemm_tflops / fp8_peak, 4), "traffic": traffic,
                         "kernel": kernel, "peak_note": f"dense FP8 = 2 x {pk['source']} bf16 burst",
                         "frac_of_sustained": round(gemm_tflops / fp8_peak_sus, 4) if fp8_peak_sus else None},
            "gemm": {"ms": round(gemm_ms, 4), "tflops": round(gemm_tflops, 1)},
            "cast": {"ms": round(cast_ms, 4), "bytes": cast_bytes, "gbs": round(cast_gbs, 1),
                     "frac_hbm": round(cast_gbs / pk["hbm_gbs"], 4), "peak_gbs": pk["hbm_gbs"]},
            "cast_sweep": sweep,
            "workloads": workloads,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "gpu_launches": 2 * K,
        }
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ other workloads
def _median_ms(fn, reps, flush=None, warm=3):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def run_workloads(dev, pk, reps):
    """The smaller workloads of the method's pages, each timed with CUDA events
    (median of `reps`):

    - forward GEMM N=4096, K=7168 at M = 64, 128 (HBM-bound: W's bytes
      dominate) and 4096 (tensor-bound), L2 flushed before each repetition,
      and at M = 64, 128 as 32 GEMMs back to back over 8 distinct weights;
    - the Linear layer's step, X [4096, 7168], dY [4096, 4096], W [4096, 7168]:
      weight cast (W's 128x128 block cast, which also writes W^T's scale
      grid), forward (X cast along features and tokens in one pass + GEMM),
      backward (dY cast both ways in one pass + dgrad GEMM reading W's cast
      MN-major + fp32 wgrad GEMM on the token-axis casts),
      L2 flushed before each step; and its weight gradient with the operands
      cast from transposed views against cast in place and read MN-major;
    - the low-latency per-token cast (hidden 4096, group 32, packed UE8M0) at
      1, 64 and 512 tokens: eager with a flushed L2, and the device time per
      cast inside a captured CUDA graph of 50 casts;
    - a GEMM whose output feeds the next FP8 layer: bf16 output plus the
      per-token cast, against the cast fused into the GEMM's epilogue;
    - the M-grouped contiguous GEMM of a mixture-of-experts layer: 8 experts
      of about 2048 tokens each, N=4096, K=7168, L2 flushed.
    Returns (dict, number of this library's kernel launches timed).
    """
    import torch

    from quantised_linear_layers_gb300 import linear, ops
    from quantised_linear_layers_gb300 import synthetic as syn

    P = ops.SF_PACKED_UE8M0
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    out, launches = {}, 0

    w = syn.randn((4096, 7168), seed=syn.SEED_W, mul=0.02, device=str(dev))
    wq, ws = ops.fp8_cast_per_block(w, P)
    rows = []
    for m in (64, 128, 4096):
        x = syn.randn((m, 7168), seed=syn.SEED_X, device=str(dev))
        xq, xs = ops.fp8_cast_per_token(x, 128, P, sf_mn_major=True)
        d = torch.empty((m, 4096), dtype=torch.bfloat16, device=dev)
        ms = _median_ms(lambda: ops.gemm_fp8_nt_bf16(xq, xs, wq, ws, P, out=d), reps, flush)
        launches += reps
        byts = m * 7168 + 4096 * 7168 + m * 4096 * 2 + 4 * (m + 4096 // 128) * (7168 // 512)
        fl = 2 * m * 4096 * 7168
        rows.append({"m": m, "n": 4096, "k": 7168, "us": round(ms * 1e3, 2),
                     "tflops": round(fl / ms / 1e9, 1), "gbs": round(byts / ms / 1e6, 1),
                     "frac_hbm": round(byts / ms / 1e6 / pk["hbm_gbs"], 3)})
    out["gemm_fwd_n4096_k7168_cold_l2"] = rows



    x = syn.randn((4096, 7168), seed=syn.SEED_X, device=str(dev))
    dy = syn.randn((4096, 4096), seed=syn.SEED_DY, device=str(dev))
    w8 = linear.FP8Weight(w, P)
    torch.cuda.synchronize()
    ev = []
    for i in range(3 + reps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record()
        w8.update(w)
        e[1].record()
        _, xc = linear.forward_saving(x, w8)
        e[2].record()
        linear.backward(dy, w8, xc)
        e[3].record()
        if i >= 3:
            ev.append(e)
            launches += 6
    torch.cuda.synchronize()
    part = [statistics.median(e[j].elapsed_time(e[j + 1]) for e in ev) for j in range(3)]
    step = statistics.median(e[0].elapsed_time(e[3]) for e in ev)
    fl = 2 * 4096 * 4096 * 7168
    out["linear_step_4096x4096x7168_cold_l2"] = {
        "us_weight_casts": round(part[0] * 1e3, 1), "us_fwd": round(part[1] * 1e3, 1),
        "us_bwd": round(part[2] * 1e3, 1),
        "us_step": round(step * 1e3, 1), "tflops_step": round(3 * fl / step / 1e9, 1),
        "tflops_without_weight_casts": round(3 * fl / (step - part[0]) / 1e9, 1)}
    # the weight gradient with transposed casts against MN-major operands
    t_tr = _median_ms(lambda: linear.wgrad(dy, x, P, mn_major=False), reps, flush)
    t_mn = _median_ms(lambda: linear.wgrad(dy, x, P, mn_major=True), reps, flush)
    launches += 6 * reps
    out["wgrad_transposed_vs_mn_major_4096x7168x4096"] = {
        "us_transposed_casts": round(t_tr * 1e3, 1), "us_mn_major": round(t_mn * 1e3, 1)}
    del x, dy, w8, w, wq, ws

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

    t_un = _median_ms(unfused, reps, flush)
    t_fu = _median_ms(fused, reps, flush)
    launches += 3 * reps
    fl = 2 * 4096 * 7168 * 4096
    out["gemm_cast_fused_4096x7168x4096_cold_l2"] = {
        "us_gemm_bf16_then_cast": round(t_un * 1e3, 1), "us_fused": round(t_fu * 1e3, 1),
        "tflops_unfused": round(fl / t_un / 1e9, 1), "tflops_fused": round(fl / t_fu / 1e9, 1),
        "hbm_bytes_saved": 4096 * 7168 * 2 * 2}
    del xaq, xas, wbq, wbs, y, yq, ys

    rows = []
    G = 50
    for t in (1, 64, 512):
        xt = syn.randn_row_exp(t, 4096, device=str(dev))
        q = torch.empty((t, 4096), dtype=torch.float8_e4m3fn, device=dev)
        sf = ops.empty_sf(t, ops.sf_shape(4096, 32, P), P, dev)
        f = lambda: ops.fp8_cast_per_token(xt, 32, P, out=q, out_sf=sf)
        eager = _median_ms(f, reps, flush)
        launches += reps
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            f()
            s.synchronize()
            with torch.cuda.graph(g, stream=s):
                for _ in range(G):
                    f()
        torch.cuda.current_stream().wait_stream(s)
        per = _median_ms(lambda: g.replay(), reps) / G
        launches += reps * G
        byts = t * 4096 * 3 + t * 32 * 4
        rows.append({"tokens": t, "bytes": byts, "us_eager_cold_l2": round(eager * 1e3, 2),
                     "us_per_cast_in_graph": round(per * 1e3, 2)})
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
    ms = _median_ms(lambda: ops.m_grouped_gemm_fp8_nt_bf16_contiguous(xgq, xgs, wg, wgs, idx, P, out=dg),
                    reps, flush)
    launches += reps
    fl = 2 * sum(tokens) * 4096 * 7168
    out["grouped_gemm_8experts_n4096_k7168_cold_l2"] = {
        "tokens": tokens, "m_aligned": mg, "us": round(ms * 1e3, 1), "tflops_valid_rows": round(fl / ms / 1e9, 1),
        "tflops_incl_padding": round(2 * mg * 4096 * 7168 / ms / 1e9, 1)}
    del xgq, xgs, wg, wgs, dg

    # small M back to back, as in decoding: 32 GEMMs in a row over 8 distinct
    # weights (8 x 29.4 MB > L2), one event pair around the sequence
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

        ms = _median_ms(seq, max(3, reps // 4)) / 32
        launches += 32 * max(3, reps // 4)
        byts = m * 7168 + 4096 * 7168 + m * 4096 * 2 + 4 * (m + 4096 // 128) * (7168 // 512)
        rows.append({"m": m, "us_per_gemm": round(ms * 1e3, 2), "gbs": round(byts / ms / 1e6, 1),
                     "frac_hbm": round(byts / ms / 1e6 / pk["hbm_gbs"], 3)})
    out["gemm_fwd_small_m_back_to_back_8_weights"] = rows
    del wcopies
    assert ops.device_status() == 0
    return out, launches


# ------------------------------------------------------------------ reference arm
def run_reference(args, world, rank):
    """The CPU oracle timed on the host cores, on a bounded sample per step."""
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
    # one whole step of the workload at the sampled rate (the GEMM's 2mnk flop)
    ms_full = 2.0 * m * n * k / (value * 1e12) * 1e3 if value > 0 else None
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_full, "ms_per_step_note": "whole step extrapolated from the sample",
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
