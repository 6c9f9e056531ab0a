#!/usr/bin/env python3
"""Benchmark: lossless BF16 exponent codec on GB300, one JSON line on stdout.

A step is one pass of the whole hot path over one synthetic buffer: zc_compress in auto mode
(statistics pass, window base, encode + single-pass chunk scan) followed by zc_decompress, on
the 4096 x 14336 FSDP gradient-bucket workload resident in HBM.  The L2 cache is flushed
between steps, outside the timed region: a 256 MiB buffer is written and then read back, so
the cache holds none of the step's data and no dirty lines whose write-back the next kernel
would pay for.  Each step is timed with CUDA events on the stream the library launches on.
A second pass of the same K steps brackets every library kernel with CUDA events (for the
per-kernel durations behind `roofline`); those events cost the GPU about 2 us each, so `value`
comes from the first pass, which has none.

value = BF16 input bytes (2n) of all ranks per second of compress+decompress.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                  [--profile]

--impl reference times the plain C oracle on the host cores (one core) on a bounded sample of
the same workload.  With N > 1 (torchrun), every rank runs its own replica: the codec has no
collective, so scaling is weak.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compress+decompress GB/s on BF16 input (% of HBM peak); compression ratio"
DEFAULT_WORKLOAD = "grad_bucket_4096x14336"
L2_FLUSH_BYTES = 256 << 20
KERNEL_NAMES = {1: "stats", 2: "encode", 3: "decode"}
KERNEL_SOURCES = {"stats": "zc_stats.cu", "encode": "zc_encode.cu", "decode": "zc_decode.cu"}


# ---------------------------------------------------------------------------- ranks


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_group(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist

    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """The slowest rank's value (every rank gets it)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.marks: list[float] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())
            self.marks.append(time.time())

    def window(self, t0: float, t1: float):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line, t in zip(self.lines, self.marks):
            if getattr(self, "t0", 0) - 0.06 <= t <= getattr(self, "t1", 1e18) + 0.06:
                rows.append([c.strip() for c in line.split(",")])
        if not rows:
            rows = [[c.strip() for c in line.split(",")] for line in self.lines[-3:]]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, v in zip(self.REASONS, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------- helpers


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def source_sha(kernel: str) -> str:
    path = os.path.join(ROOT, "lossless_bf16_compression_gb300", "csrc", KERNEL_SOURCES[kernel])
    h = hashlib.sha256()
    for p in (path, os.path.join(ROOT, "lossless_bf16_compression_gb300", "csrc", "zc_common.cuh")):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this exact
    kernel source; None otherwise."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = source_sha(kernel)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload \
                    and parts[2] == want:
                return int(parts[3])
    return None


def cpu_baseline(x, budget_s: float = 10.0):
    """The oracle, as it stands, single-threaded on this host, on whole-buffer round trips
    repeated until `budget_s` seconds have passed (at least one)."""
    import oracle

    oracle.build()
    reps, t_total = 0, 0.0
    while reps == 0 or t_total < budget_s:
        t0 = time.perf_counter()
        s = oracle.compress(x)
        st, _ = oracle.decompress(s, x.size)
        t_total += time.perf_counter() - t0
        reps += 1
        if st != oracle.OK:
            raise RuntimeError("oracle round trip failed")
    return {"value": round(2 * x.size * reps / t_total / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} x whole-buffer round trip ({x.size} values, {t_total:.1f} s), "
                      f"host {os.uname().machine}, {os.cpu_count()} cores available"}


# ---------------------------------------------------------------------------- our arm


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    from lossless_bf16_compression_gb300 import binding as zc
    from lossless_bf16_compression_gb300 import build as zbuild
    from lossless_bf16_compression_gb300 import workloads

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the codec has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_group(world, "nccl")
    if rank == 0:
        zbuild.build()
    barrier(dist)
    zc.lib()

    x = workloads.make(args.workload)
    n = x.size
    xd = torch.from_numpy(x.view(np.int16)).to(device)
    cap = zc.zc_max_compressed_bytes(n)
    out = torch.empty(cap, dtype=torch.uint8, device=device)
    dec = torch.empty(n, dtype=torch.int16, device=device)
    ob = torch.zeros(1, dtype=torch.int64, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    def flush_l2():
        flush.zero_()  # evict everything: 2x the L2 capacity
        flush.view(torch.int32).sum()  # then read it back, leaving only clean lines behind
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    xp, op, dp, obp = xd.data_ptr(), out.data_ptr(), dec.data_ptr(), ob.data_ptr()

    def step():
        rc = zc.zc_compress(xp, n, zc.ZC_BASE_AUTO, op, obp, sh)
        rc |= zc.zc_decompress(op, dp, n, sh)
        if rc:
            raise RuntimeError(f"codec call failed: {rc}")

    zc.zc_status(sh, 1)
    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if args.profile:  # the plain step loop only, for profiler captures: no timing extras
        for _ in range(args.steps):
            flush_l2()
            step()
        torch.cuda.synchronize()
        st = zc.zc_status(sh, 1)
        ok = st == zc.ZC_OK and torch.equal(dec, xd)
        if rank == 0:
            print(json.dumps({"profile_run": args.workload, "n": n, "steps": args.steps, "verified": bool(ok)}))
        if not ok:
            raise SystemExit("profile run self-check failed")
        return

    def timed_steps(kernel_events):
        """K steps, L2 flushed before each (outside its events); per-kernel CUDA events too when
        asked (each event record costs the GPU about 2 us, so they stay out of the pass that
        gives `value`)."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if kernel_events:
            zc.zc_timing_collect()
            zc.zc_timing_enable(1)
        barrier(dist)
        torch.cuda.synchronize()
        t0 = time.time()
        for i in range(args.steps):
            flush_l2()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        t1 = time.time()
        recs = []
        if kernel_events:
            zc.zc_timing_enable(0)
            recs = zc.zc_timing_collect(1 << 20)
        return [s.elapsed_time(e) for s, e in zip(starts, ends)], recs, t0, t1

    # pass 1: the steps that give `value`, with the clock record
    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.start()
    step_ms, _, t_wall0, t_wall1 = timed_steps(kernel_events=False)
    clk = None
    if clocks:
        clocks.window(t_wall0, t_wall1)
        clk = clocks.stop()
    # pass 2: the same number of steps with every library kernel bracketed by CUDA events on its
    # stream, for per-kernel durations (the roofline) and the launch count
    _, records, _, _ = timed_steps(kernel_events=True)

    total_ms = max_over_ranks(sum(step_ms), dist, device)
    st = zc.zc_status(sh, 1)
    ok = st == zc.ZC_OK and torch.equal(dec, xd)
    total_bytes = int(ob.item())
    e0 = int(out[7].item())

    # per-kernel device time over the timed region
    per = {}
    for kid, ms in records:
        per.setdefault(KERNEL_NAMES.get(kid, str(kid)), []).append(ms)
    avg = {k: sum(v) / len(v) for k, v in per.items()}
    C = total_bytes
    alg = {"stats": 2 * n, "encode": 2 * n + C, "decode": C + 2 * n}
    dominant = max(avg, key=lambda k: avg[k] * len(per[k]))
    peak, peak_kind = measured_peaks()
    achieved = alg[dominant] / (avg[dominant] * 1e-3) / 1e9
    comp_ms = avg.get("stats", 0.0) + avg.get("encode", 0.0)
    dec_ms = avg.get("decode", 0.0)

    # End to end through the C ABI: every step copies its input from pinned host memory, runs
    # zc_compress + zc_decompress, and copies the decoded tensor back to pinned host memory.
    # Consecutive steps overlap on three streams with two sets of buffers, as a data pipeline
    # would run: step i's copy back (device to host) runs while step i+1's input is copied in
    # (host to device); the two directions use separate copy engines.
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    yh = [torch.empty(n, dtype=torch.int16).pin_memory() for _ in range(2)]
    xd2, out2, dec2, ob2 = [xd, torch.empty_like(xd)], [out, torch.empty_like(out)], \
        [dec, torch.empty_like(dec)], [ob, torch.zeros_like(ob)]
    s_in, s_codec, s_out = (torch.cuda.Stream(device) for _ in range(3))
    in_done, codec_done, out_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_step(i):
        b = i % 2
        if i >= 2:
            s_in.wait_event(codec_done[b])  # step i-2's compress has read xd2[b]
        with torch.cuda.stream(s_in):
            xd2[b].copy_(xh, non_blocking=True)
        in_done[b].record(s_in)
        s_codec.wait_event(in_done[b])
        if i >= 2:
            s_codec.wait_event(out_done[b])  # step i-2's decoded tensor has left dec2[b]
        rc = zc.zc_compress(xd2[b].data_ptr(), n, zc.ZC_BASE_AUTO, out2[b].data_ptr(), ob2[b].data_ptr(),
                            s_codec.cuda_stream)
        rc |= zc.zc_decompress(out2[b].data_ptr(), dec2[b].data_ptr(), n, s_codec.cuda_stream)
        if rc:
            raise RuntimeError(f"codec call failed: {rc}")
        codec_done[b].record(s_codec)
        s_out.wait_event(codec_done[b])
        with torch.cuda.stream(s_out):
            yh[b].copy_(dec2[b], non_blocking=True)
        out_done[b].record(s_out)

    e2e_steps = max(3, min(args.steps, 50))
    for i in range(4):  # warm-up
        e2e_step(i)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(s_in)
    for i in range(4, 4 + e2e_steps):
        e2e_step(i)
    e_end.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / e2e_steps, dist, device)
    last = (4 + e2e_steps - 1) % 2
    ok = ok and torch.equal(yh[last], xh) and zc.zc_status(s_codec.cuda_stream, 1) == zc.ZC_OK

    if rank != 0:
        return
    ms_per_step = total_ms / args.steps
    value = 2 * n * world / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u16",
        "data": "synthetic",
        "config": {"workload": args.workload, "n": n, "chunk": 4096, "base": "auto",
                   "l2": "flushed between steps (256 MiB write + read, outside the timed region)",
                   "kernel_times": "a second pass of K steps with CUDA events around each launch "
                                   "(they add about 14 us per step, so value comes from a pass without them)",
                   "parallelism": f"{world} independent replicas"},
        "compression_ratio": round(2 * n / C, 4),
        "stream_bytes": C,
        "e0": e0,
        "compress_gbs": round(2 * n / (comp_ms * 1e-3) / 1e9, 2) if comp_ms else None,
        "decompress_gbs": round(2 * n / (dec_ms * 1e-3) / 1e9, 2) if dec_ms else None,
        "kernel_us": {k: round(v * 1e3, 2) for k, v in avg.items()},
        "hbm_frac_by_kernel": {k: round(alg[k] / (avg[k] * 1e-3) / 1e9 / peak, 4) for k in avg},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "algorithmic_bytes": alg[dominant], "traffic": profiled_traffic(dominant, args.workload)},
        "e2e": {"value": round(2 * n * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": 2 * n, "d2h_bytes_per_step": 2 * n,
                "pipeline": "consecutive steps overlap on 3 streams, 2 buffer sets; no L2 flush"},
        "gpu_launches": len(records),  # library kernels launched in K steps (pass 2; pass 1 is identical)
        "clocks": clk,
        "verified": bool(ok),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x)
    print(json.dumps(line), flush=True)
    if not ok:
        raise SystemExit("bench self-check failed: the round trip was not exact")


# ---------------------------------------------------------------------------- reference arm


def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores: each step is a round trip of a bounded
    sample of the workload, sized so that all warm-up and timed steps take about a minute."""
    if rank != 0:
        return
    import oracle
    from lossless_bf16_compression_gb300 import workloads

    oracle.build()
    x = workloads.make(args.workload)
    probe = x[: 1 << 20]
    t0 = time.perf_counter()
    oracle.decompress(oracle.compress(probe), probe.size)
    per_value = (time.perf_counter() - t0) / probe.size
    m = int(min(x.size, max(1 << 16, 60.0 / (args.steps + args.warmup) / per_value)))
    sample = x[:m]
    for _ in range(args.warmup):
        oracle.decompress(oracle.compress(sample), m)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        s = oracle.compress(sample)
        st, _ = oracle.decompress(s, m)
        times.append(time.perf_counter() - t0)
        if st != oracle.OK:
            raise SystemExit("oracle round trip failed")
    ms = 1e3 * sum(times) / len(times)
    value = 2 * m / (ms * 1e-3) / 1e9
    desc = f"first {m} of {x.size} values per step, single-threaded, host {os.uname().machine}"
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u16", "data": "synthetic", "impl": "reference",
        "config": {"workload": args.workload, "n": int(x.size), "chunk": 4096, "base": "auto"},
        "compression_ratio": round(2 * m / s.size, 4),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="run warm-up + steps of the bare step loop (for ncu), print no bench line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
