#!/usr/bin/env python3
"""Benchmark: lossless BF16 exponent codec on GB300, one JSON line on stdout.

A step is one pass of the whole hot path over one synthetic buffer resident in HBM:
zc_compress in auto mode (statistics pass, window base, encode + single-pass chunk scan)
followed by zc_decompress.  The default workload is the largest single-GPU configuration,
2^29 N(0, 1) BF16 values (1 GiB).  The L2 cache is flushed between steps, outside the timed
region: a 256 MiB buffer is written and then read back, so the cache holds none of the step's
data and no dirty lines whose write-back the next kernel would pay for.  Steps are timed with
CUDA events on the stream the library launches on.

value = BF16 input bytes (2n) of all ranks per second of compress + decompress.

The same line also carries, for the default workload:
  compress / decompress    each operation timed on its own (an event between the two calls):
                           GB/s of BF16 input, algorithmic bytes (4n + C and C + 2n) per second
                           and their fraction of the measured HBM copy bandwidth;
  roofline                 the dominant kernel, from a pass with CUDA events around every
                           library kernel;
  e2e, cpu_baseline        the step through the C ABI with host buffers, and the oracle on the
                           host cores on a bounded sample;
and unless --no-extras:
  configs                  the same compress / decompress figures for every configuration of at
                           least 64M values (MoE activations, the adversarial tensor, N(0, 1) at
                           2^26 .. 2^29), L2 flushed between steps;
  sweep                    latency and GB/s per size for N(0, 1) buffers of 2^15 .. 2^29 values,
                           each compressed and decompressed 100 times back to back on one stream;
                           up to 2^22 values also the same 100 round trips replayed from a CUDA graph
                           (the device's time without the host's per-call cost).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                  [--no-extras] [--profile]

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
DEFAULT_WORKLOAD = "sweep_2^29"
# configurations of at least 64M values: the target of the roofline fractions
SINGLE_LAUNCH_MAX = 1 << 25  # the largest tensor zc_compress takes in one launch on a GB300
TARGET_CONFIGS = ["moe_a2a_16384x7168", "adversarial_256m", "sweep_2^26", "sweep_2^27", "sweep_2^28", "sweep_2^29"]
# the other configurations of the workload list (below the 64M-value line of the target)
OTHER_CONFIGS = ["weight_1m", "grad_bucket_4096x14336"]
SWEEP_SIZES = list(range(15, 30))  # 2^15 .. 2^29 values (64 KiB .. 1 GiB)
SWEEP_REPS = 100
L2_FLUSH_BYTES = 256 << 20
KERNEL_NAMES = {1: "stats", 2: "encode", 3: "decode", 4: "raw_form", 5: "small", 6: "medium", 7: "fused",
                8: "refit_stats", 9: "refit_encode"}
KERNEL_SOURCES = {"stats": "zc_stats.cu", "encode": "zc_encode.cu", "decode": "zc_decode.cu",
                  "raw_form": "zc_encode.cu", "small": "zc_small.cu", "medium": "zc_small.cu",
                  "fused": "zc_fused.cu", "refit_stats": "zc_stats.cu", "refit_encode": "zc_encode.cu"}


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
    """nvidia-smi samples of SM clock and throttle reasons while the timed regions run."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    PERIOD_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.marks: list[float] = []
        self.windows: list[tuple[float, float]] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
        """A timed region, by host wall clock (its GPU work was synchronized at both ends)."""
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        slack = 1.5 * self.PERIOD_MS / 1e3
        rows = [[c.strip() for c in line.split(",")] for line, t in zip(self.lines, self.marks)
                if any(a - slack <= t <= b + slack for a, b in self.windows)]
        if not rows:
            rows = [[c.strip() for c in line.split(",")] for line in self.lines[-3:]]
        sm = [float(r[1]) for r in rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, v in zip(self.REASONS, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "timed_s": round(sum(b - a for a, b in self.windows), 3)}


# ---------------------------------------------------------------------------- helpers


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def source_sha(kernel: str) -> str:
    """Hash of the kernel's source file and every header of the library (the kernels share code
    through them), so that profiled counters are used only for the exact source they came from."""
    csrc = os.path.join(ROOT, "lossless_bf16_compression_gb300", "csrc")
    h = hashlib.sha256()
    files = [KERNEL_SOURCES[kernel]] + sorted(f for f in os.listdir(csrc) if f.endswith((".cuh", ".h")))
    for name in files:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this exact kernel
    source: (bytes, workload it was taken on).  A capture on a smaller N(0, 1) sweep size is
    scaled to this one by the number of values (the traffic of these kernels grows in proportion
    to n at these sizes).  (None, None) when there is none."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None, None
    want = source_sha(kernel)
    scaled = (None, None)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) < 4 or line.startswith("#") or parts[0] != kernel or parts[2] != want:
                continue
            if parts[1] == workload:
                return int(parts[3]), workload
            if parts[1].startswith("sweep_2^") and workload.startswith("sweep_2^"):
                k0, k1 = int(parts[1][8:]), int(workload[8:])
                scaled = (int(parts[3]) << (k1 - k0) if k1 >= k0 else int(parts[3]) >> (k0 - k1), parts[1])
    return scaled


def cpu_baseline(x, budget_s: float = 10.0):
    """The oracle, as it stands, single-threaded on this host, on a round trip of the first M
    values of the workload, M sized from a 2^20-value probe so the round trip takes about
    `budget_s` seconds."""
    import oracle

    oracle.build()
    probe = x[: 1 << 20]
    t0 = time.perf_counter()
    oracle.decompress(oracle.compress(probe), probe.size)
    per_value = (time.perf_counter() - t0) / probe.size
    m = int(min(x.size, max(1 << 20, budget_s / per_value)))
    sample = x[:m]
    t0 = time.perf_counter()
    s = oracle.compress(sample)
    st, _ = oracle.decompress(s, m)
    dt = time.perf_counter() - t0
    if st != oracle.OK:
        raise RuntimeError("oracle round trip failed")
    return {"value": round(2 * m / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"one round trip of the first {m} of {x.size} values ({dt:.1f} s), "
                      f"host {os.uname().machine}, {os.cpu_count()} cores available, 1 used"}


# ---------------------------------------------------------------------------- our arm


class Codec:
    """Device buffers sized for up to `n_max` values and the library calls of one step."""

    def __init__(self, zc, torch, device, n_max):
        self.zc, self.torch, self.device = zc, torch, device
        self.xd = torch.empty(n_max, dtype=torch.int16, device=device)
        self.out = torch.empty(zc.zc_max_compressed_bytes(n_max), dtype=torch.uint8, device=device)
        self.dec = torch.empty(n_max, dtype=torch.int16, device=device)
        self.ob = torch.zeros(1, dtype=torch.int64, device=device)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.stream = torch.cuda.current_stream(device)
        self.sh = self.stream.cuda_stream
        self.n = 0

    def load(self, x):
        import numpy as np

        self.n = x.size
        self.xd[:self.n].copy_(self.torch.from_numpy(x.view(np.int16)))
        self.dec[:self.n].zero_()

    def flush_l2(self):
        self.flush.zero_()  # evict everything: 2x the L2 capacity
        self.flush.view(self.torch.int32).sum()  # then read it back, leaving only clean lines

    def compress(self):
        rc = self.zc.zc_compress(self.xd.data_ptr(), self.n, self.zc.ZC_BASE_AUTO, self.out.data_ptr(),
                                 self.ob.data_ptr(), self.sh)
        if rc:
            raise RuntimeError(f"zc_compress failed: {rc}")

    def decompress(self):
        rc = self.zc.zc_decompress(self.out.data_ptr(), self.dec.data_ptr(), self.n, self.sh)
        if rc:
            raise RuntimeError(f"zc_decompress failed: {rc}")

    def verified(self) -> bool:
        st = self.zc.zc_status(self.sh, 1)
        return st == self.zc.ZC_OK and bool(self.torch.equal(self.dec[:self.n], self.xd[:self.n]))

    def stream_bytes(self) -> int:
        return int(self.ob.item())

    def compress_path(self) -> str:
        """Which way the last compression went (the control block at the head of the workspace)."""
        import numpy as np

        n = self.n
        if n <= SINGLE_LAUNCH_MAX:
            return "one launch"
        ws = (self.zc.zc_max_stream_bytes(n) + 255) // 256 * 256
        words = self.out[ws:ws + 256].cpu().numpy().view(np.uint32)
        raw = " (raw pass)" if words[84 // 4] else ""
        if words[240 // 4]:  # the sample was not confident, or the guess did not hold
            return "statistics + encode" + raw
        return "speculative: one read of the input"

    def e0(self) -> int:
        return int(self.out[7].item())

    def flushed_steps(self, steps, split, clocks=None, dist=None):
        """`steps` steps, L2 flushed before each outside its events.  split=False: one event pair
        per step (start, end); split=True: an event between compress and decompress as well.
        Returns per-step milliseconds: (compress+decompress,) or (compress, decompress)."""
        torch = self.torch
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3 if split else 2)] for _ in range(steps)]
        barrier(dist)
        torch.cuda.synchronize()
        t0 = time.time()
        for e in ev:
            self.flush_l2()
            e[0].record(self.stream)
            self.compress()
            if split:
                e[1].record(self.stream)
            self.decompress()
            e[-1].record(self.stream)
        torch.cuda.synchronize()
        barrier(dist)
        if clocks:
            clocks.window(t0, time.time())
        if split:
            return [e[0].elapsed_time(e[1]) for e in ev], [e[1].elapsed_time(e[2]) for e in ev]
        return ([e[0].elapsed_time(e[1]) for e in ev],)

    def replayed(self, reps):
        """The same `reps` round trips captured once in a CUDA graph and replayed: mean ms per round
        trip without the host's per-call cost (None when the calls cannot be captured)."""
        torch = self.torch
        try:
            side = torch.cuda.Stream(self.device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                sh = side.cuda_stream
                with torch.cuda.graph(g, stream=side):
                    for _ in range(reps):
                        self.zc.zc_compress(self.xd.data_ptr(), self.n, self.zc.ZC_BASE_AUTO, self.out.data_ptr(),
                                            self.ob.data_ptr(), sh)
                        self.zc.zc_decompress(self.out.data_ptr(), self.dec.data_ptr(), self.n, sh)
            self.dec[:self.n].zero_()
            g.replay()
            torch.cuda.synchronize()
            if not self.verified():  # the replay must really have run the codec
                return None
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(self.stream)
            g.replay()
            b.record(self.stream)
            torch.cuda.synchronize()
            del g
            return a.elapsed_time(b) / reps
        except Exception:  # noqa: BLE001 -- capture is optional; the plain numbers stand
            torch.cuda.synchronize()
            return None

    def back_to_back(self, reps, clocks=None):
        """`reps` compress+decompress round trips back to back on one stream (no flush), then
        `reps` compresses alone and `reps` decompresses alone: mean ms of each."""
        torch = self.torch
        t = []
        t_wall = time.time()
        for what in ("round_trip", "compress", "decompress"):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(self.stream)
            for _ in range(reps):
                if what != "decompress":
                    self.compress()
                if what != "compress":
                    self.decompress()
            b.record(self.stream)
            torch.cuda.synchronize()
            t.append(a.elapsed_time(b) / reps)
        if clocks:
            clocks.window(t_wall, time.time())
        return t


def loopback_steps(zc, torch, cd, steps, clocks=None, dist=None):
    """`steps` zc_loopback calls (auto mode), L2 flushed before each outside its events; the
    decoded values are checked against the input."""
    n = cd.n
    out = torch.empty(zc.zc_loopback_bytes(n), dtype=torch.uint8, device=cd.device)
    ob = torch.zeros(1, dtype=torch.int64, device=cd.device)
    vals = cd.dec[:n]

    def call():
        rc = zc.zc_loopback(cd.xd.data_ptr(), n, zc.ZC_BASE_AUTO, out.data_ptr(), ob.data_ptr(), vals.data_ptr(),
                            cd.sh)
        if rc:
            raise RuntimeError(f"zc_loopback failed: {rc}")

    for _ in range(3):
        cd.flush_l2()
        call()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.time()
    for e in ev:
        cd.flush_l2()
        e[0].record(cd.stream)
        call()
        e[1].record(cd.stream)
    torch.cuda.synchronize()
    if clocks:
        clocks.window(t0, time.time())
    ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    ok = zc.zc_status(cd.sh, 1) == zc.ZC_OK and bool(torch.equal(vals, cd.xd[:n]))
    ok = ok and int(ob.item()) == cd.stream_bytes() and bool(torch.equal(out[:int(ob.item())], cd.out[:int(ob.item())]))
    del out
    return {"us": round(ms * 1e3, 2), "gbs_input": round(2 * n / ms / 1e6, 1), "verified": ok}


def op_figures(n, C, comp_ms, dec_ms, peak, path=None):
    """Compress and decompress figures of one workload from their mean times.  Compress
    frac_of_peak counts 4n + C bytes (the statistics pass and the coding pass, the definition the
    target is stated in); frac_of_one_pass counts 2n + C (one read of the input and one write of
    the stream: what the speculative path moves when its guess holds, and a lower bound for any
    path)."""
    return {
        "n": n, "stream_bytes": C, "compression_ratio": round(2 * n / C, 4),
        "stream_form": "raw" if C == 32 + (2 * n + 15) // 16 * 16 else "coded",
        "compress": {"us": round(comp_ms * 1e3, 2), "gbs_input": round(2 * n / comp_ms / 1e6, 1),
                     "gbs_algorithmic": round((4 * n + C) / comp_ms / 1e6, 1),
                     "frac_of_peak": round((4 * n + C) / comp_ms / 1e6 / peak, 4),
                     "frac_of_one_pass": round((2 * n + C) / comp_ms / 1e6 / peak, 4),
                     **({"path": path} if path else {})},
        "decompress": {"us": round(dec_ms * 1e3, 2), "gbs_input": round(2 * n / dec_ms / 1e6, 1),
                       "gbs_algorithmic": round((C + 2 * n) / dec_ms / 1e6, 1),
                       "frac_of_peak": round((C + 2 * n) / dec_ms / 1e6 / peak, 4)},
    }


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
    peak, peak_kind = measured_peaks()

    x = workloads.make(args.workload)
    n = x.size
    extras = not args.no_extras and world == 1 and not args.profile
    n_max = max(n, 1 << 29) if extras else n
    cd = Codec(zc, torch, device, n_max)
    cd.load(x)

    def step():
        cd.compress()
        cd.decompress()

    zc.zc_status(cd.sh, 1)
    for _ in range(args.warmup):
        cd.flush_l2()
        step()
    torch.cuda.synchronize()
    if args.profile:  # the plain step loop only, for profiler captures: no timing extras
        for _ in range(args.steps):
            cd.flush_l2()
            step()
        torch.cuda.synchronize()
        ok = cd.verified()
        if rank == 0:
            print(json.dumps({"profile_run": args.workload, "n": n, "steps": args.steps, "verified": ok}))
        if not ok:
            raise SystemExit("profile run self-check failed")
        return

    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.start()
    # pass 1: the steps that give `value` (one event pair per step)
    (step_ms,) = cd.flushed_steps(args.steps, split=False, clocks=clocks, dist=dist)
    total_ms = max_over_ranks(sum(step_ms), dist, device)
    # pass 2: compress and decompress timed apart (an event between the two calls)
    comp, dec = cd.flushed_steps(args.steps, split=True, clocks=clocks, dist=dist)
    comp_ms, dec_ms = sum(comp) / len(comp), sum(dec) / len(dec)
    # pass 3: every library kernel bracketed by CUDA events on its stream, for per-kernel
    # durations (the roofline) and the launch count; those events cost the GPU about 2 us each
    # and break the overlap of the statistics and encode kernels, so no other figure uses them
    zc.zc_timing_collect()
    zc.zc_timing_enable(1)
    cd.flushed_steps(args.steps, split=False, clocks=clocks, dist=dist)
    zc.zc_timing_enable(0)
    records = zc.zc_timing_collect(1 << 20)
    ok = cd.verified()
    # pass 4: the loopback, compress and decompress in one launch (chunks decoded as they reach
    # the stream), against the same steps run one call after the other
    lb = loopback_steps(zc, torch, cd, args.steps, clocks, dist)
    ok = ok and lb["verified"]
    C = cd.stream_bytes()
    e0 = cd.e0()

    per = {}
    for kid, ms in records:
        per.setdefault(KERNEL_NAMES.get(kid, str(kid)), []).append(ms)
    avg = {k: sum(v) / len(v) for k, v in per.items()}
    raw_stream = C == 32 + (2 * n + 15) // 16 * 16 and int(cd.out[6].item()) == 0
    # A raw stream is written by one of two steps, each reading the values and writing them
    # behind the header: the encode kernel's raw pass when the statistics pass predicted it
    # (nothing is coded then; the control block at the head of the workspace says so), else the
    # raw-form step after coding.
    ws = (zc.zc_max_stream_bytes(n) + 255) // 256 * 256
    raw_pass = raw_stream and int(cd.out[ws + 84:ws + 88].cpu().numpy().view(np.uint32)[0]) == 1
    raw_by = ("encode (raw pass)" if raw_pass else "raw_form") if raw_stream else None
    alg = {"stats": 2 * n, "encode": 4 * n if raw_pass else 2 * n + C, "decode": C + 2 * n,
           "raw_form": 4 * n if raw_stream and not raw_pass else 0, "fused": 4 * n + C}
    dominant = max((k for k in avg if alg.get(k)), key=lambda k: avg[k] * len(per[k]))
    achieved = alg[dominant] / (avg[dominant] * 1e-3) / 1e9
    traffic, traffic_from = profiled_traffic(dominant, args.workload)

    # per-configuration figures and the small-message sweep (rank 0 of a single-GPU run)
    configs, sweep = {}, {}
    if extras:
        head = {"compress_ms": comp_ms, "decompress_ms": dec_ms, "C": C, "e0": e0, "ok": ok}
        for k in SWEEP_SIZES:
            name = f"sweep_2^{k}"
            cd.load(x if name == args.workload else workloads.make(name))
            m = cd.n
            for _ in range(3):
                step()
            bt = cd.back_to_back(SWEEP_REPS, clocks=clocks)
            sweep[name] = {"n": m, "round_trip_us": round(bt[0] * 1e3, 2), "compress_us": round(bt[1] * 1e3, 2),
                           "decompress_us": round(bt[2] * 1e3, 2),
                           "gbs_input": round(2 * m / bt[0] / 1e6, 1), "verified": cd.verified()}
            if k <= 22:  # small messages: the device's own time per round trip, without host calls
                rp = cd.replayed(SWEEP_REPS)
                sweep[name]["graph_round_trip_us"] = round(rp * 1e3, 2) if rp else None
                sweep[name]["verified"] = sweep[name]["verified"] and cd.verified()
            if name in TARGET_CONFIGS:
                if name == args.workload:
                    c_ms, d_ms, Cc, ee, okc = head["compress_ms"], head["decompress_ms"], head["C"], head["e0"], ok
                else:
                    c, d = cd.flushed_steps(args.steps, split=True, clocks=clocks)
                    c_ms, d_ms, Cc, ee, okc = sum(c) / len(c), sum(d) / len(d), cd.stream_bytes(), cd.e0(), \
                        cd.verified()
                configs[name] = {**op_figures(m, Cc, c_ms, d_ms, peak, cd.compress_path()), "e0": ee,
                                 "verified": okc, "target": True}
        for name in TARGET_CONFIGS + OTHER_CONFIGS:
            if name in configs:
                continue
            cd.load(x if name == args.workload else workloads.make(name))
            for _ in range(3):
                step()
            c, d = cd.flushed_steps(args.steps, split=True, clocks=clocks)
            configs[name] = {**op_figures(cd.n, cd.stream_bytes(), sum(c) / len(c), sum(d) / len(d), peak,
                                          cd.compress_path()),
                             "e0": cd.e0(), "verified": cd.verified(), "target": name in TARGET_CONFIGS}
        cd.load(x)
    clk = clocks.stop() if clocks else None

    # End to end through the C ABI: every step copies its input from pinned host memory, runs
    # zc_compress + zc_decompress, and copies the decoded tensor back to pinned host memory.
    # Consecutive steps overlap on three streams with two sets of buffers, as a data pipeline
    # would run: step i's copy back (device to host) runs while step i+1's input is copied in
    # (host to device); the two directions use separate copy engines.
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    yh = [torch.empty(n, dtype=torch.int16).pin_memory() for _ in range(2)]
    xd2 = [cd.xd[:n], torch.empty(n, dtype=torch.int16, device=device)]
    out2 = [cd.out, torch.empty(zc.zc_max_compressed_bytes(n), dtype=torch.uint8, device=device)]
    dec2 = [cd.dec[:n], torch.empty(n, dtype=torch.int16, device=device)]
    ob2 = [cd.ob, torch.zeros_like(cd.ob)]
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
    head = op_figures(n, C, comp_ms, dec_ms, peak, cd.compress_path())
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
                   "passes": "value: K steps with one event pair each; compress/decompress: K more steps with "
                             "an event between the two calls; kernel_us and roofline: K more steps with events "
                             "around every library kernel",
                   "parallelism": f"{world} independent replicas"},
        "compression_ratio": head["compression_ratio"],
        "stream_bytes": C,
        "e0": e0,
        "compress": head["compress"],
        "decompress": head["decompress"],
        "loopback": {**lb, "sequential_us": round((comp_ms + dec_ms) * 1e3, 2),
                     "speedup_vs_sequential": round((comp_ms + dec_ms) * 1e3 / lb["us"], 3),
                     "what": "zc_loopback: compress and decompress in one launch, each chunk decoded as soon as "
                             "its bytes are in the stream; sequential = zc_compress then zc_decompress"},
        "kernel_us": {k: round(v * 1e3, 2) for k, v in avg.items()},
        "hbm_frac_by_kernel": {k: round(alg[k] / (avg[k] * 1e-3) / 1e9 / peak, 4) for k in avg if alg.get(k)},
        "stream_form": "raw" if raw_stream else "coded",
        "raw_written_by": raw_by,
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "algorithmic_bytes": alg[dominant], "traffic": traffic,
                     "traffic_from": traffic_from},
        "e2e": {"value": round(2 * n * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": 2 * n, "d2h_bytes_per_step": 2 * n,
                "pipeline": "consecutive steps overlap on 3 streams, 2 buffer sets; no L2 flush"},
        "gpu_launches": len(records),  # library kernels launched in the K steps of pass 3
        "clocks": clk,
        "verified": bool(ok),
    }
    if configs:
        line["configs"] = configs
    if sweep:
        line["sweep"] = sweep
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x)
    print(json.dumps(line), flush=True)
    bad = [k for k, v in {**configs, **sweep}.items() if not v["verified"]]
    if not ok or bad:
        raise SystemExit(f"bench self-check failed: the round trip was not exact ({bad or args.workload})")


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
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-configuration figures and the size sweep")
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
