#!/usr/bin/env python3
"""Throughput of the fused PSNR-noise + moment statistics on GB300.

One step = one batch of synthetic planes already resident in HBM through
``vqx_plane_stats_submit`` + ``vqx_plane_stats_finish`` (the whole hot path,
the work of one ``vqx_plane_stats`` call: load, per-pixel terms, exact integer
reduction, per-frame sums, read-back, conclusion in double).  Steps are
pipelined one deep: batch i + 1 is enqueued before batch i is waited on and
concluded.  The default batch is 32 frame pairs of 3840x2160 16-bit luma
(1.06 GB, larger than L2, so no flush is needed between steps).

Prints ONE JSON line (rank 0).  ``value`` is whole-job frame pairs/s; ``e2e``
is the same metric through ``vqx_plane_stats_host`` with the planes in pinned
host memory (copies inside the timed region); ``roofline`` is the fused
kernel's algorithmic bytes per launch over its CUDA-event launch time against
the measured HBM copy bandwidth; ``cpu_baseline`` is the CPU oracle on this
host's cores on a bounded sample.

``--impl reference`` times the CPU oracle itself as the reference arm (there is
no runnable reference implementation of this path).  Under torchrun (N > 1)
every rank runs its own batch (frames are independent: weak scaling, no
collective in the data path); rank 0 prints.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "frame pairs/s and HBM GB/s (fused PSNR+moments), 3840x2160 16-bit, 1 GB300"
UNIT = "frame pairs/s"


def chroma_workloads(wlo):
    """The two 4:2:0 chroma planes that go with the luma workload ``wlo``:
    half the width and height, the same content recipe, their own seeds."""
    import dataclasses

    return [dataclasses.replace(wlo, name=wlo.name + "_c%d" % k, width=max(1, wlo.width // 2),
                                height=max(1, wlo.height // 2), seed=wlo.seed + 1000 * k)
            for k in (1, 2)]


def metric_for(op, wlo):
    if op == "stats":
        return METRIC
    what = {"int_psnr": "integer psnr", "ordered": "fused PSNR+moments, CPU-order replay",
            "planes420": "fused PSNR+moments, 4:2:0 Y+Cb+Cr",
            "scores": "fused PSNR+moments and integer psnr, one read"}[op]
    return "frame pairs/s and HBM GB/s (%s), %dx%d %d-bit, 1 GB300" % (
        what, wlo.width, wlo.height, wlo.bpc)
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=None, help="workload name (default: the 3840x2160 16-bit batch)")
    p.add_argument("--e2e-steps", type=int, default=60)
    p.add_argument("--e2e-repeats", type=int, default=5,
                   help="timed regions of e2e steps; the e2e figure is their median")
    p.add_argument("--repeats", type=int, default=21,
                   help="at least this many timed regions of K steps; value is their median")
    p.add_argument("--min-timed-seconds", type=float, default=1.5,
                   help="repeat the timed region until about this much wall time has passed, so "
                        "that the clock sampler sees the GPU under load")
    p.add_argument("--inst-repeats", type=int, default=5,
                   help="instrumented regions for the per-launch kernel times")
    p.add_argument("--config-seconds", type=float, default=0.4,
                   help="the same, for each of the other measured configurations")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other measured configurations after the headline")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--op", choices=["stats", "int_psnr", "scores", "ordered", "planes420", "hvs"],
                   default="stats",
                   help="stats: the fused float_psnr + moments pass (the headline); int_psnr: "
                        "the integer psnr (vqx_plane_int_psnr); scores: both from one read "
                        "(vqx_plane_scores); ordered: the CPU-order replay "
                        "past 2^53 units (vqx_plane_stats_ordered_submit / _finish); "
                        "planes420: the workload as the luma of 4:2:0 video, Y, Cb and Cr "
                        "through one vqx_planes_stats call a step; hvs: psnr_hvs plane sums "
                        "of a batch of term planes (vqx_psnr_hvs_sum_submit / _finish)")
    p.add_argument("--record-traffic", metavar="NCU_REP", default=None,
                   help="write the DRAM traffic record of the fused kernel from an ncu report "
                        "(read here with ncu -i; needs no GPU) and exit")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value, pg=None, device=None):
    """The maximum of ``value`` over all ranks (the slowest rank's time), or
    ``value`` itself without a process group."""
    if pg is None:
        return value
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, frames_per_rank, steps, seconds):
    """Whole-job frame pairs per second: every rank's frames over the slowest
    rank's time (weak scaling: each rank reduces its own batch)."""
    return world * frames_per_rank * steps / seconds


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 100 ms, stamped with host time when read."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "100"]
        if gpu_id is not None:
            cmd += ["-i", str(gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside:  # a short timed region: take the samples nearest to it
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            inside = [p for _, p in near]
            note = "no sample inside the timed region; nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower() == "active"})
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        pw = [num(p[3]) for p in inside if num(p[3]) is not None]
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": num(inside[0][2]),
            "reasons": reasons,
            "power_w_max": max(pw) if pw else None,
            "samples": len(inside),
            "note": note,
        }


def gpu_smi_id(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------- roofline inputs
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The sources that define the fused kernel (its device code) and its launch
# (segment planning, grid, flags); the other headers hold other entry points'
# kernels, which cannot change this one.
FUSED_SOURCES = ("vqx_kernels.cuh", "vqx_plane_stats.cu")


def kernel_source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_full_reference_gb300", "csrc")
    for name in FUSED_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "fused_stream_traffic.json")
KERNEL_LABEL = "fused_stream_tma<%d, 16, 1536, 2, DenseSource, TermSums<%d>>"
# the capture the traffic record is taken from (the plain command runs first)
TRAFFIC_CAPTURE = ("ncu --set full --clock-control none -k regex:fused_stream -s 3 -c 1 "
                   "-o prof_fused_stream python bench.py --steps 3 --warmup 3 --no-cpu --no-e2e "
                   "--no-configs --repeats 1 --min-timed-seconds 0 --inst-repeats 1")


def recorded_traffic(workload_name):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary,
    or None when the kernel sources changed since it was taken."""
    path = TRAFFIC_RECORD
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_digest():
        return None
    per = rec.get("per_launch_bytes", {}).get(workload_name)
    return float(per) if per is not None else None


def write_traffic_record(report, wlo):
    """Read the fused kernel's launch from an ncu report (``ncu -i``, no GPU
    needed) and write the traffic record that ``recorded_traffic`` reads,
    keyed by the current kernel sources."""
    import csv

    out = subprocess.run(["ncu", "-i", report, "--page", "raw", "--csv"], capture_output=True,
                         text=True, check=True).stdout
    rows = list(csv.reader(out.splitlines()))
    hdr, units = rows[0], rows[1]
    launches = [dict(zip(hdr, zip(units, r))) for r in rows[2:]]
    launches = [d for d in launches if "fused_stream_tma" in d.get("Kernel Name", ("", ""))[1]]
    if not launches:
        raise SystemExit("no fused_stream_tma launch in %s" % report)
    d = launches[0]
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
             "ns": 1e-3, "us": 1.0, "ms": 1e3, "s": 1e6,
             "nsecond": 1e-3, "usecond": 1.0, "msecond": 1e3, "second": 1e6}

    def val(name):
        unit, v = d[name]
        return float(v.replace(",", "")) * scale.get(unit, 1.0)

    rd, wr = val("dram__bytes_read.sum"), val("dram__bytes_write.sum")
    bps = 1 if wlo.bpc == 8 else 2
    rec = {
        "kernel": KERNEL_LABEL % (wlo.bpc, wlo.bpc),
        "source_sha256": kernel_source_digest(),
        "per_launch_bytes": {wlo.name: rd + wr},
        "dram_bytes_read": rd,
        "dram_bytes_write": wr,
        "algorithmic_bytes": 2 * wlo.width * wlo.height * bps * wlo.n_frames,
        "gpu_dram_throughput_pct": float(d["gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed"][1]),
        "duration_us": val("gpu__time_duration.sum"),
        "command": TRAFFIC_CAPTURE,
    }
    with open(TRAFFIC_RECORD, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec))
    return 0


# ---------------------------------------------------------------- CPU oracle timing
def time_oracle(wlo, ref, dist, seconds, cores, rows=None, min_rounds=1, op="stats", extra=()):
    """Run the CPU oracle over frames (or bands of ``rows`` rows) of the batch
    on ``cores`` threads until ``seconds`` have passed.  Returns (pairs/s,
    pairs done, elapsed s).  ctypes drops the GIL inside the C calls.
    ``extra``: (ref, dist) arrays of half-size planes taken with each frame
    (the chroma of 4:2:0 video), half the rows of each band."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    orc = oracle.load()
    n, h, w = ref.shape
    band = h if rows is None else max(1, min(rows, h))
    stride = w * ref.itemsize

    def one(k):
        f = k % n
        y0 = (k * 7919) % (h - band + 1) if band < h else 0
        if op != "int_psnr":
            orc.batch(ref[f, y0 : y0 + band], dist[f, y0 : y0 + band], w, band, stride, wlo.bpc, 1)
        if op in ("int_psnr", "scores"):
            orc.int_psnr(ref[f, y0 : y0 + band], dist[f, y0 : y0 + band], w, band, stride, wlo.bpc, 1)
        for cr, cd in extra:
            ch, cw = cr.shape[1:]
            cb = max(1, min(ch, band // 2))
            c0 = min(y0 // 2, ch - cb)
            orc.batch(cr[f, c0 : c0 + cb], cd[f, c0 : c0 + cb], cw, cb, cw * cr.itemsize, wlo.bpc, 1)
        return band

    done_rows = 0
    k = 0
    t0 = time.perf_counter()
    rounds = 0
    with ThreadPoolExecutor(cores) as ex:
        while True:
            done_rows += sum(ex.map(one, range(k, k + cores)))
            k += cores
            rounds += 1
            if rounds >= min_rounds and time.perf_counter() - t0 >= seconds:
                break
    el = time.perf_counter() - t0
    pairs = done_rows / h
    return pairs / el, pairs, el


# ---------------------------------------------------------------- reference arm
def run_reference(args, wlo):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cores = host_cores()
    frames = list(range(min(wlo.n_frames, max(cores, 1))))
    ref, dist = wlo.generate(frames)
    extra = [c.generate(frames) for c in chroma_workloads(wlo)] if args.op == "planes420" else ()
    # size one step so that warm-up plus timed steps take about two minutes
    per_step_s = min(0.5, 120.0 / max(args.steps + args.warmup, 1))
    rate, _, _ = time_oracle(wlo, ref, dist, 0.0, 1, rows=64, op=args.op, extra=extra)  # calibration
    rows_per_s = rate * wlo.height
    rows = int(max(1, min(wlo.height, rows_per_s * per_step_s)))
    for _ in range(args.warmup):
        time_oracle(wlo, ref, dist, 0.0, cores, rows=rows, op=args.op, extra=extra)
    t0 = time.perf_counter()
    pairs = 0.0
    for _ in range(args.steps):
        _, p, _ = time_oracle(wlo, ref, dist, 0.0, cores, rows=rows, op=args.op, extra=extra)
        pairs += p
    el = time.perf_counter() - t0
    value = pairs / el
    sample = ("%d bands of %d rows (of %d) of %s frames per step, one band per thread"
              % (cores, rows, wlo.height, wlo.name))
    line = {
        "impl": "reference",
        "metric": metric_for(args.op, wlo),
        "value": value,
        "unit": UNIT,
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": el * 1e3 / max(args.steps, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int64 squares, u64 sums" if args.op == "int_psnr" else "f32 terms, f64 sums",
        "data": "synthetic",
        "config": {"workload": wlo.name, "frames": wlo.n_frames, "width": wlo.width,
                   "height": wlo.height, "bpc": wlo.bpc, "oracle": "plain C, raster-order double sums"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def repeat_count(region_s, min_repeats, min_seconds, cap=5000):
    """How many timed regions to run: at least ``min_repeats``, and enough
    to fill ``min_seconds`` of wall time at ``region_s`` seconds a region
    (so that the clock sampler sees the GPU under load), at most ``cap``."""
    want = min_repeats
    if region_s > 0:
        want = max(want, int(math.ceil(min_seconds / region_s)))
    return int(min(max(want, 1), max(cap, min_repeats)))


def summarize_regions(region_ms, steps):
    """Median, minimum and maximum of the timed regions (ms, K steps each),
    and the median's time per step."""
    s = sorted(region_ms)
    return {"repeats": len(s), "median_ms": statistics.median(s), "min_ms": s[0], "max_ms": s[-1],
            "p10_ms": s[int(0.1 * (len(s) - 1))], "p90_ms": s[int(0.9 * (len(s) - 1))],
            "ms_per_step": statistics.median(s) / max(steps, 1)}


class BenchDevice:
    """What every measurement on this rank shares: torch, the binding, the
    device, the launching stream and the process group."""

    def __init__(self, world, local):
        import torch

        __import__("__graft_entry__").build()
        import exact_full_reference_gb300 as vqx

        self.torch, self.vqx, self.so = torch, vqx, vqx.library()
        self.world, self.pg = world, None
        if world > 1:
            import torch.distributed as dist

            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
            self.pg = dist
        torch.cuda.set_device(local)
        self.dev = torch.cuda.current_device()
        self.stream = torch.cuda.Stream()
        self.sh = self.stream.cuda_stream
        self.l2_bytes = getattr(torch.cuda.get_device_properties(self.dev), "L2_cache_size", 0) or (129 << 20)

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()


OP_API = {"stats": "vqx_plane_stats", "int_psnr": "vqx_plane_int_psnr",
          "scores": "vqx_plane_scores", "ordered": "vqx_plane_stats_ordered",
          "planes420": "vqx_planes_stats"}


class Stepper:
    """Pipelined steps of submit / finish pairs and their timed regions.
    Subclasses provide submit(), finish(handle), ``flush`` (an L2-sized
    batch: each step timed on its own after overwriting the L2) and
    ``scratch`` (the buffer that overwrites it)."""

    flush = False
    scratch = None

    def steps(self, k):
        """k whole steps, pipelined: batch i + 1 is enqueued before batch i is
        waited on and concluded, so the device runs the next batch's kernels
        while the host concludes this one."""
        prev = None
        for _ in range(k):
            cur = self.submit()
            if prev is not None:
                self.finish(prev)
            prev = cur
        if prev is not None:
            self.finish(prev)

    def flushed_steps(self, k):
        """k steps, each after an L2 flush; returns the summed step time (ms)."""
        torch, stream = self.ctx.torch, self.ctx.stream
        total = 0.0
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        for _ in range(k):
            with torch.cuda.stream(stream):
                self.scratch.zero_()
            e0.record(stream)
            self.finish(self.submit())
            e1.record(stream)
            e1.synchronize()
            total += e0.elapsed_time(e1)
        return total

    def region(self, steps, instrumented):
        """K steps between a barrier + synchronize on both sides, timed with
        CUDA events on the launching stream (L2-sized batches: each step after
        a flush, flush excluded).  With ``instrumented`` the library also
        records CUDA events around its kernels inside every call, which costs
        the overlap of consecutive launches, so throughput comes from the
        uninstrumented regions.  Returns (max-over-ranks ms, wall t0, t1)."""
        ctx = self.ctx
        torch = ctx.torch
        ctx.barrier()
        torch.cuda.synchronize()
        ctx.vqx.profile_enable(instrumented)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        if self.flush:
            ms = self.flushed_steps(steps)
        else:
            ev0.record(ctx.stream)
            self.steps(steps)  # the last conclusion is inside the region too
            ev1.record(ctx.stream)
        torch.cuda.synchronize()
        t1 = time.time()
        if not self.flush:
            ms = ev0.elapsed_time(ev1)
        ctx.barrier()
        ctx.vqx.profile_enable(False)
        return reduce_max(ms, ctx.pg, ctx.dev), t0, t1

    def measure(self, steps, warmup, min_repeats, min_seconds, inst_repeats):
        """Warm up, then the timed regions (repeated: at least min_repeats and
        about min_seconds of wall time, the same count on every rank), then
        inst_repeats instrumented regions for the per-launch kernel times."""
        ctx = self.ctx
        self.steps(max(warmup, 3))
        ctx.torch.cuda.synchronize()
        calib_ms, c0, c1 = self.region(steps, False)
        reps = repeat_count(c1 - c0, min_repeats, min_seconds)
        reps = int(reduce_max(reps, ctx.pg, ctx.dev))
        ctx.vqx.profile_read(reset=True)
        regions, t_first, t_last = [], None, None
        for _ in range(reps):
            ms, t0, t1 = self.region(steps, False)
            regions.append(ms)
            t_first = t0 if t_first is None else t_first
            t_last = t1
        counted = ctx.vqx.profile_read(reset=True)
        for _ in range(max(inst_repeats, 1)):
            self.region(steps, True)
        prof = ctx.vqx.profile_read(reset=True)
        return {"regions": summarize_regions(regions, steps), "counted": counted, "prof": prof,
                "t0": t_first, "t1": t_last, "reps": reps}


class Batch(Stepper):
    """One workload's planes on the device and the op's submit / finish
    calls on them (the call a user makes; arguments only)."""

    def __init__(self, ctx, wlo, op):
        import ctypes

        import numpy as np

        torch, vqx, so = ctx.torch, ctx.vqx, ctx.so
        self.ctx, self.wlo, self.op = ctx, wlo, op
        self.ref, self.dist = wlo.generate()
        n, h, w = self.ref.shape
        self.n = n
        stride = w * wlo.bytes_per_sample
        self.rbytes = self.ref.reshape(-1).view(np.uint8)
        self.dbytes = self.dist.reshape(-1).view(np.uint8)
        self.d_ref = torch.from_numpy(self.rbytes).to(ctx.dev)
        self.d_dist = torch.from_numpy(self.dbytes).to(ctx.dev)
        torch.cuda.synchronize()
        self.chroma_np, chroma_dev = [], []
        self.out = np.zeros(n, vqx.INT_PSNR_DTYPE if op == "int_psnr" else vqx.FRAME_STATS_DTYPE)
        self.out2 = np.zeros(n, vqx.INT_PSNR_DTYPE)  # scores: the integer psnr records
        if op == "planes420":
            self.out = np.zeros((n, 3), vqx.FRAME_STATS_DTYPE)
            for c in chroma_workloads(wlo):
                cr, cd = c.generate()
                self.chroma_np.append((cr, cd))
                chroma_dev.append((torch.from_numpy(cr.reshape(-1).view(np.uint8)).to(ctx.dev),
                                   torch.from_numpy(cd.reshape(-1).view(np.uint8)).to(ctx.dev), c))
            self._chroma_dev = chroma_dev
            self.descs = (vqx.PlaneDesc * 3)(
                vqx.PlaneDesc(self.d_ref.data_ptr(), self.d_dist.data_ptr(), w, h, stride, 0),
                *[vqx.PlaneDesc(tr.data_ptr(), td.data_ptr(), c.width, c.height,
                                c.width * c.bytes_per_sample, 0) for tr, td, c in chroma_dev])
        self.geometry = (w, h, stride, wlo.bpc, n)
        # the planes are written once, before any step: batches may start
        # reading them while the batch ahead finishes
        args = (self.d_ref.data_ptr(), self.d_dist.data_ptr(), w, h, stride, wlo.bpc, n, ctx.sh,
                vqx.VQX_SUBMIT_PLANES_READY)
        out_p, out2_p = self.out.ctypes.data, self.out2.ctypes.data
        if op == "planes420":
            descs = self.descs

            def submit_call(handle):
                return so.vqx_planes_stats_submit(descs, 3, wlo.bpc, n, ctx.sh,
                                                  vqx.VQX_SUBMIT_PLANES_READY, handle)

            def finish_call(handle):
                return so.vqx_planes_stats_finish(handle, out_p)
        else:
            sub = getattr(so, {"ordered": "vqx_plane_stats_ordered_submit"}.get(
                op, "vqx_plane_%s_submit" % op))
            fin = getattr(so, {"ordered": "vqx_plane_stats_ordered_finish"}.get(
                op, "vqx_plane_%s_finish" % op))

            def submit_call(handle):
                return sub(*args, handle)

            if op == "scores":
                def finish_call(handle):
                    return fin(handle, out_p, out2_p)
            else:
                def finish_call(handle):
                    return fin(handle, out_p)
        self._submit_call, self._finish_call = submit_call, finish_call
        self.flush = (self.rbytes.nbytes + self.dbytes.nbytes) < 2 * ctx.l2_bytes
        self.scratch = (torch.empty(2 * ctx.l2_bytes, dtype=torch.uint8, device=ctx.dev)
                        if self.flush else None)
        self._ctypes = ctypes

    @property
    def plane_bytes(self):
        return int(self.rbytes.nbytes + self.dbytes.nbytes
                   + sum(cr.nbytes + cd.nbytes for cr, cd in self.chroma_np))

    def submit(self):
        handle = self._ctypes.c_void_p()
        rc = self._submit_call(self._ctypes.byref(handle))
        if rc != 0:
            raise RuntimeError("submit: %s" % self.ctx.vqx.status_string(rc))
        return handle

    def finish(self, handle):
        rc = self._finish_call(handle)
        if rc != 0:
            raise RuntimeError("finish: %s" % self.ctx.vqx.status_string(rc))


def kernel_label(op, wlo):
    if op == "int_psnr" and wlo.bpc == 16:
        return "fused_stream_tma<16, 16, 1536, 2, DenseSource, SseSums16>"
    if op == "scores" and wlo.bpc == 16:
        return "fused_stream_tma<16, 16, 1536, 2, DenseSource, TermSums16Sse>"
    if op == "ordered" and wlo.bpc == 16 and wlo.width * wlo.height > 2 ** 21:
        return "ordered_block_sums"
    if op == "planes420":
        return "fused_stream_tma, three planes (Y, Cb, Cr) timed together"
    return KERNEL_LABEL % (wlo.bpc, wlo.bpc)


def kernel_roofline(prof, peak):
    launches = max(prof["stage1_launches"], 1)
    avg_ms = prof["stage1_ms"] / launches
    bytes_per_launch = prof["stage1_bytes"] / launches
    achieved = bytes_per_launch / (avg_ms / 1e3) / 1e9 if avg_ms > 0 else 0.0
    return avg_ms, bytes_per_launch, achieved, achieved / peak


def link_ceiling(ctx, rbytes, dbytes, repeats=5):
    """A plain copy of the batch's planes from pinned host memory to the
    device (torch copy_ on the launching stream, both planes, back to back),
    timed with CUDA events; the median of ``repeats``.  Returns GB/s."""
    torch = ctx.torch
    h = [torch.from_numpy(b).pin_memory() for b in (rbytes, dbytes)]
    d = [torch.empty(b.nbytes, dtype=torch.uint8, device=ctx.dev) for b in (rbytes, dbytes)]
    times = []
    for i in range(repeats + 1):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(ctx.stream)
        with torch.cuda.stream(ctx.stream):
            for dd, hh in zip(d, h):
                dd.copy_(hh, non_blocking=True)
        e1.record(ctx.stream)
        e1.synchronize()
        if i:  # the first copy is a warm-up
            times.append(e0.elapsed_time(e1))
    return (rbytes.nbytes + dbytes.nbytes) / (statistics.median(times) / 1e3) / 1e9


def run_ours(args, wlo):
    import ctypes

    import numpy as np

    rank, world, local = dist_env()
    ctx = BenchDevice(world, local)
    torch, vqx, so = ctx.torch, ctx.vqx, ctx.so
    b = Batch(ctx, wlo, args.op)
    n, h, w = b.ref.shape
    stride = w * wlo.bytes_per_sample

    clocks = ClockSampler(gpu_smi_id(torch, ctx.dev))
    time.sleep(0.3)
    m = b.measure(args.steps, args.warmup, args.repeats, args.min_timed_seconds, args.inst_repeats)
    time.sleep(0.2)
    clocks.stop()
    reg = m["regions"]
    value = job_throughput(world, n, args.steps, reg["median_ms"] / 1e3)

    # roofline of the fused kernel, from the events recorded inside the calls
    peak, peak_kind = measured_peak()
    avg_ms, bytes_per_launch, achieved, frac = kernel_roofline(m["prof"], peak)
    traffic = recorded_traffic(wlo.name) if args.op == "stats" else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": frac, "traffic": traffic, "peak_source": peak_kind,
                "timing": "CUDA events recorded by the library around each launch in %d "
                          "instrumented regions of the same %d steps"
                          % (max(args.inst_repeats, 1), args.steps),
                "kernel": kernel_label(args.op, wlo), "avg_launch_us": avg_ms * 1e3,
                "bytes_per_launch": bytes_per_launch,
                "stage2_avg_us": m["prof"]["stage2_ms"] / max(m["prof"]["stage1_launches"], 1) * 1e3}

    # end to end: planes in pinned host memory, copies inside the timed region
    e2e = None
    if not args.no_e2e and args.op == "stats":
        h_ref = torch.from_numpy(b.rbytes).pin_memory()
        h_dist = torch.from_numpy(b.dbytes).pin_memory()
        e2e_out = np.zeros(n, vqx.FRAME_STATS_DTYPE)
        e2e_args = (h_ref.data_ptr(), h_dist.data_ptr(), w, h, stride, wlo.bpc, n, ctx.sh,
                    e2e_out.ctypes.data)
        for _ in range(3):
            rc = so.vqx_plane_stats_host(*e2e_args)
            if rc != 0:
                raise RuntimeError("vqx_plane_stats_host: %s" % vqx.status_string(rc))
        assert e2e_out.tobytes() == b.out.tobytes(), "host-memory path disagrees with the device path"
        k = max(1, min(args.e2e_steps, args.steps))
        regions = []
        for _ in range(max(args.e2e_repeats, 1)):
            ctx.barrier()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(k):
                so.vqx_plane_stats_host(*e2e_args)
            torch.cuda.synchronize()
            regions.append(reduce_max(time.perf_counter() - t0, ctx.pg, ctx.dev))
        el = statistics.median(regions)
        e2e_value = job_throughput(world, n, k, el)
        link = link_ceiling(ctx, b.rbytes, b.dbytes)
        e2e_gbs = e2e_value / world * wlo.pair_bytes / 1e9
        e2e = {"value": e2e_value, "unit": UNIT, "steps": k, "repeats": len(regions),
               "statistic": "median of the repeated regions (wall clock, blocking calls)",
               "value_min": job_throughput(world, n, k, max(regions)),
               "value_max": job_throughput(world, n, k, min(regions)),
               "h2d_bytes_per_step": int(b.rbytes.nbytes + b.dbytes.nbytes),
               "d2h_bytes_per_step": int(n * ctypes.sizeof(ctypes.c_uint64) * 6),
               "api": "vqx_plane_stats_host (pinned host planes)",
               "h2d_gbs": e2e_gbs, "link_gbs": link, "link_frac": e2e_gbs / link,
               "link": "a plain pinned-host-to-device copy_ of the same planes on the same "
                       "stream, CUDA events, median of 5"}
        del h_ref, h_dist

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cores = host_cores()
        sub = list(range(min(n, cores)))
        ex = [(cr[sub], cd[sub]) for cr, cd in b.chroma_np]
        rate, pairs, el = time_oracle(wlo, b.ref[sub], b.dist[sub], args.cpu_seconds, cores,
                                      op=args.op, extra=ex)
        rate1, pairs1, el1 = time_oracle(wlo, b.ref[:1], b.dist[:1], min(args.cpu_seconds, 4.0), 1,
                                         op=args.op, extra=[(cr[:1], cd[:1]) for cr, cd in b.chroma_np])
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "%.1f frame pairs of %s (whole frames, one per thread) in %.1f s"
                         % (pairs, wlo.name, el),
               "single_core": {"value": rate1, "sample": "%.1f frame pairs on one thread in %.1f s"
                                                         % (pairs1, el1)}}

    # the other configurations of the measured set, timed the same way after
    # the headline (each batch placed on the device in turn)
    configs = None
    if args.op == "stats" and not args.no_configs and args.workload in (None, wlo.name):
        from exact_full_reference_gb300 import workloads as wl

        planes_bytes = b.plane_bytes
        del b
        torch.cuda.empty_cache()
        configs = {}
        for name in wl.BENCH_CONFIGS:
            if name == wlo.name:
                continue
            cw = wl.WORKLOADS[name]
            cb = Batch(ctx, cw, "stats")
            cm = cb.measure(args.steps, args.warmup, args.repeats, args.config_seconds,
                            args.inst_repeats)
            cr = cm["regions"]
            c_ms, c_bytes, c_ach, c_frac = kernel_roofline(cm["prof"], peak)
            step_gbs = cw.pair_bytes * cw.n_frames / (cr["ms_per_step"] / 1e3) / 1e9
            configs[name] = {
                "value": job_throughput(world, cw.n_frames, args.steps, cr["median_ms"] / 1e3),
                "unit": UNIT, "ms_per_step": cr["ms_per_step"],
                "us_per_call": cr["ms_per_step"] * 1e3,
                "repeats": cr["repeats"], "min_ms": cr["min_ms"], "max_ms": cr["max_ms"],
                "step_gbs": step_gbs, "step_frac": step_gbs / peak,
                "kernel": KERNEL_LABEL % (cw.bpc, cw.bpc), "kernel_avg_launch_us": c_ms * 1e3,
                "kernel_frac": c_frac,
                "l2": ("batch smaller than twice the L2: L2 overwritten before every step, steps "
                       "timed one by one, flush excluded" if cb.flush else
                       "inputs %.2f GB per step, larger than the L2; no flush, steps pipelined"
                       % (cb.plane_bytes / 1e9)),
                "gpu_launches_per_region": int(cm["counted"]["kernel_launches"] // max(cm["reps"], 1)),
            }
            del cb
            torch.cuda.empty_cache()
    else:
        planes_bytes = b.plane_bytes

    if rank == 0:
        pipeline = ("batch i + 1 submitted before batch i is finished (%s_submit with "
                    "VQX_SUBMIT_PLANES_READY / _finish)" % OP_API[args.op])
        if args.op == "planes420":
            pipeline += "; Y, Cb, Cr"
        is_flush = (n * wlo.pair_bytes) < 2 * ctx.l2_bytes
        line = {
            "metric": metric_for(args.op, wlo),
            "value": value,
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": max(args.warmup, 3),
            "ms_per_step": reg["ms_per_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("u%d samples, %s" % (8 if wlo.bpc == 8 else 16,
                      "f32 terms, u64 sums" if args.op in ("stats", "ordered", "planes420")
                      else "f32 terms and exact integer squares, u64 sums" if args.op == "scores"
                      else "exact integer squares, u64 sums")),
            "data": "synthetic",
            "hbm_gbs": value * wlo.pair_bytes * (1.5 if args.op == "planes420" else 1.0) / 1e9 / world,
            "timing": {"repeats": reg["repeats"], "statistic": "median of the repeated regions",
                       "region_ms": {k: reg[k] for k in ("median_ms", "min_ms", "p10_ms", "p90_ms",
                                                        "max_ms")},
                       "value_min": job_throughput(world, n, args.steps, reg["max_ms"] / 1e3),
                       "value_max": job_throughput(world, n, args.steps, reg["min_ms"] / 1e3)},
            "config": {"workload": wlo.name, "frames_per_gpu": n, "width": w, "height": h,
                       "bpc": wlo.bpc, "batch_bytes": planes_bytes,
                       "l2": "inputs %.2f GB per step, larger than the 129 MB L2; no flush"
                             % (planes_bytes / 1e9),
                       "pipeline": pipeline,
                       "parallelism": "frames independent per GPU" if world > 1 else "1 GPU"},
            "e2e": e2e,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "clocks": clocks.summary(m["t0"], m["t1"]),
            "gpu_launches": int(m["counted"]["kernel_launches"] // max(m["reps"], 1)),
            "gpu_launches_all_repeats": int(m["counted"]["kernel_launches"]),
        }
        if is_flush:
            line["config"]["l2"] = ("batch smaller than twice the L2: L2 overwritten (%d MB) before "
                                    "every step, steps timed one by one, flush excluded"
                                    % (2 * ctx.l2_bytes >> 20))
            line["config"]["pipeline"] = "none (each step timed on its own after the flush)"
        if args.op == "planes420":
            line["config"]["planes"] = "Y %dx%d, Cb and Cr %dx%d per frame" % (
                w, h, max(1, w // 2), max(1, h // 2))
        if configs is not None:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    if ctx.pg is not None:
        ctx.pg.destroy_process_group()
    return 0


# ---------------------------------------------------------------- psnr_hvs plane sums
HVS_UNIT = "planes/s"


def hvs_metric(hw):
    return "planes/s and HBM GB/s (psnr_hvs plane sums), %d terms a plane (%dx%d luma), 1 GB300" % (
        hw.n_terms, hw.width, hw.height)


def time_oracle_hvs(hw, terms, seconds, cores, n_terms=None):
    """The oracle's plane sums of ``terms`` (one plane, or its first
    ``n_terms`` terms, per thread) until ``seconds`` have passed.  Returns
    (planes/s, planes done, elapsed s)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    orc = oracle.load()
    n = terms.shape[1] if n_terms is None else n_terms

    def one(k):
        orc.hvs(terms[k % terms.shape[0], :n], hw.bpc)
        return n

    done = 0
    k = 0
    t0 = time.perf_counter()
    while True:
        with ThreadPoolExecutor(cores) as ex:
            done += sum(ex.map(one, range(k, k + cores)))
        k += cores
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    planes = done / terms.shape[1]
    return planes / el, planes, el


def run_hvs_reference(args, hw):
    rank, _, _ = dist_env()
    if rank != 0:
        return 0
    cores = host_cores()
    terms = hw.generate(range(min(hw.n_planes, max(cores, 1))))
    per_step_s = min(0.5, 120.0 / max(args.steps + args.warmup, 1))
    rate, _, _ = time_oracle_hvs(hw, terms[:1], 0.0, 1, n_terms=min(hw.n_terms, 1 << 20))
    n = int(max(1, min(hw.n_terms, rate * hw.n_terms * per_step_s)))
    for _ in range(args.warmup):
        time_oracle_hvs(hw, terms, 0.0, cores, n_terms=n)
    t0 = time.perf_counter()
    planes = 0.0
    for _ in range(args.steps):
        _, p, _ = time_oracle_hvs(hw, terms, 0.0, cores, n_terms=n)
        planes += p
    el = time.perf_counter() - t0
    value = planes / el
    line = {
        "impl": "reference", "metric": hvs_metric(hw), "value": value, "unit": HVS_UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": hw.name, "planes": hw.n_planes, "terms_per_plane": hw.n_terms,
                   "oracle": "plain C, one float running sum per plane"},
        "cpu_baseline": {"value": value, "unit": HVS_UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d planes' first %d terms per step, one plane per thread"
                                   % (cores, n)},
        "e2e": {"value": value, "unit": HVS_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class HvsBatch(Stepper):
    """A batch of psnr_hvs term planes on the device and its submit / finish
    calls (vqx_psnr_hvs_sum_submit / _finish)."""

    def __init__(self, ctx, hw):
        import ctypes

        import numpy as np

        torch, vqx = ctx.torch, ctx.vqx
        self.ctx, self.hw = ctx, hw
        self.terms = hw.generate()
        self.n_planes, self.n_terms = self.terms.shape
        self.d_terms = torch.from_numpy(self.terms).to(ctx.dev)
        torch.cuda.synchronize()
        self.out = np.zeros(self.n_planes, vqx.HVS_PLANE_DTYPE)
        self._ctypes = ctypes
        if self.terms.nbytes < 2 * ctx.l2_bytes:
            raise SystemExit("psnr_hvs bench batches must be larger than twice the L2")

    def submit(self, ptr=None):
        vqx = self.ctx.vqx
        handle = self._ctypes.c_void_p()
        rc = self.ctx.so.vqx_psnr_hvs_sum_submit(
            ptr or self.d_terms.data_ptr(), self.n_terms, self.n_terms, self.n_planes, self.hw.bpc,
            self.ctx.sh, vqx.VQX_SUBMIT_PLANES_READY if ptr is None else 0, self._ctypes.byref(handle))
        if rc != 0:
            raise RuntimeError("submit: %s" % vqx.status_string(rc))
        return handle

    def finish(self, handle):
        rc = self.ctx.so.vqx_psnr_hvs_sum_finish(handle, self.out.ctypes.data)
        if rc != 0:
            raise RuntimeError("finish: %s" % self.ctx.vqx.status_string(rc))


def run_hvs(args, hw):
    """One step = one batch of term planes resident in HBM through
    vqx_psnr_hvs_sum_submit + _finish (tables, walk, read-back, score),
    pipelined one deep like the plane statistics, timed the same way."""
    rank, world, local = dist_env()
    ctx = BenchDevice(world, local)
    torch = ctx.torch
    b = HvsBatch(ctx, hw)
    n_planes, n_terms = b.n_planes, b.n_terms

    clocks = ClockSampler(gpu_smi_id(torch, ctx.dev))
    time.sleep(0.3)
    m = b.measure(args.steps, args.warmup, args.repeats, args.min_timed_seconds, args.inst_repeats)
    time.sleep(0.2)
    clocks.stop()
    reg = m["regions"]
    value = job_throughput(world, n_planes, args.steps, reg["median_ms"] / 1e3)
    peak, peak_kind = measured_peak()
    avg_ms, bytes_per_launch, achieved, frac = kernel_roofline(m["prof"], peak)
    launches = max(m["prof"]["stage1_launches"], 1)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": frac, "traffic": None, "peak_source": peak_kind,
                "timing": "CUDA events recorded by the library around each launch in %d "
                          "instrumented regions of the same %d steps"
                          % (max(args.inst_repeats, 1), args.steps),
                "kernel": "hvs_tables_tma", "avg_launch_us": avg_ms * 1e3,
                "bytes_per_launch": bytes_per_launch,
                "walk_avg_us": m["prof"]["stage2_ms"] / launches * 1e3}

    e2e = None
    if not args.no_e2e:
        h_terms = torch.from_numpy(b.terms).pin_memory()
        d_e2e = torch.empty_like(b.d_terms)
        k = max(1, min(args.e2e_steps, args.steps))
        regions = []
        for _ in range(max(args.e2e_repeats, 1)):
            ctx.barrier()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(k):
                with torch.cuda.stream(ctx.stream):
                    d_e2e.copy_(h_terms, non_blocking=True)
                b.finish(b.submit(d_e2e.data_ptr()))
            torch.cuda.synchronize()
            regions.append(reduce_max(time.perf_counter() - t0, ctx.pg, ctx.dev))
        el = statistics.median(regions)
        e2e = {"value": job_throughput(world, n_planes, k, el), "unit": HVS_UNIT, "steps": k,
               "repeats": len(regions),
               "statistic": "median of the repeated regions (wall clock, blocking calls)",
               "h2d_bytes_per_step": int(b.terms.nbytes),
               "d2h_bytes_per_step": int(n_planes * 16),
               "api": "copy of pinned host terms on the call's stream, then vqx_psnr_hvs_sum_submit / _finish"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cores = host_cores()
        sub = b.terms[: min(n_planes, cores)]
        rate, planes, el = time_oracle_hvs(hw, sub, args.cpu_seconds, cores)
        cpu = {"value": rate, "unit": HVS_UNIT, "cores": cores, "kind": "oracle",
               "sample": "%.1f whole planes of %s (one per thread) in %.1f s" % (planes, hw.name, el)}

    if rank == 0:
        line = {
            "metric": hvs_metric(hw), "value": value, "unit": HVS_UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": reg["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "hbm_gbs": value * 4 * n_terms / 1e9 / world,
            "timing": {"repeats": reg["repeats"], "statistic": "median of the repeated regions",
                       "region_ms": {k: reg[k] for k in ("median_ms", "min_ms", "p10_ms", "p90_ms",
                                                        "max_ms")}},
            "config": {"workload": hw.name, "planes_per_gpu": n_planes, "terms_per_plane": n_terms,
                       "bpc": hw.bpc, "batch_bytes": int(b.terms.nbytes),
                       "l2": "terms %.2f GB per step, larger than the 129 MB L2; no flush"
                             % (b.terms.nbytes / 1e9),
                       "pipeline": "batch i + 1 submitted before batch i is finished "
                                   "(vqx_psnr_hvs_sum_submit with VQX_SUBMIT_PLANES_READY / _finish)",
                       "parallelism": "planes independent per GPU" if world > 1 else "1 GPU"},
            "e2e": e2e, "roofline": roofline, "cpu_baseline": cpu,
            "clocks": clocks.summary(m["t0"], m["t1"]),
            "gpu_launches": int(m["counted"]["kernel_launches"] // max(m["reps"], 1)),
            "gpu_launches_all_repeats": int(m["counted"]["kernel_launches"]),
            "replayed_leaves_max": int(b.out["replayed_leaves"].max()),
        }
        print(json.dumps(line), flush=True)
    if ctx.pg is not None:
        ctx.pg.destroy_process_group()
    return 0


def main():
    args = parse_args()
    from exact_full_reference_gb300 import workloads as wl

    if args.op == "hvs":
        hw = wl.HVS_WORKLOADS[args.workload or wl.HVS_HEADLINE]
        return run_hvs_reference(args, hw) if args.impl == "reference" else run_hvs(args, hw)
    wlo = wl.WORKLOADS[args.workload or wl.HEADLINE]
    if args.record_traffic:
        return write_traffic_record(args.record_traffic, wlo)
    if args.impl == "reference":
        return run_reference(args, wlo)
    return run_ours(args, wlo)


if __name__ == "__main__":
    sys.exit(main())
