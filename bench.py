#!/usr/bin/env python3
"""Benchmark: TMA tiled round trip of a 16384x16384 fp16 tensor (512 MiB) on GB300.

One step = one pass of the whole hot path over the workload: every box of the
source (128x64 with 128-byte swizzle by default; 64x256 unswizzled with --box
64x256) is loaded by the tensor-map engine into a shared-memory stage
(arrive.expect_tx + cp.async.bulk.tensor) and stored to the destination
(cp.async.bulk.tensor store + bulk group), i.e. one atb_tile_roundtrip launch
with the library's default pipeline shape.  The maps are encoded once per
tensor, outside the device-timed region.

Prints ONE JSON line (rank 0):
  value      HBM GB/s moved (bytes read + bytes written) / device time, inputs
             resident in HBM, timed with CUDA events on the launching stream
  e2e        the same metric through the public call with HOST buffers:
             pinned H2D of the input, encode, round trip, D2H of the output
  roofline   the round-trip kernel against the measured copy bandwidth
  cpu_baseline  the plain CPU oracle on one host core, and (all_cores) the
             same round trip split over every host core
  sweep / ablations  stage sweep and the thread-issued copies beside it
  workloads  the smaller workloads, L2-warm and after an L2 flush

``--impl reference`` times the oracle instead (the reference arm).
Inputs (512 MiB in + 512 MiB out) exceed the 129 MB L2, so no flush is needed.
Multi-GPU (torchrun): every rank moves its own full replica; no collective on
the data path; value = bytes of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

NOMINAL_HBM_GBS = 8000.0
REF_BOX_BUDGET = 250_000  # reference arm: boxes over the whole run (~0.2 ms each)
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "tile_pipeline_roundtrip_f16_16384.md")
KERNEL_SOURCES = [os.path.join(ROOT, "async_bulk_tensor_gb300", "csrc", f) for f in ("pipeline.cu", "ptx.cuh")]


# ---------------------------------------------------------------------------
# distributed plumbing (timing only; the data path has no collective)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def init_dist(world_size: int, backend: str):
    import torch.distributed as dist

    if world_size > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world_size > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(dist, local_seconds: float, local_units: float, device=None):
    """Whole-job throughput: units of all ranks / the slowest rank's time."""
    seconds = max_over_ranks(dist, local_seconds, device)
    units = local_units
    if dist is not None:
        import torch

        t = torch.tensor([local_units], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        units = float(t.item())
    return units, seconds


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    def __init__(self, gpu_id: str, period_ms: int = 100):
        self.proc = None
        self.cmd = ["nvidia-smi", f"--query-gpu={','.join(CLOCK_FIELDS)}", "--format=csv,noheader,nounits",
                    "-lms", str(period_ms), "-i", str(gpu_id)]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        mhz, max_mhz, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < len(CLOCK_FIELDS):
                continue
            try:
                mhz.append(float(parts[1]))
                max_mhz = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max_mhz,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ---------------------------------------------------------------------------
# peaks and the committed ncu traffic figure
# ---------------------------------------------------------------------------
def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic():
    """(bytes per full-workload launch, note) from the committed ncu summary, or
    (None, why) when it is missing or the kernel source changed since."""
    try:
        text = open(TRAFFIC_PROFILE).read()
    except OSError:
        return None, "no committed ncu summary"
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    if not m or not h:
        return None, "summary lacks traffic or source hash"
    if h.group(1) != kernel_source_hash():
        return None, "kernel changed since the ncu capture"
    return int(m.group(1)), "ncu dram__bytes_read.sum + dram__bytes_write.sum of one full-size launch"


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def time_launches(torch, stream, fn, steps: int, warmup: int, dist=None, device=None) -> float:
    """Seconds for `steps` calls of fn() on `stream` (CUDA events), after warm-up."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
    stream.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            fn()
        end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    barrier(dist)
    return start.elapsed_time(end) / 1e3


def single_steps(torch, stream, fn, n: int):
    """Milliseconds of n steps, each bracketed by its own pair of events."""
    out = []
    with torch.cuda.stream(stream):
        for _ in range(n):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            out.append(a.elapsed_time(b))
    return out


def run_gpu(args):
    import numpy as np
    import torch

    import async_bulk_tensor_gb300 as atb
    import datagen

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = init_dist(world, "nccl")
    atb.init_device()
    atb.device_status()
    stream = torch.cuda.Stream(device=device)

    w = datagen.C5A if args.box == "64x256" else datagen.C5B
    launch = dict(stages=args.stages, ctas_per_sm=args.ctas_per_sm, store_groups=args.store_groups,
                  poll_suspend_ns=args.poll_suspend_ns, consumer=args.consumer)
    src_h = datagen.storage(w)
    nbytes = w.storage_bytes
    src = torch.from_numpy(src_h).to(device)
    dst = torch.zeros(nbytes, dtype=torch.uint8, device=device)
    ms = atb.encode_tiled(w.dtype, src, w.dims, w.strides, w.box, w.swizzle)
    md = atb.encode_tiled(w.dtype, dst, w.dims, w.strides, w.box, w.swizzle)
    tiles = atb.grid_tiles(ms)
    bytes_per_step = 2 * nbytes  # every element read once and written once (all boxes in bounds)

    def step():
        atb.tile_roundtrip(ms, md, stream=stream, **launch)

    # correctness of the timed configuration before timing it
    with torch.cuda.stream(stream):
        step()
    launch_shape = atb.last_launch()  # what the library resolved for the timed launches
    stream.synchronize()
    atb.check_device(stream)
    verified = bool(torch.equal(src, dst))
    if not verified:
        raise SystemExit("round trip output differs from its input; refusing to time it")
    dst.zero_()

    visible = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    gpu_id = visible[local_rank] if local_rank < len(visible) else str(local_rank)
    with ClockSampler(gpu_id) as clocks:
        seconds = time_launches(torch, stream, step, args.steps, args.warmup, dist, device)
    atb.check_device(stream)
    per_step = single_steps(torch, stream, step, 20)
    units, max_seconds = aggregate(dist, seconds, float(bytes_per_step) * args.steps, device)
    value = units / max_seconds / 1e9
    ms_per_step = max_seconds / args.steps * 1e3
    kernel_avg_s = seconds / args.steps  # one launch per step: the launch's own duration
    achieved = bytes_per_step / kernel_avg_s / 1e9

    result = {"metric": "TMA tiled round trip HBM GB/s (read+write)", "value": round(value, 1), "unit": "GB/s",
              "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
              "data": "synthetic (seeded normal(0,1) fp16)"}
    result["config"] = {
        "workload": w.name, "tensor": "16384x16384 fp16 row-major (512 MiB)",
        "box": args.box, "swizzle": w.swizzle, "tiles_per_step": tiles,
        "stages": args.stages or "library default",
        "ctas_per_sm": args.ctas_per_sm or "library default",
        "store_groups": args.store_groups or "library default",
        "launch": "programmatic dependent launch",
        "consumer": ("library default (one-thread drain; for 4-32 KiB stages its own ring: 64 KiB of stages per SM "
                     "for boxes in load plus store groups, each stage freed before the next store)"
                     if args.consumer == "auto" else args.consumer),
        "launch_shape": launch_shape,
        "parallelism": f"replicas x{world}",
        "l2": "inputs larger than L2 (512 MiB read + 512 MiB written per step); no flush",
    }
    result["tiles_per_s"] = round(tiles * args.steps * world / max_seconds, 1)
    result["single_steps"] = {"n": len(per_step), "ms_median": round(statistics.median(per_step), 5),
                              "ms_best": round(min(per_step), 5),
                              "GBps_median": round(bytes_per_step / statistics.median(per_step) / 1e6, 1),
                              "GBps_best": round(bytes_per_step / min(per_step) / 1e6, 1),
                              "note": "each step timed alone between events (launch gap included)"}
    peak, peak_kind = hbm_peak()
    traffic, traffic_note = committed_traffic()
    result["roofline"] = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                          "frac": round(achieved / peak, 4), "traffic": traffic,
                          "peak_source": f"{peak_kind} hbm_gbs (copy, read+write)",
                          "traffic_note": traffic_note, "frac_of_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4)}
    result["gpu_launches"] = args.steps
    result["clocks"] = clocks.summary()

    if rank == 0 and not args.no_extras:
        result["sweep"] = stage_sweep(torch, atb, datagen, device, stream, src, dst, args)
        result["ablations"] = ablations(torch, atb, device, stream, src, dst, nbytes, args)
        atb.check_device(stream)
        result["workloads"] = workload_lines(torch, atb, datagen, device, stream, args)
    if not args.no_e2e:
        result["e2e"] = end_to_end(torch, atb, w, device, stream, src_h, nbytes, bytes_per_step, args, dist)
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(w, src_h)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


SMEM_PER_SM = 228 * 1024  # GB300: shared memory one SM can hold for resident CTAs


def stage_sweep(torch, atb, datagen, device, stream, src, dst, args):
    """Workload 5 over ring shapes.  Every cell names its launch shape: stages,
    CTAs per SM, store groups in flight and KiB of stages per SM.  Rows:
      default_rule   stages 2/3/4/6/8, CTAs per SM from the library's rule
                     (about 96 KiB of stages per SM), two store groups;
      fixed_96KiB    about 96 KiB of stages per SM, split between more stages
                     and fewer CTAs or the reverse;
      ctas_1, ctas_2 CTAs per SM held at one or two while the ring deepens;
      drain_release_before_store
                     the one-thread drain freeing each stage before the next
                     store, one CTA per SM, over stages x store groups (the
                     library's own drain ring is one of these cells).
    Every cell but the last row's takes the consumer the library picks for an
    explicit shape.  A shape that does not fit one CTA's shared memory is
    reported as infeasible."""
    out = {}
    steps = max(50, min(400, args.steps // 10))
    for w, box in ((datagen.C5A, "64x256"), (datagen.C5B, "128x64_sw128")):
        ms = atb.encode_tiled(w.dtype, src, w.dims, w.strides, w.box, w.swizzle)
        md = atb.encode_tiled(w.dtype, dst, w.dims, w.strides, w.box, w.swizzle)
        stage_kib = atb.box_bytes(ms) // 1024

        def cell(stages, per_sm, groups=2, **kw):
            try:
                smem = atb.pipeline_smem_bytes(ms, stages)
            except atb.AtbError as e:
                return f"infeasible: {e.name}"
            if smem * per_sm > SMEM_PER_SM:
                return f"infeasible: {per_sm} CTAs of {smem} bytes exceed the SM's shared memory"
            g = min(groups, stages)
            sec = time_launches(torch, stream, lambda: atb.tile_roundtrip(
                ms, md, stream=stream, stages=stages, ctas_per_sm=per_sm, store_groups=g, **kw), steps, 5)
            return {"GBps": round(2 * w.storage_bytes * steps / sec / 1e9, 1), "stages": stages, "ctas_per_sm": per_sm,
                    "store_groups": g, "kib_per_sm": stages * stage_kib * per_sm}

        rows = {"default_rule": {}, "fixed_96KiB": {}, "ctas_1": {}, "ctas_2": {}}
        for stages in (2, 3, 4, 6, 8):
            rule = max(1, min(8, (96 * 1024) // (stages * atb.box_bytes(ms))))
            rows["default_rule"][f"s{stages}"] = cell(stages, rule)
        for stages in (1, 2, 3, 6):
            per_sm = (96 * 1024) // (stages * atb.box_bytes(ms))
            if per_sm >= 1 and stages * per_sm * atb.box_bytes(ms) == 96 * 1024:
                rows["fixed_96KiB"][f"s{stages}c{per_sm}"] = cell(stages, per_sm)
        for per_sm, key in ((1, "ctas_1"), (2, "ctas_2")):
            for stages in (2, 3, 4, 6, 8, 12):
                rows[key][f"s{stages}"] = cell(stages, per_sm)
        # stages - store groups = stages holding boxes being loaded or landed
        before = ((3, 1), (4, 2), (5, 3), (4, 1), (5, 1)) if stage_kib >= 32 else \
            ((5, 1), (6, 2), (7, 3), (8, 4), (10, 6), (6, 3), (7, 4), (7, 2), (8, 3))
        rows["drain_release_before_store"] = {
            f"s{st}g{g}": cell(st, 1, g, consumer="drain", release="before_store") for st, g in before}
        out[box] = rows
        extra = {}
        for promo in ("128B", "256B"):  # L2 promotion of the source map, default pipeline
            mp = atb.encode_tiled(w.dtype, src, w.dims, w.strides, w.box, w.swizzle, promo)
            sec = time_launches(torch, stream, lambda: atb.tile_roundtrip(mp, md, stream=stream), steps, 5)
            extra[f"l2promotion{promo}"] = round(2 * w.storage_bytes * steps / sec / 1e9, 1)
        for name, kw in (("without_pdl", dict(pdl=False)), ("ring_check", dict(checks=atb.CHECK_RING)),
                         ("consumer_drain", dict(consumer="drain")), ("consumer_warp", dict(consumer="warp")),
                         ("release_after_store", dict(consumer="drain", release="after_store")),
                         ("release_before_store", dict(consumer="drain", release="before_store"))):
            sec = time_launches(torch, stream, lambda: atb.tile_roundtrip(ms, md, stream=stream, **kw), steps, 5)
            extra[name] = round(2 * w.storage_bytes * steps / sec / 1e9, 1)
        out[box]["library_default_variants"] = extra
    return out


def box_inbound_bytes(dims, box, esize, coords):
    """Bytes of each listed box that fall inside the tensor (clipped volume)."""
    import numpy as np

    c = np.asarray(coords, dtype=np.int64)
    vol = np.ones(len(c), dtype=np.int64)
    for d in range(len(dims)):
        lo = np.maximum(c[:, d], 0)
        hi = np.minimum(c[:, d] + box[d], dims[d])
        vol *= np.maximum(hi - lo, 0)
    return int(vol.sum()) * esize


def workload_lines(torch, atb, datagen, device, stream, args):
    """The smaller workloads, timed L2-warm (back to back) and after an L2 flush
    (a read of a 512 MiB scratch buffer before every timed launch, outside the
    events; a read leaves no dirty lines for the timed launch to write back)."""
    import numpy as np

    flush = torch.ones(512 << 20, dtype=torch.uint8, device=device)
    flush64 = flush.view(torch.int64)
    out = {}

    def timed(fn, reps_warm, reps_cold):
        warm = time_launches(torch, stream, fn, reps_warm, 5) / reps_warm
        cold = 0.0
        with torch.cuda.stream(stream):
            for i in range(reps_cold):
                flush_sum = flush64.sum()  # reads 512 MiB: evicts the workload, leaves only clean lines
                del flush_sum
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                b.synchronize()
                cold += a.elapsed_time(b) / 1e3
        return warm, cold / reps_cold

    def line(bytes_moved, boxes, warm, cold):
        return {"bytes_per_launch": bytes_moved, "boxes": boxes,
                "l2_warm": {"us": round(warm * 1e6, 2), "GBps": round(bytes_moved / warm / 1e9, 1)},
                "l2_flushed": {"us": round(cold * 1e6, 2), "GBps": round(bytes_moved / cold / 1e9, 1)}}

    def dev_bytes(h):
        return torch.from_numpy(np.ascontiguousarray(h)).to(device)

    # 1: one 64x64 fp32 tile, one CTA, one stage
    w = datagen.C1
    src, dst = dev_bytes(datagen.storage(w)), torch.zeros(w.storage_bytes, dtype=torch.uint8, device=device)
    ms = atb.encode_tiled(w.dtype, src, w.dims, w.strides, w.box, w.swizzle)
    md = atb.encode_tiled(w.dtype, dst, w.dims, w.strides, w.box, w.swizzle)
    warm, cold = timed(lambda: atb.tile_roundtrip(ms, md, stream=stream, stages=1, ctas=1), 2000, 50)
    out[w.name] = line(2 * 16384, 1, warm, cold)

    # 2: 924 boxes of 64x256 fp16, 132 CTAs each walking its row strip
    w = datagen.C2
    src, dst = dev_bytes(datagen.storage(w)), torch.zeros(w.storage_bytes, dtype=torch.uint8, device=device)
    ms = atb.encode_tiled(w.dtype, src, w.dims, w.strides, w.box, w.swizzle)
    md = atb.encode_tiled(w.dtype, dst, w.dims, w.strides, w.box, w.swizzle)
    warm, cold = timed(lambda: atb.tile_roundtrip(ms, md, stream=stream, ctas=w.ctas, schedule=w.schedule),
                       500, 30)
    out[w.name] = line(2 * w.storage_bytes, 924, warm, cold)
    lib_default_warm, lib_default_cold = timed(lambda: atb.tile_roundtrip(ms, md, stream=stream), 500, 30)
    out[w.name + "_library_default_grid"] = line(2 * w.storage_bytes, 924, lib_default_warm, lib_default_cold)

    # 3: ragged bf16 full grid gathered into packed swizzled images
    w = datagen.C3
    src = dev_bytes(datagen.storage(w))
    ms = atb.encode_tiled(w.dtype, src, w.dims, w.strides, w.box, w.swizzle)
    n = atb.grid_tiles(ms)
    packed = torch.empty(n * atb.box_bytes(ms), dtype=torch.uint8, device=device)
    warm, cold = timed(lambda: atb.tile_load(ms, None, 0, packed, stream=stream), 500, 30)
    out[w.name] = line(10000 * 3000 * 2 + n * atb.box_bytes(ms), n, warm, cold)

    # 4: 4096 random boxes of a permuted 3-D fp32 view: gather, then store.  The
    # workload's origins are uniform over every element offset (three in four
    # boxes start off the 16-byte grid along x); the same count of origins drawn
    # on the 16-byte grid is timed beside them.
    w = datagen.C4
    src = dev_bytes(datagen.storage(w))
    ms = atb.encode_tiled(w.dtype, src, w.dims, w.strides, w.box, w.swizzle)
    bb = atb.box_bytes(ms)
    fresh = torch.full((w.storage_bytes,), 0xFF, dtype=torch.uint8, device=device)
    mf = atb.encode_tiled(w.dtype, fresh, w.dims, w.strides, w.box, w.swizzle)
    for tag, coords_h in (("", datagen.workload_coords(w)),
                          ("_grid16B_origins", datagen.random_box_origins(w.dims, w.box, w.esize, w.n_random,
                                                                         w.seed + 1000, align_bytes=16))):
        coords = dev_bytes(coords_h.view(np.uint8))
        n = len(coords_h)
        packed = torch.empty(n * bb, dtype=torch.uint8, device=device)
        inb = box_inbound_bytes(w.dims, w.box, w.esize, coords_h)
        warm, cold = timed(lambda: atb.tile_load(ms, coords, n, packed, stream=stream), 500, 30)
        out[w.name + tag + "_load"] = line(inb + n * bb, n, warm, cold)
        if not tag:
            for pf in (4, 16):
                warm, cold = timed(lambda: atb.tile_load(ms, coords, n, packed, stream=stream, prefetch_boxes=pf),
                                   500, 30)
                out[w.name + f"_load_prefetch{pf}"] = line(inb + n * bb, n, warm, cold)
        warm, cold = timed(lambda: atb.tile_store(mf, coords, n, packed, stream=stream), 500, 30)
        out[w.name + tag + "_store"] = line(n * bb + inb, n, warm, cold)
        warm, cold = timed(lambda: atb.tile_roundtrip(ms, mf, coords, n, stream=stream), 500, 30)
        out[w.name + tag + "_roundtrip"] = line(2 * inb, n, warm, cold)
        del packed
    fits = fixed_cost_fits(torch, atb, datagen, device, stream, timed, dev_bytes, src, ms, mf)
    out["fixed_cost_fits"] = fits
    # every short line's fraction of the measured copy peak after an L2 flush, whole and net of the fixed
    # cost T0 fitted for its kind of launch
    peak, _ = hbm_peak()
    for name, fit_key in ((datagen.C2.name, "c2_round_trip"), (datagen.C2.name + "_library_default_grid",
                                                               "c2_round_trip"),
                          (datagen.C3.name, "c3_gather"), (w.name + "_load", "c4_gather"),
                          (w.name + "_store", "c4_store"), (w.name + "_roundtrip", "c4_roundtrip"),
                          (w.name + "_grid16B_origins_load", "c4_gather"),
                          (w.name + "_grid16B_origins_store", "c4_store"),
                          (w.name + "_grid16B_origins_roundtrip", "c4_roundtrip")):
        ln, t0 = out[name], fits[fit_key]["fixed_us"] * 1e-6
        cold = ln["l2_flushed"]["us"] * 1e-6
        ln["l2_flushed"]["frac_of_peak"] = round(ln["bytes_per_launch"] / cold / 1e9 / peak, 3)
        ln["l2_flushed"]["net_of_fixed"] = {"fixed_us": fits[fit_key]["fixed_us"], "fit": fit_key,
                                            "frac_of_peak": round(ln["bytes_per_launch"] / max(cold - t0, 1e-9)
                                                                  / 1e9 / peak, 3)}
    del src, fresh

    # the fp32 update between load and store: 16384 x 8192 fp32 (512 MiB), box 32x128, 128B swizzle
    rows, cols = 8192, 16384
    a32 = torch.empty(rows * cols * 4, dtype=torch.uint8, device=device)
    a32.view(torch.float32).normal_()
    b32 = torch.empty_like(a32)
    ma = atb.encode_tiled("f32", a32, (cols, rows), (4, cols * 4), (32, 128), "128B")
    mb = atb.encode_tiled("f32", b32, (cols, rows), (4, cols * 4), (32, 128), "128B")
    warm, cold = timed(lambda: atb.tile_roundtrip_add_f32(ma, mb, 1.0, stream=stream), 300, 10)
    out["f32_16384x8192_add1_roundtrip"] = line(2 * rows * cols * 4, atb.grid_tiles(ma), warm, cold)
    warm, cold = timed(lambda: atb.tile_roundtrip(ma, mb, stream=stream), 300, 10)
    out["f32_16384x8192_plain_roundtrip"] = line(2 * rows * cols * 4, atb.grid_tiles(ma), warm, cold)
    # traversal step 2 along rows: every other row of each 64-row box, gathered to packed images
    ms2 = atb.encode_tiled("f32", a32, (cols, rows), (4, cols * 4), (32, 64), "128B", elem_strides=(1, 2))
    bb2 = atb.box_bytes(ms2)
    n2 = atb.grid_tiles(ms2)
    packed2 = torch.empty(n2 * bb2, dtype=torch.uint8, device=device)
    warm, cold = timed(lambda: atb.tile_load(ms2, None, 0, packed2, stream=stream), 300, 10)
    out["f32_16384x8192_step2_rows_gather"] = line(2 * n2 * bb2, n2, warm, cold)
    del packed2
    # the same 32x128 boxes given as a coordinate list (the grid's own origins, x fastest): the
    # listed gather and the listed round trip read every origin from the list
    gx, gy = np.meshgrid(np.arange(cols // 32, dtype=np.int32) * 32, np.arange(rows // 128, dtype=np.int32) * 128)
    listed = torch.from_numpy(np.stack([gx.ravel(), gy.ravel()], 1).reshape(-1).copy()).to(device)
    nl = listed.numel() // 2
    packed_l = torch.empty(nl * atb.box_bytes(ma), dtype=torch.uint8, device=device)
    warm, cold = timed(lambda: atb.tile_load(ma, listed, nl, packed_l, stream=stream), 300, 10)
    out["f32_16384x8192_listed_gather"] = line(2 * rows * cols * 4, nl, warm, cold)
    warm, cold = timed(lambda: atb.tile_roundtrip(ma, mb, listed, nl, stream=stream), 300, 10)
    out["f32_16384x8192_listed_roundtrip"] = line(2 * rows * cols * 4, nl, warm, cold)
    del packed_l
    atb.check_device(stream)
    return out


def fixed_cost_fits(torch, atb, datagen, device, stream, timed, dev_bytes, src4, ms4, mf4):
    """Each short launch as T(n) = T0 + n * t: the same launch over n boxes for
    several n, timed after an L2 flush, and a least-squares line through the
    points.  T0 is what a launch costs before and around its boxes (launch,
    ramp-up of the first DRAM reads, drain of the last stores); bytes per box
    / t is the rate the kernel sustains in between.  Fractions are of the
    measured copy peak."""
    import numpy as np

    peak, _ = hbm_peak()

    def fit(label, ns, bytes_per_box, make_fn):
        pts = []
        for n in ns:
            _, cold = timed(make_fn(n), 20, 20)
            pts.append((n, cold))
        x = np.array([p[0] for p in pts], dtype=np.float64)
        y = np.array([p[1] for p in pts], dtype=np.float64)
        t, t0 = np.polyfit(x, y, 1)
        full = pts[-1]
        return {"points_us": {int(n): round(c * 1e6, 2) for n, c in pts}, "fixed_us": round(t0 * 1e6, 2),
                "marginal_GBps": round(bytes_per_box / t / 1e9, 1),
                "marginal_frac_of_peak": round(bytes_per_box / t / 1e9 / peak, 3),
                "full_launch_frac_of_peak": round(full[0] * bytes_per_box / full[1] / 1e9 / peak, 3),
                "full_launch_net_of_fixed_frac": round(full[0] * bytes_per_box / (full[1] - t0) / 1e9 / peak, 3),
                "what": label}

    w = datagen.C4
    coords_h = datagen.workload_coords(w)
    coords = dev_bytes(coords_h.view(np.uint8))
    bb = atb.box_bytes(ms4)
    packed = torch.empty(len(coords_h) * bb, dtype=torch.uint8, device=device)
    inb_per_box = box_inbound_bytes(w.dims, w.box, w.esize, coords_h) / len(coords_h)
    ns4 = (512, 1024, 2048, 3072, 4096)
    out = {"c4_gather": fit("workload 4 gather, first n of its 4096 listed boxes", ns4, inb_per_box + bb,
                            lambda n: (lambda: atb.tile_load(ms4, coords, n, packed, stream=stream))),
           "c4_store": fit("workload 4 store, first n of its 4096 listed boxes", ns4, inb_per_box + bb,
                           lambda n: (lambda: atb.tile_store(mf4, coords, n, packed, stream=stream))),
           "c4_roundtrip": fit("workload 4 round trip, first n of its 4096 listed boxes", ns4, 2 * inb_per_box,
                               lambda n: (lambda: atb.tile_roundtrip(ms4, mf4, coords, n, stream=stream)))}
    # workload 3 over its first box rows (47 boxes each, the last column ragged)
    w = datagen.C3
    src3 = dev_bytes(datagen.storage(w))
    maps3 = {}
    for box_rows in (10, 20, 40, 60, 78):
        m3 = atb.encode_tiled(w.dtype, src3, (w.dims[0], box_rows * w.box[1]), w.strides, w.box, w.swizzle)
        maps3[atb.grid_tiles(m3)] = m3
    n3max = max(maps3)
    packed3 = torch.empty(n3max * atb.box_bytes(m3), dtype=torch.uint8, device=device)
    per_box3 = (w.dims[0] * 2 * w.box[1] * 78) / n3max + atb.box_bytes(m3)  # in-bound bytes + image, per box
    out["c3_gather"] = fit("workload 3 gather over its first box rows", sorted(maps3), per_box3,
                           lambda n: (lambda: atb.tile_load(maps3[n], None, 0, packed3, stream=stream)))
    # workload 2 over its first rows: the same 64 x 256 boxes, n = 7 column tiles x row strips
    w = datagen.C2
    src2 = dev_bytes(datagen.storage(w))
    dst2 = torch.zeros(w.storage_bytes, dtype=torch.uint8, device=device)
    maps = {}
    for strips in (16, 33, 66, 99, 132):
        rows = strips * 64
        maps[strips * 7] = (atb.encode_tiled(w.dtype, src2, (w.dims[0], rows), w.strides, w.box, w.swizzle),
                            atb.encode_tiled(w.dtype, dst2, (w.dims[0], rows), w.strides, w.box, w.swizzle))
    out["c2_round_trip"] = fit("workload 2 round trip over its first row strips (library grid)", sorted(maps),
                               2 * 64 * 256 * 2,
                               lambda n: (lambda: atb.tile_roundtrip(maps[n][0], maps[n][1], stream=stream)))
    # host side of one call: ctypes marshalling and the library's launch, with the GPU kept busy
    busy = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    w = datagen.C1
    s1 = dev_bytes(datagen.storage(w))
    d1 = torch.zeros_like(s1)
    m1s = atb.encode_tiled(w.dtype, s1, w.dims, w.strides, w.box, w.swizzle)
    m1d = atb.encode_tiled(w.dtype, d1, w.dims, w.strides, w.box, w.swizzle)
    with torch.cuda.stream(stream):
        for _ in range(4):
            busy.zero_()
        t0 = time.perf_counter()
        for _ in range(200):
            atb.tile_roundtrip(m1s, m1d, stream=stream, stages=1, ctas=1)
        host = (time.perf_counter() - t0) / 200
    stream.synchronize()
    out["host_us_per_call"] = {"value": round(host * 1e6, 2),
                               "what": "Python binding + library enqueue of one round-trip call (CPU clock, GPU busy)"}
    return out


def ablations(torch, atb, device, stream, src, dst, nbytes, args):
    steps = max(50, min(400, args.steps // 10))
    res = {}
    for name, fn in (("cpasync_ldgsts", atb.copy_cpasync), ("ldst_global_v4", atb.copy_ldst_v4),
                     ("cudaMemcpyAsync_d2d", atb.copy_memcpy)):
        s = time_launches(torch, stream, lambda: fn(src, dst, nbytes, stream=stream), steps, 5)
        res[name] = round(2 * nbytes * steps / s / 1e9, 1)
    return res


def end_to_end(torch, atb, w, device, stream, src_h, nbytes, bytes_per_step, args, dist):
    """Through the public host-buffer call: per step, encode the maps and run
    atb_tile_roundtrip_host (pinned H2D of the input, round trip, D2H of the
    output, overlapped slab by slab)."""
    src_pin = torch.from_numpy(src_h).pin_memory()
    out_pin = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    src = torch.empty(nbytes, dtype=torch.uint8, device=device)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def step():
        ms = atb.encode_tiled(w.dtype, src, w.dims, w.strides, w.box, w.swizzle)
        md = atb.encode_tiled(w.dtype, dst, w.dims, w.strides, w.box, w.swizzle)
        atb.tile_roundtrip_host(ms, md, src_pin, out_pin, args.slabs, stream=stream, stages=args.stages,
                                ctas_per_sm=args.ctas_per_sm)

    steps = max(3, args.e2e_steps)
    seconds = time_launches(torch, stream, step, steps, 3, dist, device)
    atb.check_device(stream)
    ok = bool(torch.equal(out_pin, src_pin))  # the whole host output of the last step
    units, max_s = aggregate(dist, seconds, float(bytes_per_step) * steps, device)
    # the host link this box gives the same buffers: one H2D and one D2H copy of the whole tensor at once, on
    # two streams, no kernel (the ceiling of any host-buffer round trip of this size)
    up, down = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    link = []
    for _ in range(4):
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        with torch.cuda.stream(up):
            src.copy_(src_pin, non_blocking=True)
        with torch.cuda.stream(down):
            out_pin.copy_(dst, non_blocking=True)
        torch.cuda.synchronize(device)
        link.append(2 * nbytes / (time.perf_counter() - t0) / 1e9)
    link_gbs = max(link[1:])
    value = units / max_s / 1e9
    return {"value": round(value, 1), "unit": "GB/s", "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": nbytes, "steps": steps, "ms_per_step": round(max_s / steps * 1e3, 3),
            "slabs": args.slabs or 12, "call": "atb_tile_roundtrip_host", "verified": ok,
            "host_link_bidirectional_GBps": round(link_gbs, 1), "frac_of_host_link": round(value / link_gbs, 3)}


def cpu_baseline(w, src_h, repeats: int = 4):
    """The oracle as it stands, single-threaded: `repeats` full round trips of the workload."""
    import numpy as np

    import oracle

    v = oracle.View(w.esize, w.dims, w.strides, w.box, w.swizzle)
    coords = oracle.grid_coords(v)
    dst = np.zeros_like(src_h)
    t0 = time.perf_counter()
    for _ in range(repeats):
        oracle.roundtrip(v, src_h, v, dst, coords)
    dt = time.perf_counter() - t0
    matches = bool(np.array_equal(dst, src_h))
    return {"value": round(2 * w.storage_bytes * repeats / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{repeats} full round trips of {w.name} ({len(coords)} boxes, 1 GiB moved each), "
                      f"single thread, {dt:.2f} s; host has {os.cpu_count()} cores",
            "matches_input": matches,
            "all_cores": cpu_baseline_threaded(w, src_h, v, coords, 2 * repeats)}


def cpu_baseline_threaded(w, src_h, v, coords, repeats: int):
    """The same oracle round trip on every host core: the grid's boxes split
    into one contiguous run per thread.  The oracle is C behind ctypes, which
    releases the GIL for the call, so the threads run in parallel; grid boxes
    are disjoint, so the threads write disjoint bytes."""
    import threading

    import numpy as np

    import oracle

    threads = max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)
    parts = np.array_split(coords, threads)
    dst = np.zeros_like(src_h)

    def work():
        for _ in range(repeats):
            pool = [threading.Thread(target=oracle.roundtrip, args=(v, src_h, v, dst, part)) for part in parts]
            for t in pool:
                t.start()
            for t in pool:
                t.join()

    t0 = time.perf_counter()
    work()
    dt = time.perf_counter() - t0
    return {"value": round(2 * w.storage_bytes * repeats / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "sample": f"{repeats} full round trips of {w.name}, {threads} threads over contiguous box runs, "
                      f"{dt:.2f} s",
            "matches_input": bool(np.array_equal(dst, src_h))}


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle, timed on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    import numpy as np

    import datagen
    import oracle

    rank, _, world = dist_env()
    if rank != 0:
        return
    w = datagen.C5A if args.box == "64x256" else datagen.C5B
    v = oracle.View(w.esize, w.dims, w.strides, w.box, w.swizzle)
    coords = oracle.grid_coords(v)
    # Boxes per step: as given, else sized so that warm-up plus timed steps
    # stay under about a minute of single-core oracle work.
    sample_tiles = args.ref_tiles or max(8, min(1024, REF_BOX_BUDGET // (args.steps + args.warmup)))
    sample = coords[:sample_tiles]
    src_h = datagen.storage(w)
    dst = np.zeros_like(src_h)
    bytes_per_step = 2 * len(sample) * oracle.box_bytes(v)
    for _ in range(args.warmup):
        oracle.roundtrip(v, src_h, v, dst, sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.roundtrip(v, src_h, v, dst, sample)
    dt = time.perf_counter() - t0
    value = bytes_per_step * args.steps / dt / 1e9
    desc = (f"first {len(sample)} of {len(coords)} boxes of {w.name} per step "
            f"({bytes_per_step / 2**20:.0f} MiB moved), single thread")
    print(json.dumps({
        "impl": "reference", "metric": "TMA tiled round trip HBM GB/s (read+write)", "value": round(value, 4),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded normal(0,1) fp16)",
        "config": {"workload": w.name, "box": args.box, "sample": desc},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=8000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["atb", "reference"], default="atb")
    p.add_argument("--box", choices=["64x256", "128x64"], default="128x64")
    p.add_argument("--stages", type=int, default=0, help="0 = library default")
    p.add_argument("--ctas-per-sm", type=int, default=0, help="0 = library default")
    p.add_argument("--store-groups", type=int, default=0, help="0 = library default")
    p.add_argument("--poll-suspend-ns", type=int, default=0, help="mbarrier poll suspend hint (0 = default)")
    p.add_argument("--consumer", choices=["auto", "drain", "warp"], default="auto",
                   help="tile-grid consumer (auto = the library's choice)")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--slabs", type=int, default=0, help="host round trip slabs (0 = library default)")
    p.add_argument("--ref-tiles", type=int, default=0,
                   help="boxes per reference-arm step (0 = sized from --steps/--warmup)")
    p.add_argument("--no-extras", action="store_true", help="skip the stage sweep and ablations")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
