#!/usr/bin/env python3
"""Benchmark of the guided-NVFP4 hot path of TRACE on GB300.

One step = one pass of the whole path over one batch of the workload:
  rollout side:  segment amax + NVFP4 quantisation with the compact record
  record:        guide pack (codes -> compact words), guide unpack (round trip)
  training side: segment amax + rollout-guided fake quantisation (bf16 out,
                 STE mask)
The default workload is the long-rollout KV stream (48 layers x K/V x 131072
tokens x 4 heads x 128, 6.44 G elements per tensor, guide in 4096-token
chunks).  Inputs are synthetic (seeded generators), resident in HBM, and far
larger than L2, so no flush is needed between steps.

Metric: algorithmic bytes in + out of every kernel of the step per second
(GB/s = 1e9 B/s); per-kernel GB/s and the HBM-roofline fraction of the
dominant kernel come from CUDA events recorded by the library around each
launch on its own stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5]
                  [--guide compact|full] [--impl ours|reference]

``--impl reference`` times the CPU oracle (the plain single-threaded
definition) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "guided NVFP4 fake-quant GB/s (bytes in+out) and % of GB300 HBM peak"
# algorithmic bytes per element of each kernel (reads + writes)
# (the fused rollout kernel moves x once through HBM: its quantisation pass
# re-reads x from L2)
KERNEL_BYTES = {"amax": 2.0, "rollout_quant": 2.8125, "rollout_fused": 2.8125,
                "guide_pack": 0.75, "guide_unpack": 2.8125, "fakequant_compact": 4.4375,
                "fakequant_full": 4.6875, "ste_backward": 4.125}


def kernel_bytes(name: str, guide: str) -> float:
    return KERNEL_BYTES["fakequant_" + guide] if name == "fakequant" else KERNEL_BYTES[name]


def step_bytes_per_elem(guide: str) -> float:
    """The step's work in bytes per element: every row's bytes in + out (the
    amax row counted on both sides), however the kernels are fused."""
    fq = KERNEL_BYTES["fakequant_" + guide]
    return (KERNEL_BYTES["amax"] * 2 + KERNEL_BYTES["rollout_quant"] + KERNEL_BYTES["guide_pack"]
            + KERNEL_BYTES["guide_unpack"] + fq)


# DRAM bytes per element (read + write) of the dominant kernel from one ncu
# capture (profiles/), valid only for the kernel source it was taken on; a
# changed source reports traffic as null.
MEASURED_TRAFFIC = {
    "fakequant_compact": {"bytes_per_elem": 4.454, "kernels_sha1": "deea475f5272"},
}


def kernels_sha1() -> str:
    """Hash of the fake-quant kernel's code (its own file and the shared
    device helpers, comments and blank space removed): a code change there
    makes the stored traffic stale, a comment edit does not."""
    import hashlib
    import re
    h = hashlib.sha1()
    for name in ("trace_fakequant.cu", "trace_device.cuh"):
        with open(os.path.join(ROOT, "fp4_rollout_guided_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:12]


def measured_traffic(kind: str, elems: int):
    m = MEASURED_TRAFFIC.get("fakequant_" + kind)
    if not m or m["kernels_sha1"] != kernels_sha1():
        return None
    return round(m["bytes_per_elem"] * elems / 1e9, 3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(1.0)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s, p in zip(sm, power) if p > 0.3 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "samples": len(sm), "power_w_max": max(power), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, use_cuda):
    if world <= 1:
        return None
    import torch.distributed as dist
    dist.init_process_group("nccl" if use_cuda else "gloo")
    return dist


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample(w, rows):
    """First `rows` rows of training segment 0 with the rollout segments that
    fall inside them (drawn on the host by the same generator)."""
    from fp4_rollout_guided_gb300 import synth
    x, r = synth.segment_inputs(w, 0, "cpu")
    rows = min(rows, x.shape[0])
    cuts = w.seg_r[(w.seg_r > 0) & (w.seg_r < rows)]
    seg_r = np.concatenate([[0], cuts, [rows]]).astype(np.int64)
    return synth.to_u16(x[:rows]), synth.to_u16(r[:rows]), seg_r


def oracle_step(xu, ru, seg_r, guide_kind):
    import oracle
    codes, bs, gs, guide = oracle.rollout_quant(ru, seg_r)
    oracle.guide_pack(codes)
    oracle.guide_unpack(ru, guide, bs, gs, seg_r)
    kind = oracle.GUIDE_COMPACT if guide_kind == "compact" else oracle.GUIDE_FULL
    oracle.train_fakequant(xu, None, kind, guide if guide_kind == "compact" else codes, bs, gs,
                           seg_r, want_codes=False, want_stats=False)


def oracle_rows_for(w, seconds, guide_kind):
    """Rows of a sample that takes about `seconds` of oracle time."""
    probe = max(w.seg_r[1] - w.seg_r[0], 1) if w.n_seg_r > 1 else 256
    probe = int(min(probe, 4096 if w.cols <= 256 else 256))
    xu, ru, sr = oracle_sample(w, probe)
    t = time.perf_counter()
    oracle_step(xu, ru, sr, guide_kind)
    dt = max(time.perf_counter() - t, 1e-3)
    rows = int(probe * seconds / dt)
    quantum = int(w.seg_r[1] - w.seg_r[0]) if w.n_seg_r > 1 else 1
    quantum = max(1, min(quantum, 4096))
    rows = max(quantum, rows // quantum * quantum)
    return rows


def cpu_baseline(w, guide_kind, seconds=12.0):
    import oracle
    oracle.build()
    rows = oracle_rows_for(w, seconds, guide_kind)
    xu, ru, sr = oracle_sample(w, rows)
    t = time.perf_counter()
    oracle_step(xu, ru, sr, guide_kind)
    dt = time.perf_counter() - t
    elems = xu.size
    gbs = step_bytes_per_elem(guide_kind) * elems / dt / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"rows 0..{rows} of training segment 0 ({elems} elements, "
                      f"{len(sr) - 1} rollout segments), one full step, {dt:.2f} s"}


def run_reference(args, w):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    import oracle
    oracle.build()
    rows = oracle_rows_for(w, 1.5, args.guide)
    xu, ru, sr = oracle_sample(w, rows)
    for _ in range(args.warmup):
        oracle_step(xu, ru, sr, args.guide)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(xu, ru, sr, args.guide)
    dt = (time.perf_counter() - t) / max(args.steps, 1)
    value = step_bytes_per_elem(args.guide) * xu.size / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "sample_rows": rows, "sample_elements": int(xu.size)},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: rows 0..{rows} of training segment 0 "
                                       f"({xu.size} elements)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the GPU path
# ---------------------------------------------------------------------------

def mem_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def run_ours(args, w0):
    from fp4_rollout_guided_gb300 import build, shard, synth, trace
    world, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, True)
    build.build()
    plan = shard.weak_plan(world, rank, args.seed)
    w = synth.workload(w0.cfg, seed=plan.seed)
    elems = w.elems
    h = trace.Handle(local)
    if args.no_fuse:
        h.set_option("fused_amax", 0)

    t_gen = time.perf_counter()
    x, r = synth.make_inputs(w, dev)
    rows, cols = w.rows, w.cols
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    bs = torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev)
    gs = torch.empty((w.n_seg_r,), dtype=torch.float32, device=dev)
    guide = torch.empty((rows, cols // 16), dtype=torch.int32, device=dev)
    packed = torch.empty_like(guide)
    unpacked = torch.empty_like(codes)
    y = torch.empty_like(x)
    mask = torch.empty((rows, cols // 32), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    t_gen = time.perf_counter() - t_gen
    kind = args.guide

    def step(xd, rd, stats=None):
        h.rollout_quant(rd, w.seg_r, out=(codes, bs, gs, guide))
        h.guide_pack(codes, out=packed)
        h.guide_unpack(rd, guide, bs, gs, w.seg_r, out=unpacked)
        h.train_fakequant(xd, w.seg_t, kind, guide if kind == "compact" else codes, bs, gs,
                          w.seg_r, out=(y, mask, None), stats=stats)

    # correctness guard: the round trip of the record and stats of one step
    st = trace.new_stats(dev)
    step(x, r, st)
    torch.cuda.synchronize()
    stats = trace.stats_dict(st)
    record_ok = bool(torch.equal(packed, guide) and torch.equal(unpacked, codes))

    clocks = ClockSampler(local) if rank == 0 else None
    for _ in range(args.warmup):
        step(x, r)
    torch.cuda.synchronize()
    barrier(dist)
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step(x, r)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    ms = ev0.elapsed_time(ev1) / max(args.steps, 1)
    ms = max_over_ranks(dist, ms, dev)

    # per-kernel times from the library's own events, same steps again
    h.profile(True)
    for _ in range(args.steps):
        step(x, r)
    times = h.collect()
    h.profile(False)
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None

    waits = h.device_status()           # 0, or 6 if an in-kernel wait ran out
    if waits != 0:
        raise SystemExit("an in-kernel wait ran out during the timed steps")
    launches = sum(n for n, _ in times.values())
    bpe = step_bytes_per_elem(kind)
    value = bpe * elems * world / (ms * 1e-3) / 1e9
    fused = times.get("rollout_fused", (0, 0.0))[0] > 0
    peak, peak_src = load_peaks()
    kernels = {}
    for name, (n, tot) in times.items():
        if n == 0:
            continue
        b = kernel_bytes(name, kind)
        avg = tot / n
        gbs = b * elems / (avg * 1e-3) / 1e9
        kernels[name] = {"launches": n, "avg_ms": round(avg, 4), "bytes_per_elem": b,
                         "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4)}
    dom = max(kernels, key=lambda k: kernels[k]["avg_ms"] * kernels[k]["launches"])
    roof = {"bound": "hbm", "kernel": dom, "achieved": kernels[dom]["gbs"], "peak": peak,
            "unit": "GB/s", "frac": round(kernels[dom]["gbs"] / peak, 4),
            "traffic": measured_traffic(kind, elems) if dom == "fakequant" else None,
            "traffic_unit": "GB per launch", "peak_source": peak_src}

    e2e = measure_e2e(args, h, w, x, r, step, dev, bpe, (y, mask, guide, bs, gs)) \
        if not args.no_e2e else None
    e2e_v = None if e2e is None else max_over_ranks(dist, e2e["ms"], dev)

    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(w, kind)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "io_dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "elements_per_gpu": elems,
                       "segments_train": w.n_seg_t, "segments_rollout": w.n_seg_r,
                       "guide": kind,
                       "step": ("rollout_fused(amax+quant)" if fused else "amax+rollout_quant")
                       + ", guide_pack, guide_unpack, amax+guided_fakequant",
                       "step_bytes_per_elem": bpe,
                       "l2": "inputs larger than L2 (no flush needed)",
                       "parallelism": f"replica-per-gpu x{world}"},
            "percent_of_hbm_peak": round(100 * value / world / peak, 2),
            "kernels": kernels, "roofline": roof, "gpu_launches": launches,
            "clocks": clk, "cpu_baseline": base,
            "e2e": None if e2e is None else {
                "value": round(bpe * e2e["elems"] * world / (e2e_v * 1e-3) / 1e9, 1),
                "unit": "GB/s", "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e_v, 3), "scope": e2e["scope"],
                "pipeline": "per training segment: H2D (x, r on two streams), kernels, D2H overlap",
                "matches_device_step": e2e["matches_device_step"]},
            "mismatch": {"rtn_rate": stats["mismatch_rtn"] / max(stats["n_elems"], 1),
                         "guided_rate": stats["mismatch_guided"] / max(stats["n_elems"], 1),
                         "hist_rtn": stats["hist_rtn"], "hist_guided": stats["hist_guided"]},
            "record_round_trip_ok": record_ok,
            "generation_s": round(t_gen, 2),
        }
        print(json.dumps(line), flush=True)
    h.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def measure_e2e(args, h, w, x, r, step, dev, bpe, outs):
    """Same step through the public API with the inputs in pinned host memory
    (see _e2e_rows), on the whole workload when the host can pin it."""
    y, mask, guide, bs, gs = outs
    in_bytes = x.numel() * 2 * 2
    out_bytes = sum(t.numel() * t.element_size() for t in (y, mask, guide, bs, gs))
    need = in_bytes + out_bytes
    # every local rank pins its own buffers: share the host's free memory
    local_ranks = max(1, int(os.environ.get("LOCAL_WORLD_SIZE", "1")))
    avail = mem_available_bytes() // local_ranks
    scope = "whole workload"
    rows = w.rows
    if avail and need * 1.6 > avail:
        # keep pinned memory within the host's means: a leading row range of
        # whole training segments (same kernels, fewer rows)
        frac = avail / (need * 1.6)
        k = max(1, int(w.n_seg_t * frac))
        rows = int(w.seg_t[k])
        scope = f"first {k} of {w.n_seg_t} training segments (host memory)"
    if rows != w.rows:
        return None if rows == 0 else _e2e_rows(args, h, w, x, r, dev, bpe, rows, scope)
    return _e2e_rows(args, h, w, x, r, dev, bpe, rows, scope, step=step, outs=outs)


def _e2e_rows(args, h, w, x, r, dev, bpe, rows, scope, step=None, outs=None):
    """The step through the public API on host-resident inputs: pinned x and
    r go in and y, the STE mask and the compact record (words, block scales,
    global scales) come back, streamed per training segment on three CUDA
    streams (fp4_rollout_guided_gb300.pipeline), all inside the timed region."""
    from fp4_rollout_guided_gb300 import pipeline
    seg_t = w.seg_t[w.seg_t <= rows]
    seg_r = w.seg_r[w.seg_r <= rows]
    x_h = torch.empty((rows, w.cols), dtype=torch.bfloat16, pin_memory=True)
    r_h = torch.empty_like(x_h, pin_memory=True)
    x_h.copy_(x[:rows])
    r_h.copy_(r[:rows])
    streamer = pipeline.HostStreamedStep(h, rows, w.cols, seg_t, seg_r, args.guide)
    host_outs = streamer.host_outputs()

    n_e2e = max(3, min(args.steps, 10))
    for _ in range(2):
        streamer.run(x_h, r_h, host_outs)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        streamer.run(x_h, r_h, host_outs)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / n_e2e
    # the streamed outputs are the one-call step's, bit for bit
    same = None
    if outs is not None:
        same = all(torch.equal(hst.to(dev, non_blocking=False), dv)
                   for hst, dv in zip(host_outs, outs))
    h2d = x_h.numel() * 2 + r_h.numel() * 2
    d2h = sum(t.numel() * t.element_size() for t in host_outs)
    del streamer
    torch.cuda.empty_cache()
    return {"ms": ms, "elems": rows * w.cols, "h2d": h2d, "d2h": d2h, "scope": scope,
            "matches_device_step": same}


def run_transport(args, w):
    """Guide-record transport on one GPU: device -> pinned host (export),
    host -> file (write + fsync), file -> pinned host (read), pinned host ->
    device (import), for the full record (4-bit codes) and the compact one
    (2 bits per element), on the same rollout output.  Prints one JSON line."""
    import tempfile
    from fp4_rollout_guided_gb300 import build, synth, trace
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    h = trace.Handle(0)
    x, r = synth.make_inputs(w, dev)
    del x
    codes, bs, gs, guide = h.rollout_quant(r, w.seg_r)
    del r
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    res = {}
    tmp = tempfile.mkdtemp(prefix="trace_record_")
    try:
        for kind, g in (("full", codes), ("compact", guide)):
            size = trace.record_size(kind, w.rows, w.cols, w.n_seg_r)
            host = torch.empty(size, dtype=torch.uint8, pin_memory=True)
            out = (torch.empty_like(g), torch.empty_like(bs), torch.empty_like(gs))
            for _ in range(args.warmup):
                h.record_export(g, bs, gs, w.seg_r, out=host)
                h.record_import(host, out=out)
            torch.cuda.synchronize()
            d2h, h2d = [], []
            for _ in range(args.steps):
                a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
                a.record(stream)
                h.record_export(g, bs, gs, w.seg_r, out=host, wait=False)
                b.record(stream)
                h.record_import(host, out=out)
                c.record(stream)
                c.synchronize()
                d2h.append(a.elapsed_time(b))
                h2d.append(b.elapsed_time(c))
            assert torch.equal(out[0], g) and torch.equal(out[1], bs)
            path = os.path.join(tmp, f"{kind}.trg")
            t0 = time.perf_counter()
            trace.save_record(host, path)
            with open(path, "rb+") as f:
                os.fsync(f.fileno())
            t_write = time.perf_counter() - t0
            t0 = time.perf_counter()
            back = trace.load_record(path)
            t_read = time.perf_counter() - t0
            assert torch.equal(back, host)
            os.remove(path)
            del back
            ms_d2h, ms_h2d = statistics.median(d2h), statistics.median(h2d)
            res[kind] = {"record_bytes": size, "guide_bytes": g.numel() * g.element_size(),
                         "d2h_ms": round(ms_d2h, 4), "d2h_gbs": round(size / ms_d2h / 1e6, 2),
                         "h2d_ms": round(ms_h2d, 4), "h2d_gbs": round(size / ms_h2d / 1e6, 2),
                         "disk_write_ms": round(t_write * 1e3, 2),
                         "disk_read_ms": round(t_read * 1e3, 2)}
    finally:
        os.rmdir(tmp)
    line = {"metric": "guide record transport (device->host->disk->host->device)",
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "config": {"workload": w.name, "rows": w.rows, "cols": w.cols,
                       "rollout_segments": w.n_seg_r},
            "full": res["full"], "compact": res["compact"],
            "compact_over_full_bytes": round(res["compact"]["record_bytes"]
                                             / res["full"]["record_bytes"], 4),
            "disk_note": "write includes fsync; read is from the page cache"}
    print(json.dumps(line), flush=True)
    h.close()
    return 0


def run_backward(args, w):
    """The straight-through backward (grad_in = grad_out where the STE mask
    bit is 1) over the workload, with the mask of one guided fake
    quantisation of its training tensor.  Prints one JSON line."""
    from fp4_rollout_guided_gb300 import build, synth, trace
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    h = trace.Handle(0)
    x, r = synth.make_inputs(w, dev)
    codes, bs, gs, guide = h.rollout_quant(r, w.seg_r)
    y, mask, _, _ = h.train_fakequant(x, w.seg_t, "compact", guide, bs, gs, w.seg_r)
    del r, codes, guide, y
    g = x  # any bf16 tensor of the shape serves as the incoming gradient
    out = torch.empty_like(g)
    for _ in range(args.warmup):
        h.ste_backward(g, mask, out=out)
    torch.cuda.synchronize()
    h.profile(True)
    for _ in range(args.steps):
        h.ste_backward(g, mask, out=out)
    t = h.collect()
    h.profile(False)
    torch.cuda.synchronize()
    n, tot = t["ste_backward"]
    ms = tot / max(n, 1)
    bpe = KERNEL_BYTES["ste_backward"]
    gbs = bpe * w.elems / (ms * 1e-3) / 1e9
    peak, src = load_peaks()
    line = {"metric": "STE backward GB/s (bytes in+out)", "value": round(gbs, 1), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "elements": w.elems, "bytes_per_elem": bpe},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_source": src},
            "gpu_launches": n}
    print(json.dumps(line), flush=True)
    h.close()
    return 0


def run_gemm(args):
    """The f4 consumer: NVFP4 GEMM over rollout codes on one GPU.  Weights W
    [N, K] are quantised once; each step quantises the activations X [M, K]
    (rollout quantiser writing the scales in the tensor-core tile layout) and runs
    Y = X W^T (cuBLASLt block-scaled E2M1 GEMM, bf16 out).  Prints one JSON
    line with the GEMM's TFLOP/s against the FP4 tensor peak."""
    from fp4_rollout_guided_gb300 import build, trace
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    h = trace.Handle(0)
    M, N, K = args.gemm_shape
    g = torch.Generator(device=dev).manual_seed(args.seed)
    x = (torch.randn((M, K), generator=g, device=dev) * 2.0).to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    b = h.nvfp4_operand(w)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    a = h.nvfp4_operand(x)

    def step():
        h.nvfp4_operand(x, out=a)
        h.nvfp4_gemm(a, b, out=y)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    h.profile(True)
    for _ in range(args.steps):
        step()
    t = h.collect()
    h.profile(False)
    torch.cuda.synchronize()
    flops = 2.0 * M * N * K
    g_n, g_ms = t["nvfp4_gemm"]
    gemm_ms = g_ms / max(g_n, 1)
    peak, src = load_peaks()
    bf16_peak = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"] \
        if src == "measured" else 1900.0
    fp4_peak = bf16_peak * 13.5 / 2.25      # dense FP4 / BF16 nominal ratio
    tflops = flops / (gemm_ms * 1e-3) / 1e12
    quant = {k: round(v[1] / max(v[0], 1), 4) for k, v in t.items() if v[0] and k != "nvfp4_gemm"}
    line = {"metric": "NVFP4 GEMM over rollout codes (TFLOP/s)", "value": round(tflops, 1),
            "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "e2m1",
            "data": "synthetic",
            "config": {"workload": f"Y[{M},{N}] = X[{M},{K}] W[{N},{K}]^T, X quantised each step",
                       "out": "bf16"},
            "gemm_ms": round(gemm_ms, 4), "quantise_ms": quant,
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1),
                         "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                         "frac": round(tflops / fp4_peak, 4),
                         "peak_source": f"{src} bf16 x 6 (dense FP4 / BF16 nominal)"}}
    print(json.dumps(line), flush=True)
    h.close()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--guide", default="compact", choices=["compact", "full"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fuse", action="store_true",
                    help="rollout side as two kernels (amax, then quantiser)")
    ap.add_argument("--backward", action="store_true",
                    help="time the straight-through backward instead")
    ap.add_argument("--gemm", action="store_true",
                    help="time the NVFP4 GEMM over rollout codes instead")
    ap.add_argument("--gemm-shape", type=int, nargs=3, default=[16384, 8192, 8192],
                    metavar=("M", "N", "K"))
    ap.add_argument("--transport", action="store_true",
                    help="time the guide record's device/host/disk round trip instead")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)   # at least three untimed warm-up steps
    from fp4_rollout_guided_gb300 import synth
    w = synth.workload(args.workload, seed=args.seed)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.transport:
        return run_transport(args, w)
    if args.gemm:
        return run_gemm(args)
    if args.backward:
        return run_backward(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
