#!/usr/bin/env python3
"""Benchmark of the guided-NVFP4 hot path of TRACE on GB300.

One step = one pass of the whole hot path over one batch of the workload:
  rollout side:  segment amax + NVFP4 quantisation with the compact record
  record:        guide pack (codes -> compact words), guide unpack (round trip)
  training side: segment amax + rollout-guided fake quantisation (bf16 out,
                 STE mask)
The default workload is the long-rollout KV stream (48 layers x K/V x 131072
tokens x 4 heads x 128, 6.44 G elements per tensor, guide in 4096-token
chunks).  Inputs are synthetic (seeded generators), resident in HBM, and far
larger than L2, so no flush is needed between steps.

Metric: the guided fake quantiser's GB/s (its algorithmic bytes in + out,
4.4375 B per element with the compact record, 4.6875 with the full one,
1 GB/s = 1e9 B/s) from CUDA events the library records around each launch
on the launch's own stream, and its fraction of the measured HBM copy peak.
The whole step's row bytes per second are reported beside it (step_gbs), and
so are the other four workloads (per-kernel GB/s, elements/s, roofline
fraction, mismatch rates before and after guidance; compact-vs-full
agreement on the 262144 x 4096 expert activations).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5]
                  [--guide compact|full] [--impl ours|reference]

``--impl reference`` times the CPU oracle (the plain single-threaded
definition, run segment-parallel on every host core) on bounded samples of
the same workload, with the same metric.
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
                "rollout_delayed": 2.8125,
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
    "fakequant_compact": {"bytes_per_elem": 4.370, "kernels_sha1": "b0ff45a279f8"},
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


def oracle_step(xu, ru, seg_r, guide_kind, amax_t=None):
    """One step of the oracle on a sample (rows of one training segment)."""
    import oracle
    codes, bs, gs, guide = oracle.rollout_quant(ru, seg_r)
    oracle.guide_pack(codes)
    oracle.guide_unpack(ru, guide, bs, gs, seg_r)
    kind = oracle.GUIDE_COMPACT if guide_kind == "compact" else oracle.GUIDE_FULL
    oracle.train_fakequant(xu, None, kind, guide if guide_kind == "compact" else codes, bs, gs,
                           seg_r, want_codes=False, want_stats=False,
                           amax_t=None if amax_t is None else [amax_t])


def row_pieces(seg_r, piece_rows=512):
    """(first row, end row, rollout segment) pieces of at most piece_rows
    rows that never cross a rollout segment boundary."""
    out = []
    for k, (a, b) in enumerate(zip(seg_r[:-1], seg_r[1:])):
        for p in range(int(a), int(b), piece_rows):
            out.append((p, min(p + piece_rows, int(b)), k))
    return out


def parallel_maxima(u, seg, n_threads):
    """Per-segment maxima of |u| on a thread pool (exact: a max of maxima)."""
    import oracle
    pieces = row_pieces(seg)
    part = oracle.parallel_map(lambda q: (q[2], float(oracle.segment_amax(u[q[0]:q[1]])[0])),
                               pieces, n_threads)
    m = np.zeros(len(seg) - 1, dtype=np.float32)
    for k, v in part:
        m[k] = max(m[k], v)
    return m


def oracle_step_parallel(xu, ru, seg_r, guide_kind, n_threads=None):
    """The same step on every host core.  The sample's training maximum and
    each rollout segment's maximum come first (maxima of row pieces); then
    every piece of rows is quantised, packed, unpacked and fake-quantised on
    its own with those maxima given, which is the whole step's result
    (segments are independent once their maxima are known)."""
    import oracle
    seg = [0, xu.shape[0]]
    amax_t = float(parallel_maxima(xu, seg, n_threads)[0])
    amax_r = parallel_maxima(ru, seg_r, n_threads)
    kind = oracle.GUIDE_COMPACT if guide_kind == "compact" else oracle.GUIDE_FULL

    def piece(q):
        a, b, k = q
        codes, bs, gs, guide = oracle.rollout_quant(ru[a:b], None, amax=amax_r[k:k + 1])
        oracle.guide_pack(codes)
        oracle.guide_unpack(ru[a:b], guide, bs, gs, None)
        oracle.train_fakequant(xu[a:b], None, kind, guide if guide_kind == "compact" else codes,
                               bs, gs, None, want_codes=False, want_stats=False,
                               amax_t=[amax_t])
    oracle.parallel_map(piece, row_pieces(seg_r), n_threads)


def oracle_fakequant_parallel(xu, gd, bs, gs, seg_r, guide_kind, n_threads=None):
    """The oracle's guided fake quantiser alone (the metric's kernel) on
    every host core: the training maximum first, then pieces of rows."""
    import oracle
    amax_t = float(parallel_maxima(xu, [0, xu.shape[0]], n_threads)[0])
    kind = oracle.GUIDE_COMPACT if guide_kind == "compact" else oracle.GUIDE_FULL
    oracle.parallel_map(
        lambda q: oracle.train_fakequant(xu[q[0]:q[1]], None, kind, gd[q[0]:q[1]], bs[q[0]:q[1]],
                                         gs[q[2]:q[2] + 1], None, want_codes=False,
                                         want_stats=False, amax_t=[amax_t]),
        row_pieces(seg_r), n_threads)


def oracle_rows_for(w, seconds, guide_kind):
    """Rows of a sample that takes about `seconds` of single-threaded oracle
    time, in whole rollout segments."""
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
    """The oracle timed on a bounded sample of the workload, single-threaded
    and segment-parallel on every host core; GB/s of the step's bytes."""
    import oracle
    oracle.build()
    rows = oracle_rows_for(w, seconds, guide_kind)
    xu, ru, sr = oracle_sample(w, rows)
    elems = xu.size
    t = time.perf_counter()
    oracle_step(xu, ru, sr, guide_kind)
    dt1 = time.perf_counter() - t
    n = oracle.threads()
    t = time.perf_counter()
    oracle_step_parallel(xu, ru, sr, guide_kind, n)
    dtn = time.perf_counter() - t
    bpe = step_bytes_per_elem(guide_kind)
    sample = (f"rows 0..{rows} of training segment 0 ({elems} elements, {len(sr) - 1} rollout "
              f"segments), one full step")
    return {"value": bpe * elems / dtn / 1e9, "unit": "GB/s", "cores": n, "threads": n,
            "nproc": os.cpu_count(), "kind": "oracle",
            "sample": sample + f", segment-parallel on {n} threads, {dtn:.2f} s",
            "single_thread": {"value": bpe * elems / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": sample + f", one thread, {dt1:.2f} s"}}


def run_reference(args, w):
    """The reference arm: the CPU oracle's guided fake quantiser (the metric's
    kernel), segment-parallel on every host core, on a sample of the same
    workload; rollout record from the oracle's own rollout quantiser."""
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    import oracle
    oracle.build()
    rows = oracle_rows_for(w, 6.0, args.guide)
    xu, ru, sr = oracle_sample(w, rows)
    codes, bs, gs, guide = oracle.rollout_quant(ru, sr)
    gd = guide if args.guide == "compact" else codes
    n = oracle.threads()
    for _ in range(args.warmup):
        oracle_fakequant_parallel(xu, gd, bs, gs, sr, args.guide, n)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_fakequant_parallel(xu, gd, bs, gs, sr, args.guide, n)
    dt = (time.perf_counter() - t) / max(args.steps, 1)
    value = KERNEL_BYTES["fakequant_" + args.guide] * xu.size / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "guide": args.guide, "sample_rows": rows,
                       "sample_elements": int(xu.size)},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": n, "threads": n,
                             "nproc": os.cpu_count(), "kind": "oracle",
                             "sample": f"each step: the guided fake quantiser over rows "
                                       f"0..{rows} of training segment 0 ({xu.size} elements, "
                                       f"{len(sr) - 1} rollout segments), segment-parallel on "
                                       f"{n} threads"},
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


class StepRunner:
    """Device buffers and the step of one workload through the public API."""

    def __init__(self, h, w, x, r, kind, dev, delayed=False):
        from fp4_rollout_guided_gb300 import trace
        self.h, self.w, self.x, self.r, self.kind, self.dev = h, w, x, r, kind, dev
        rows, cols = w.rows, w.cols
        self.codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        self.bs = torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev)
        self.gs = torch.empty((w.n_seg_r,), dtype=torch.float32, device=dev)
        self.guide = torch.empty((rows, cols // 16), dtype=torch.int32, device=dev)
        self.packed = torch.empty_like(self.guide)
        self.unpacked = torch.empty_like(self.codes)
        self.y = torch.empty_like(x)
        self.mask = torch.empty((rows, cols // 32), dtype=torch.int32, device=dev)
        self.trace = trace
        # delayed scaling: both sides scaled by the maxima the previous step
        # returned (one kernel each, the input read once); a first step here
        # supplies them (x and r are the same every step, so from then on the
        # scales equal the exact path's)
        self.delayed = delayed
        if delayed:
            self.amax_prev = torch.ones((w.n_seg_r,), dtype=torch.float32, device=dev)
            self.amax_next = torch.empty_like(self.amax_prev)
            self.amax_prev_t = torch.ones((w.n_seg_t,), dtype=torch.float32, device=dev)
            self.amax_next_t = torch.empty_like(self.amax_prev_t)
            self.step()

    def step(self, xd=None, rd=None, stats=None, kind=None):
        xd = self.x if xd is None else xd
        rd = self.r if rd is None else rd
        kind = kind or self.kind
        w, h = self.w, self.h
        if self.delayed:
            h.rollout_quant_delayed(rd, w.seg_r, self.amax_prev,
                                    out=(self.codes, self.bs, self.gs, self.guide, self.amax_next))
            self.amax_prev, self.amax_next = self.amax_next, self.amax_prev
        else:
            h.rollout_quant(rd, w.seg_r, out=(self.codes, self.bs, self.gs, self.guide))
        h.guide_pack(self.codes, out=self.packed)
        h.guide_unpack(rd, self.guide, self.bs, self.gs, w.seg_r, out=self.unpacked)
        g = self.guide if kind == "compact" else self.codes
        if self.delayed and stats is None:
            h.train_fakequant_delayed(xd, w.seg_t, self.amax_prev_t, kind, g, self.bs, self.gs,
                                      w.seg_r, out=(self.y, self.mask, self.amax_next_t))
            self.amax_prev_t, self.amax_next_t = self.amax_next_t, self.amax_prev_t
        else:
            h.train_fakequant(xd, w.seg_t, kind, g, self.bs, self.gs, w.seg_r,
                              out=(self.y, self.mask, None), stats=stats)

    def check(self):
        """One step with the counters: the record's round trip and the
        train/rollout mismatch statistics."""
        st = self.trace.new_stats(self.dev)
        self.step(stats=st)
        torch.cuda.synchronize()
        ok = bool(torch.equal(self.packed, self.guide) and torch.equal(self.unpacked, self.codes))
        return ok, self.trace.stats_dict(st)

    def timed(self, steps, warmup, dist=None, kind=None):
        """(ms per step from events around the K steps, per-kernel
        (launches, total ms) from the library's launch events over the
        same number of steps again)."""
        for _ in range(warmup):
            self.step(kind=kind)
        torch.cuda.synchronize()
        barrier(dist)
        stream = torch.cuda.current_stream()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            self.step(kind=kind)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        ms = ev0.elapsed_time(ev1) / max(steps, 1)
        self.h.profile(True)
        for _ in range(steps):
            self.step(kind=kind)
        times = self.h.collect()
        self.h.profile(False)
        torch.cuda.synchronize()
        return ms, times


def kernel_table(times, kind, elems, peak):
    kernels = {}
    for name, (n, tot) in times.items():
        if n == 0:
            continue
        b = kernel_bytes(name, kind)
        avg = tot / n
        gbs = b * elems / (avg * 1e-3) / 1e9
        kernels[name] = {"launches": n, "avg_ms": round(avg, 4), "bytes_per_elem": b,
                         "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4),
                         "elements_per_s": round(elems / (avg * 1e-3), 1)}
    return kernels


def mismatch_of(stats):
    n = max(stats["n_elems"], 1)
    return {"rtn_rate": stats["mismatch_rtn"] / n, "guided_rate": stats["mismatch_guided"] / n,
            "hist_rtn": stats["hist_rtn"], "hist_guided": stats["hist_guided"]}


def agreement_compact_full(h, w, run):
    """Fraction of elements whose guided code from the compact record equals
    the one from the full record (same training values, same rollout record)."""
    _, _, ct, _ = h.train_fakequant(run.x, w.seg_t, "compact", run.guide, run.bs, run.gs, w.seg_r,
                                    mask=False, codes=True)
    _, _, cf, _ = h.train_fakequant(run.x, w.seg_t, "full", run.codes, run.bs, run.gs, w.seg_r,
                                    mask=False, codes=True)
    d = torch.bitwise_xor(ct, cf)
    same = ((d & 0x0F) == 0).sum(dtype=torch.int64) + ((d >> 4) == 0).sum(dtype=torch.int64)
    return float(same.item()) / w.elems


def other_configs(args, h, dev, peak, skip):
    """The other workloads, one after another: per-kernel GB/s, elements/s,
    roofline fraction, mismatch before/after guidance, L2 flag; the expert
    activations 262144 x 4096 add the full-vs-compact comparison."""
    from fp4_rollout_guided_gb300 import synth
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    for cfg in (1, 2, 3, 4, 5):
        if cfg == skip:
            continue
        w = synth.workload(cfg, seed=args.seed)
        x, r = synth.make_inputs(w, dev)
        run = StepRunner(h, w, x, r, "compact", dev)
        ok, stats = run.check()
        steps = max(args.steps, 5)
        ms, times = run.timed(steps, args.warmup)
        kernels = kernel_table(times, "compact", w.elems, peak)
        fq = kernels["fakequant"]
        ws = int(KERNEL_BYTES["fakequant_compact"] * w.elems)
        entry = {"workload": w.name, "elements": w.elems, "segments_train": w.n_seg_t,
                 "segments_rollout": w.n_seg_r, "guide": "compact",
                 "fakequant_gbs": fq["gbs"], "fakequant_frac_of_hbm": fq["frac_of_hbm"],
                 "elements_per_s": fq["elements_per_s"], "ms_per_step": round(ms, 4),
                 "step_gbs": round(step_bytes_per_elem("compact") * w.elems / (ms * 1e-3) / 1e9, 1),
                 "kernels": kernels, "mismatch": mismatch_of(stats), "record_round_trip_ok": ok,
                 "fakequant_bytes": ws, "l2_bytes": l2, "l2_resident": ws <= l2}
        if cfg == 4:
            _, tf = run.timed(steps, args.warmup, kind="full")
            kf = kernel_table(tf, "full", w.elems, peak)["fakequant"]
            entry["full_guide"] = {"fakequant_gbs": kf["gbs"], "fakequant_frac_of_hbm":
                                   kf["frac_of_hbm"], "elements_per_s": kf["elements_per_s"]}
            entry["agreement_compact_vs_full"] = agreement_compact_full(h, w, run)
        out[str(cfg)] = entry
        del run, x, r
        torch.cuda.empty_cache()
    return out


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
    kind = args.guide
    run = StepRunner(h, w, x, r, kind, dev, delayed=args.delayed)
    torch.cuda.synchronize()
    t_gen = time.perf_counter() - t_gen

    # correctness guard: the round trip of the record and stats of one step
    record_ok, stats = run.check()

    clocks = ClockSampler(local) if rank == 0 else None
    ms, times = run.timed(args.steps, args.warmup, dist)
    ms = max_over_ranks(dist, ms, dev)
    clk = clocks.stop() if clocks else None

    waits = h.device_status()           # 0, or 6 if an in-kernel wait ran out
    if waits != 0:
        raise SystemExit("an in-kernel wait ran out during the timed steps")
    launches = sum(n for n, _ in times.values())
    if args.delayed:
        # each delayed call also launches the kernel that turns the given
        # maxima into global scales
        launches += times.get("rollout_delayed", (0, 0.0))[0] + times.get("fakequant", (0, 0.0))[0]
    peak, peak_src = load_peaks()
    kernels = kernel_table(times, kind, elems, peak)
    # the metric: the guided fake quantiser's bytes over its own launch time
    fq_ms = max_over_ranks(dist, kernels["fakequant"]["avg_ms"], dev)
    value = KERNEL_BYTES["fakequant_" + kind] * elems * world / (fq_ms * 1e-3) / 1e9
    bpe = step_bytes_per_elem(kind)
    step_gbs = bpe * elems * world / (ms * 1e-3) / 1e9
    fused = times.get("rollout_fused", (0, 0.0))[0] > 0
    roof = {"bound": "hbm", "kernel": "fakequant", "achieved": round(value / world, 1),
            "peak": peak, "unit": "GB/s", "frac": round(value / world / peak, 4),
            "traffic": measured_traffic(kind, elems), "traffic_unit": "GB per launch",
            "peak_source": peak_src,
            "bytes_per_launch": round(KERNEL_BYTES["fakequant_" + kind] * elems / 1e9, 3)}

    e2e = measure_e2e(args, h, w, x, r, run.step, dev, bpe,
                      (run.y, run.mask, run.guide, run.bs, run.gs)) if not args.no_e2e else None
    e2e_v = None if e2e is None else max_over_ranks(dist, e2e["ms"], dev)
    del run, x, r
    torch.cuda.empty_cache()

    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(w, kind)
    configs = None
    if world == 1 and not args.no_configs:
        configs = other_configs(args, h, dev, peak, skip=w0.cfg)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "io_dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "elements_per_gpu": elems,
                       "segments_train": w.n_seg_t, "segments_rollout": w.n_seg_r,
                       "guide": kind,
                       "step": ("rollout_delayed(quant, maxima of the previous step), "
                                "guide_pack, guide_unpack, guided_fakequant(maxima of the "
                                "previous step)" if args.delayed else
                                ("rollout_fused(amax+quant)" if fused else "amax+rollout_quant")
                                + ", guide_pack, guide_unpack, amax+guided_fakequant"),
                       "value_bytes_per_elem": KERNEL_BYTES["fakequant_" + kind],
                       "step_bytes_per_elem": bpe,
                       "l2": "inputs larger than L2 (no flush needed)",
                       "parallelism": f"replica-per-gpu x{world}"},
            "percent_of_hbm_peak": round(100 * value / world / peak, 2),
            "elements_per_s": round(elems * world / (fq_ms * 1e-3), 1),
            "step_gbs": round(step_gbs, 1),
            "step_percent_of_hbm_peak": round(100 * step_gbs / world / peak, 2),
            "kernels": kernels, "roofline": roof, "gpu_launches": launches,
            "clocks": clk, "cpu_baseline": base,
            "e2e": None if e2e is None else {
                "value": round(KERNEL_BYTES["fakequant_" + kind] * e2e["elems"] * world
                               / (e2e_v * 1e-3) / 1e9, 1),
                "unit": "GB/s", "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e_v, 3), "scope": e2e["scope"],
                "measures": "the fake quantiser's bytes per element over the time of the whole "
                            "step through the public API, inputs from and outputs to "
                            "page-locked host memory",
                "host_memory": "page-locked, huge-page backed (hostmem.host_empty)",
                "step_gbs": round(bpe * e2e["elems"] * world / (e2e_v * 1e-3) / 1e9, 1),
                "pipeline": "pieces of whole training segments: H2D (one stream), kernels, D2H "
                            "(another stream) overlap",
                "matches_device_step": e2e["matches_device_step"]},
            "mismatch": mismatch_of(stats),
            "record_round_trip_ok": record_ok,
            "configs": configs,
            "generation_s": round(t_gen, 2),
        }
        print(json.dumps(line), flush=True)
    h.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def measure_e2e(args, h, w, x, r, step, dev, bpe, outs):
    """Same step through the public API with the inputs in page-locked host
    memory (see _e2e_rows), on the whole workload when the host can hold it."""
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
        # keep page-locked memory within the host's means: a leading row range of
        # whole training segments (same kernels, fewer rows)
        frac = avail / (need * 1.6)
        k = max(1, int(w.n_seg_t * frac))
        rows = int(w.seg_t[k])
        scope = f"first {k} of {w.n_seg_t} training segments (host memory)"
    if rows != w.rows:
        return None if rows == 0 else _e2e_rows(args, h, w, x, r, dev, bpe, rows, scope)
    return _e2e_rows(args, h, w, x, r, dev, bpe, rows, scope, step=step, outs=outs)


def _e2e_rows(args, h, w, x, r, dev, bpe, rows, scope, step=None, outs=None):
    """The step through the public API on host-resident inputs: page-locked
    x and r go in and y, the STE mask and the compact record (words, block
    scales, global scales) come back, streamed in pieces of whole training
    segments on three CUDA streams (fp4_rollout_guided_gb300.pipeline), all
    inside the timed region."""
    from fp4_rollout_guided_gb300 import hostmem, pipeline
    seg_t = w.seg_t[w.seg_t <= rows]
    seg_r = w.seg_r[w.seg_r <= rows]
    # page-locked, huge-page-backed host buffers (the library's host allocator)
    x_h = hostmem.host_empty((rows, w.cols), torch.bfloat16)
    r_h = hostmem.host_empty((rows, w.cols), torch.bfloat16)
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
    from fp4_rollout_guided_gb300 import build, hostmem, synth, trace
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
            host = hostmem.host_empty((size,), torch.uint8)
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
    Y = X W^T (block-scaled E2M1 GEMM, bf16 out: the hand-written tcgen05
    kernel with 128 x 256 or 128 x 128 tiles, or cuBLASLt, --gemm-form).
    Prints one JSON line with the GEMM's TFLOP/s against the FP4 tensor peak."""
    from fp4_rollout_guided_gb300 import build, trace
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    h = trace.Handle(0)
    h.set_option("gemm", args.gemm_form)
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
    def gemm_time():
        h.profile(True)
        for _ in range(args.steps):
            step()
        t = h.collect()
        h.profile(False)
        torch.cuda.synchronize()
        g_n, g_ms = t["nvfp4_gemm"]
        return g_ms / max(g_n, 1), t

    gemm_ms, t = gemm_time()
    flops = 2.0 * M * N * K
    # the library GEMM on the same operands, for comparison (not the metric)
    lt_ms = None
    if args.gemm_form != "cublaslt":
        h.set_option("gemm", "cublaslt")
        try:
            for _ in range(args.warmup):
                step()
            lt_ms = round(gemm_time()[0], 4)
        except RuntimeError:
            lt_ms = None
        h.set_option("gemm", args.gemm_form)
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
                       "out": "bf16", "gemm": args.gemm_form},
            "gemm_ms": round(gemm_ms, 4), "quantise_ms": quant,
            "cublaslt_gemm_ms": lt_ms,
            # our kernels per step: the rollout quantiser (amax, quantisation)
            # and the GEMM kernel, or with cuBLASLt its alpha kernel instead
            "gpu_launches_per_step": 3,
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
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload report of the other four workloads")
    ap.add_argument("--delayed", action="store_true",
                    help="rollout side scaled by the previous step's maxima (one kernel)")
    ap.add_argument("--no-fuse", action="store_true",
                    help="rollout side as two kernels (amax, then quantiser)")
    ap.add_argument("--backward", action="store_true",
                    help="time the straight-through backward instead")
    ap.add_argument("--gemm", action="store_true",
                    help="time the NVFP4 GEMM over rollout codes instead")
    ap.add_argument("--gemm-shape", type=int, nargs=3, default=[16384, 8192, 8192],
                    metavar=("M", "N", "K"))
    ap.add_argument("--gemm-form", default="tc256", choices=["tc256", "tc128", "tc_pair", "cublaslt"],
                    help="GEMM form: hand-written tcgen05 kernel (tile N 256 / 128) or cuBLASLt")
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
