#!/usr/bin/env python3
"""Benchmark of greedy IoU NMS on GB300: one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gbnms|reference]
                    [--workload single_n8192] [--no-cpu-baseline]

A step is one nms_run call (the whole hot path: sort + gather, IoU mask,
resolve + map back) over the headline workload: N=8192 boxes, 300 clusters in
1280x1280, jitter N(0,15), w,h ~ U(8,200), scores Beta(2,5), IoU threshold
0.5.  Inputs are resident in HBM when the timed region starts; L2 is flushed
(a 256 MiB write) before every timed step, outside the timed events.
`value` is boxes/s over all ranks (weak scaling: each rank runs its own copy).
`e2e` is the same metric through nms_run with the host buffers: the pinned
host->device copy of boxes and scores and the device->host read of the keep
list and count are inside the timed region.

--impl reference times the CPU oracle (plain C greedy NMS, one thread) on the
same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from greedy_iou_nms_gb300 import workloads as W  # noqa: E402

METRIC = "NMS µs/call & boxes/s at N=8192; IoU Gpairs/s and mask GB/s vs roofline"
UNIT = "boxes/s"
# FP32 operations of one canonical IoU test (4 min/max, 2 sub, 2 clamp, 1 mul,
# 1 add, 1 sub, 1 div, 1 compare): the algorithmic work per pair.
OPS_PER_PAIR = 13
# How those 13 operations fall on the SM's pipes: the 4 min/max, the 2 clamps
# and the compare run on the ALU pipe (min.f32 and setp class); the 2 subs of
# the sides, the product, the sum, the union's sub and the division (charged
# as one operation) run on the FMA pipe, where the packed f32x2 forms can
# take two of them per instruction.
ALU_OPS_PER_PAIR = 7
FMA_OPS_PER_PAIR = 6
L2_FLUSH_BYTES = 256 << 20
PROBE_LIB = os.path.join(ROOT, "greedy_iou_nms_gb300", "_build", "libgbprobe.so")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.path = os.path.join(tempfile.gettempdir(), f"gbnms_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def measure_alu_peaks(torch, dev, ctas_per_sm=4, iters=2048, reps=5):
    """Measured instruction throughput of the SM (the probe library: each form
    as independent chains on ctas_per_sm CTAs of 256 threads per SM), and the
    FP32 operation roof of the canonical IoU test built from it.

    Per form: operations per second (CUDA events, best of `reps`), the SM
    clock the CTAs saw (clock64 cycles per global-timer nanosecond) and from
    the two the lane operations per SM clock.  The roof: a pair costs
    7 ALU-pipe operations (at the measured min.f32 rate), 6 FMA-pipe
    operations (at the best measured add rate, packed or not) and their
    instructions (at the best measured issue rate); the slowest of the three
    sets the pairs per SM clock, times 13 operations per pair, times the SM
    count and the clock the probe ran at."""
    import ctypes
    lib = ctypes.CDLL(PROBE_LIB)
    lib.gbprobe_form_name.restype = ctypes.c_char_p
    lib.gbprobe_ops_per_thread.restype = ctypes.c_double
    lib.gbprobe_ops_per_thread.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.gbprobe_insts_per_thread.restype = ctypes.c_double
    lib.gbprobe_insts_per_thread.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.gbprobe_launch.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p]
    sms = int(lib.gbprobe_sm_count())
    if sms <= 0:
        raise RuntimeError("probe: no SM count from the device")
    tpc = int(lib.gbprobe_threads_per_cta())
    ctas = sms * ctas_per_sm
    out = torch.empty(ctas * tpc, dtype=torch.float32, device=dev)
    cyc = torch.empty(ctas, dtype=torch.int64, device=dev)
    nsec = torch.empty(ctas, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    forms = {}
    mhz = []
    for f in range(int(lib.gbprobe_forms())):
        name = lib.gbprobe_form_name(f).decode()
        ops = lib.gbprobe_ops_per_thread(f, iters) * tpc * ctas
        ins = lib.gbprobe_insts_per_thread(f, iters) * tpc * ctas
        best_s = None
        for r in range(reps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            rc = lib.gbprobe_launch(f, ctas, iters, out.data_ptr(), cyc.data_ptr(), nsec.data_ptr(),
                                    stream.cuda_stream)
            b.record(stream)
            if rc != 0:
                raise RuntimeError(f"probe launch of {name} failed: cudaError {rc}")
            torch.cuda.synchronize()
            if r == 0:
                continue  # warm-up
            s = a.elapsed_time(b) / 1000
            best_s = s if best_s is None else min(best_s, s)
            mhz.append(1000.0 * float((cyc.double() / nsec.double()).median().item()))
        f_mhz = statistics.median(mhz[-reps:])
        # Per SM clock from the event-timed rate and the clock the CTAs
        # measured (a CTA's own span can miss part of the kernel, so only
        # its cycles per nanosecond are used).
        ops_clk = ops / best_s / (sms * f_mhz * 1e6)
        forms[name] = {"lane_ops_per_clk_per_sm": ops_clk,
                       "lane_insts_per_clk_per_sm": ops_clk * ins / ops,
                       "tops": ops / best_s / 1e12, "mhz": f_mhz}
    r_alu = forms["fmnmx"]["lane_ops_per_clk_per_sm"]
    add_form = max(("fadd", "fadd2"), key=lambda k: forms[k]["lane_ops_per_clk_per_sm"])
    r_fma = forms[add_form]["lane_ops_per_clk_per_sm"]
    ops_per_ins = r_fma / forms[add_form]["lane_insts_per_clk_per_sm"]
    r_issue = max(v["lane_insts_per_clk_per_sm"] for v in forms.values())
    t_alu = ALU_OPS_PER_PAIR / r_alu
    t_fma = FMA_OPS_PER_PAIR / r_fma
    t_issue = (ALU_OPS_PER_PAIR + FMA_OPS_PER_PAIR / ops_per_ins) / r_issue
    pairs_clk = 1.0 / max(t_alu, t_fma, t_issue)
    mhz = statistics.median(v["mhz"] for v in forms.values())
    # The roof per second: pairs per SM clock at the clock the probe ran at.
    roof_tops = OPS_PER_PAIR * pairs_clk * sms * mhz * 1e6 / 1e12
    best = max(forms, key=lambda k: forms[k]["tops"])
    return {"sm_count": sms, "probe_mhz": mhz, "ctas_per_sm": ctas_per_sm, "threads_per_cta": tpc,
            "forms": forms, "roof_pairs_per_clk_per_sm": pairs_clk, "roof_tops": roof_tops,
            "roof_bound": min((("alu", t_alu), ("fma", t_fma), ("issue", t_issue)), key=lambda x: -x[1])[0],
            "roof_add_form": add_form, "best_form": best, "best_form_tops": forms[best]["tops"]}


def bench_config(wl, world):
    """The `config` of both arms' lines (the same dict, so the two lines name
    the same workload the same way)."""
    return {"workload": wl.name, "n": wl.n, "iou_thr": wl.iou_thr, "max_out": wl.max_out,
            "l2": "flushed (256 MiB write) before every timed step",
            "parallelism": f"replicas x{world}"}


def mask_pairs(n, max_out, tile=128):
    """Pairs of the first mask launch of nms_run: the whole triangle, or with
    max_out the leading 2*max_out boxes rounded up to the mask tile width
    (when that is fewer than n)."""
    k = n
    if max_out > 0:
        k = min(n, (2 * max_out + tile - 1) // tile * tile)
    return k * (k - 1) // 2


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_over_ranks(total_ms: float, world: int, n: int, steps: int, device="cpu"):
    """Whole-job timing of `world` replicas: the slowest rank's total time
    (all_reduce MAX over the process group when world > 1) and the aggregate
    boxes/s of all ranks (each rank processes n boxes per step).  Returns
    (total_ms, value)."""
    if world > 1:
        import torch
        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms, world * n * steps / (total_ms / 1000)


def cpu_oracle_run(wl, budget_s: float):
    """Time the oracle (as it stands, one thread) on full copies of the workload
    until about budget_s seconds have passed.  Returns (boxes/s, reps, seconds)."""
    import oracle
    oracle.build()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.nms(wl.boxes, wl.scores, wl.iou_thr, class_ids=wl.class_ids,
                   batch_offsets=wl.batch_offsets, score_thr=wl.score_thr, max_out=wl.max_out)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    return wl.n * reps / dt, reps, dt


def cpu_all_cores_child(name: str, budget_s: float) -> dict:
    """The all-core timing loop of cpu_all_cores_run, in a process of its own."""
    import oracle
    wl = W.make(name, 0)
    oracle.build_cpu_baseline()
    kw = dict(class_ids=wl.class_ids, batch_offsets=wl.batch_offsets, score_thr=wl.score_thr, max_out=wl.max_out)
    oracle.cpu_baseline_nms(wl.boxes, wl.scores, wl.iou_thr, **kw)  # warm-up (thread pool, pages)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.cpu_baseline_nms(wl.boxes, wl.scores, wl.iou_thr, **kw)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    return {"value": wl.n * reps / dt, "reps": reps, "secs": dt, "threads": oracle.cpu_baseline_threads()}


def cpu_all_cores_run(wl, budget_s: float):
    """Time the multi-core CPU baseline (OpenMP bitmask and resolve,
    oracle/cpu_baseline.c) on full copies of workload wl (by its config name)
    for about budget_s seconds, in a child process: in this one PyTorch's own
    thread pool competes for the cores (the baseline ran 4 times slower).
    Returns (boxes/s, reps, seconds, threads)."""
    code = ("import sys, json; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.cpu_all_cores_child(sys.argv[1], float(sys.argv[2]))))" % ROOT)
    out = subprocess.run([sys.executable, "-c", code, wl.name, str(budget_s)], capture_output=True, text=True,
                         check=True, cwd=ROOT).stdout
    r = json.loads(out.strip().splitlines()[-1])
    return r["value"], r["reps"], r["secs"], r["threads"]


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    wl = W.make(args.workload, 0)
    per_step, reps_total = [], 0
    # Each timed step is one full oracle NMS of the workload (a bounded sample:
    # the whole --warmup/--steps run stays within a few minutes).
    for _ in range(args.warmup):
        cpu_oracle_run(wl, 0.0)
    for _ in range(args.steps):
        t0 = time.perf_counter()
        cpu_oracle_run(wl, 0.0)
        per_step.append(time.perf_counter() - t0)
        reps_total += 1
    ms = 1000 * statistics.mean(per_step)
    value = wl.n / (ms / 1000)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": bench_config(wl, ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{reps_total} full runs of {wl.name} (one per step)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def _graph_size(wl):
    """Pairs over the threshold in the upper triangle of the sorted order and
    the number of kept boxes, from the oracle."""
    import oracle
    keep = oracle.nms_single(wl.boxes, wl.scores, wl.iou_thr, max_out=wl.max_out)
    order = oracle.score_order(wl.scores)
    m = oracle.mask(np.ascontiguousarray(wl.boxes[order]), wl.iou_thr)
    bits = int(np.unpackbits(m.view(np.uint8)).sum())
    return bits, len(keep)


def time_after_flush(torch, stream, flush, launch, reps=40, trials=7):
    """Average device time of `launch` when it follows an L2 flush on the
    stream with no event between the two: CUDA events around reps x [flush;
    launch] minus CUDA events around reps x [flush], median of `trials`.
    (An event recorded between two kernels holds the next launch back by
    about 5 us on this platform and rounds to 2.048 us steps, so a kernel
    bracketed by its own events reads long; here only the two sequences are
    bracketed.)"""
    def seq(with_launch):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            flush.fill_(1)
            if with_launch:
                launch()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)
    seq(True)
    seq(False)
    d = [(seq(True) - seq(False)) / reps for _ in range(trials)]
    return statistics.median(d)


def mask_isolated_ms(g, torch, wl, dev, flush):
    """The IoU-mask kernel on its own (nms_iou_mask: the bitmask of boxes
    already in score order), timed after an L2 flush by time_after_flush.
    The boxes are put in score order on the host with numpy (descending
    score, ties to the lower index)."""
    order = np.lexsort((np.arange(wl.n), -wl.scores.astype(np.float64)))
    bs = torch.from_numpy(np.ascontiguousarray(wl.boxes[order])).to(dev)
    ldw = g.nms_mask_row_words(wl.n)
    mask = torch.empty((wl.n, ldw), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def launch():
        st = g.nms_iou_mask(bs.data_ptr(), wl.n, wl.iou_thr, mask.data_ptr(), mask.numel(), stream.cuda_stream)
        if st != g.NMS_OK:
            raise g.NmsError(st, "nms_iou_mask")
    return time_after_flush(torch, stream, flush, launch)


def time_workload(g, torch, wl, dev, flush, reps=30, fast=False, stage_reps=20):
    """Device time of one nms_run call (nms_fast_run with fast=True) on
    workload wl (inputs resident, L2 flushed before each call): median, p10
    and p90 in microseconds."""
    stream = torch.cuda.current_stream(dev)
    batched = wl.class_ids is not None or wl.batch_offsets is not None
    B = wl.batch if wl.batch_offsets is not None else 0
    C = wl.num_classes if wl.class_ids is not None else 0
    boxes = torch.from_numpy(wl.boxes).to(dev)
    scores = torch.from_numpy(wl.scores).to(dev)
    cls = torch.from_numpy(wl.class_ids).to(dev) if wl.class_ids is not None else None
    off = torch.from_numpy(wl.batch_offsets).to(dev) if wl.batch_offsets is not None else None
    cap = g.keep_capacity(wl.n, B if off is not None else None, wl.max_out)
    keep = torch.empty(max(cap, 1), dtype=torch.int64, device=dev)
    counts = torch.empty(max(B, 1), dtype=torch.int64, device=dev)
    ws = g.Workspace(wl.n, B, C, device=dev)
    score_thr = -math.inf if wl.score_thr is None else wl.score_thr

    entry = g.nms_fast_run if fast else g.nms_run

    def call():
        st = entry(boxes.data_ptr(), scores.data_ptr(), wl.n,
                       cls.data_ptr() if cls is not None else 0, C,
                       off.data_ptr() if off is not None else 0, B, wl.iou_thr, score_thr,
                       wl.max_out, keep.data_ptr(), cap, counts.data_ptr(), 0, ws.ptr, ws.bytes,
                       stream.cuda_stream)
        if st != g.NMS_OK:
            raise g.NmsError(st, "nms_run")

    for _ in range(3):
        call()
    evs = []
    for _ in range(reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    us = sorted(1000 * a.elapsed_time(b) for a, b in evs)
    q = lambda f: us[min(len(us) - 1, int(f * len(us)))]
    med = statistics.median(us)
    res = {"us_median": med, "us_p10": q(0.1), "us_p90": q(0.9), "boxes_per_s": wl.n / (med / 1e6),
           "gpairs_per_s": wl.pairs / (med / 1e6) / 1e9, "n": wl.n,
           "kept": int(counts.sum().item()), "batched": batched}
    if fast:
        return res
    # Stage durations of the same call (nms_run_timed: events between the
    # stages on the launching stream, L2 flushed before each call): for one
    # image sort | first mask launch | resolve and any later stage; batched:
    # pre-filter and segmenting | segment NMS | per-image merge.
    stage = [[], [], []]
    for it in range(3 + stage_reps):
        flush.fill_(1)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for e in ev:
            e.record(stream)
        st = g.nms_run_timed(boxes.data_ptr(), scores.data_ptr(), wl.n, cls.data_ptr() if cls is not None else 0,
                             C, off.data_ptr() if off is not None else 0, B, wl.iou_thr, score_thr, wl.max_out,
                             keep.data_ptr(), cap, counts.data_ptr(), 0, ws.ptr, ws.bytes, stream.cuda_stream, ev)
        if st != g.NMS_OK:
            raise g.NmsError(st, "nms_run_timed")
        torch.cuda.synchronize()
        if it >= 3:
            for k in range(3):
                stage[k].append(1000 * ev[k].elapsed_time(ev[k + 1]))
    s0, s1, s2 = (statistics.mean(t) for t in stage)
    if batched:
        res["stages_us"] = {"segmenting": s0, "segment_nms": s1, "merge": s2}
    else:
        res["stages_us"] = {"sort": s0, "mask": s1, "resolve": s2}
        res["mask_pairs"] = mask_pairs(wl.n, wl.max_out)
        if wl.max_out <= 0:
            res["mask_isolated_us"] = 1000 * mask_isolated_ms(g, torch, wl, dev, flush)
    return res


def time_front_end(g, torch, dev, flush, reps=20, conf_thr=0.25, max_objects=1000, iou_thr=0.45):
    """YOLO-shaped head output (16 x 25200 x 85) through the front end: the
    decode into count-header buffers alone, and decode plus greedy NMS over the
    buffers (keep flags), device time per call; the decode's prediction bytes
    against HBM."""
    preds = torch.from_numpy(W.yolo_raw(0)).to(dev)
    batch, anchors, width = preds.shape
    buf = torch.zeros((batch, 1 + 7 * max_objects), dtype=torch.float32, device=dev)
    wsd = g.nms_decode_workspace_size(batch, anchors)
    ws_d = torch.empty(max(wsd, 256), dtype=torch.uint8, device=dev)
    wsn = g.nms_boxes7_workspace_size(batch, max_objects, width - 5)
    ws_n = torch.empty(max(wsn, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def decode():
        st = g.nms_decode_boxes7(preds.data_ptr(), batch, anchors, width - 5, conf_thr, max_objects, buf.data_ptr(),
                                 0, ws_d.data_ptr(), wsd, stream.cuda_stream)
        if st != g.NMS_OK:
            raise g.NmsError(st, "nms_decode_boxes7")

    def nms():
        st = g.nms_boxes7_run(buf.data_ptr(), batch, max_objects, width - 5, iou_thr, 0, 0, ws_n.data_ptr(), wsn,
                              stream.cuda_stream)
        if st != g.NMS_OK:
            raise g.NmsError(st, "nms_boxes7_run")

    def timed(fn):
        for _ in range(3):
            fn()
        evs = []
        for _ in range(reps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(1000 * a.elapsed_time(b) for a, b in evs)

    d_us = timed(decode)
    t_us = timed(lambda: (decode(), nms()))
    pbytes = preds.numel() * 4
    return {"workload": f"yolo head output {batch}x{anchors}x{width} float32, conf > {conf_thr}, "
                        f"max_objects {max_objects}, greedy IoU {iou_thr}",
            "decode_us": d_us, "decode_plus_nms_us": t_us, "prediction_bytes": pbytes,
            "decode_gbs": pbytes / (d_us / 1e6) / 1e9,
            "candidates": int(buf[:, 0].sum().item())}


def time_lanes(g, torch, dev, flush, sizes=(1000, 3000, 16384), thr=15.0, reps=20):
    """Device time of one nms_lane_run call on the seeded lane workloads
    (workloads.lanes: candidates of one road image, 77 values each) at a
    15 px distance threshold: median us per call and lane pairs per second."""
    out = {}
    stream = torch.cuda.current_stream(dev)
    for n in sizes:
        props, scores = W.lanes(0, n=n)
        p = torch.from_numpy(props).to(dev)
        s = torch.from_numpy(scores).to(dev)
        keep = torch.empty(n, dtype=torch.int64, device=dev)
        count = torch.empty(1, dtype=torch.int64, device=dev)
        wsb = g.nms_lane_workspace_size(n)
        ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)

        def call():
            st = g.nms_lane_run(p.data_ptr(), s.data_ptr(), n, thr, 0, keep.data_ptr(), n, count.data_ptr(), 0,
                                ws.data_ptr(), wsb, stream.cuda_stream)
            if st != g.NMS_OK:
                raise g.NmsError(st, "nms_lane_run")

        for _ in range(3):
            call()
        evs = []
        for _ in range(reps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        us = statistics.median(1000 * a.elapsed_time(b) for a, b in evs)
        out[f"lanes_n{n}"] = {"us_median": us, "lane_pairs_per_s": n * (n - 1) / 2 / (us / 1e6),
                              "kept": int(count.item()), "dist_thr": thr}
    return out


def time_matrix(g, torch, wl, dev, flush, decay_thr=0.1, reps=20, decay=0):
    """Device time of one nms_matrix_run call (Gaussian decay with sigma 0.5,
    or the linear decay) on a one-image workload: median, p10, p90 in
    microseconds."""
    stream = torch.cuda.current_stream(dev)
    boxes = torch.from_numpy(wl.boxes).to(dev)
    scores = torch.from_numpy(wl.scores).to(dev)
    n = wl.n
    cap = g.keep_capacity(n, None, wl.max_out)
    keep = torch.empty(max(cap, 1), dtype=torch.int64, device=dev)
    ks = torch.empty(max(cap, 1), dtype=torch.float32, device=dev)
    count = torch.empty(1, dtype=torch.int64, device=dev)
    wsb = g.nms_matrix_workspace_size(n)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    score_thr = -math.inf if wl.score_thr is None else wl.score_thr

    def call():
        st = g.nms_matrix_run(boxes.data_ptr(), scores.data_ptr(), n, decay, 0.5, score_thr, decay_thr, wl.max_out,
                              keep.data_ptr(), ks.data_ptr(), cap, count.data_ptr(), 0, ws.data_ptr(), wsb,
                              stream.cuda_stream)
        if st != g.NMS_OK:
            raise g.NmsError(st, "nms_matrix_run")

    for _ in range(3):
        call()
    evs = []
    for _ in range(reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    us = sorted(1000 * a.elapsed_time(b) for a, b in evs)
    med = statistics.median(us)
    return {"us_median": med, "us_p10": us[len(us) // 10], "us_p90": us[min(len(us) - 1, 9 * len(us) // 10)],
            "boxes_per_s": n / (med / 1e6), "decay_thr": decay_thr, "kept": int(count.item())}


def run_gbnms(args):
    import torch
    import greedy_iou_nms_gb300 as g

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g.build()
    g.load()

    wl = W.make(args.workload, 0)
    if wl.class_ids is not None or wl.batch_offsets is not None:
        raise SystemExit("bench.py times the single-image path; use a single_* or stress_* workload")
    n = wl.n
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    boxes = torch.from_numpy(wl.boxes).to(dev)
    scores = torch.from_numpy(wl.scores).to(dev)
    cap = g.keep_capacity(n, None, wl.max_out)
    keep = torch.empty(max(cap, 1), dtype=torch.int64, device=dev)
    counts = torch.empty(1, dtype=torch.int64, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    ws = g.Workspace(n, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    score_thr = -math.inf if wl.score_thr is None else wl.score_thr

    def step():
        st = g.nms_run(boxes.data_ptr(), scores.data_ptr(), n, 0, 0, 0, 0, wl.iou_thr, score_thr,
                       wl.max_out, keep.data_ptr(), cap, counts.data_ptr(), status.data_ptr(),
                       ws.ptr, ws.bytes, sp)
        if st != g.NMS_OK:
            raise g.NmsError(st, "nms_run")

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    got = keep[: int(counts.item())].cpu().numpy()

    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for e0, e1 in evs:
        flush.fill_(1)
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    total_ms = sum(step_ms)
    clocks = sampler.stop()
    total_ms, value = aggregate_over_ranks(total_ms, world, n, args.steps, device=dev)
    ms_per_step = total_ms / args.steps

    # ---- per-stage durations of the same calls: nms_run_timed records CUDA
    # events on the launching stream between the stages (L2 flushed before
    # each call, as in the timed region).
    stage_t = [[], [], []]
    for it in range(3 + max(args.steps, 50)):  # the first 3 calls are warm-up
        flush.fill_(1)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for e in ev:
            e.record(stream)  # creates the handle; nms_run_timed records it again
        st = g.nms_run_timed(boxes.data_ptr(), scores.data_ptr(), n, 0, 0, 0, 0, wl.iou_thr,
                             score_thr, wl.max_out, keep.data_ptr(), cap, counts.data_ptr(),
                             status.data_ptr(), ws.ptr, ws.bytes, sp, ev)
        if st != g.NMS_OK:
            raise g.NmsError(st, "nms_run_timed")
        torch.cuda.synchronize()
        for k in range(3 if it >= 3 else 0):
            stage_t[k].append(ev[k].elapsed_time(ev[k + 1]))
    sort_ms, mask_ms, resolve_ms = (statistics.mean(t) for t in stage_t)  # average launch duration
    # The mask kernel timed without events between kernels (the roofline's
    # duration; the stage events above each carry the per-event launch delay).
    mask_iso_ms = mask_isolated_ms(g, torch, wl, dev, flush) if wl.max_out <= 0 else mask_ms

    # ---- end to end through the host-memory pipeline, inputs and outputs in
    # pinned host memory and every transfer inside the timed region: by
    # default the kernels move the data across the host link themselves
    # (zero-copy: a copy kernel stages the input into device memory in one
    # pass, the resolve writes the count and the kept indices into the pinned
    # output); for comparison, one host->device copy in and one device->host
    # copy out around nms_run.
    # The events bracket the graph launch (from before the host launches it
    # to the end of its last transfer); the host then reads the result.
    def time_pipe(zero_copy):
        pipe = g.HostPipeline(n, device=dev, zero_copy=zero_copy)
        pipe.load(wl.boxes, wl.scores)
        for _ in range(3):
            pipe.run(wl.iou_thr, wl.score_thr, wl.max_out)
        torch.cuda.synchronize()
        ts, hs = [], []
        for _ in range(args.steps):
            flush.fill_(1)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            a.record(stream)
            pipe.launch(wl.iou_thr, wl.score_thr, wl.max_out)  # the transfers are inside the graph
            b.record(stream)
            res = pipe.result()
            hs.append(1000 * (time.perf_counter() - t0))  # the caller's view: until the result is read
            ts.append(a.elapsed_time(b))
        return (statistics.mean(ts), pipe.in_bytes, pipe.out_bytes(wl.max_out), pipe.zero_copy,
                bool(res.tolist() == got.tolist()), statistics.mean(hs))

    e2e_ms, h2d, d2h, e2e_zc, e2e_parity, e2e_host_ms = time_pipe(True)
    cp_ms, cp_h2d, cp_d2h, _, cp_parity, cp_host_ms = time_pipe(False)
    e2e_parity = e2e_parity and cp_parity

    if rank != 0:
        return 0

    import oracle
    exp = oracle.nms_single(wl.boxes, wl.scores, wl.iou_thr, max_out=wl.max_out)
    parity = bool(got.tolist() == exp.tolist())

    peaks, peak_kind = _peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    alu = measure_alu_peaks(torch, dev)
    fp32_roof = alu["roof_tops"]
    pairs = n * (n - 1) // 2
    m_pairs = mask_pairs(n, wl.max_out)
    mask_tops = OPS_PER_PAIR * m_pairs / (mask_iso_ms / 1000) / 1e12
    Wn = (n + 63) // 64
    mask_bytes = 8 * sum(Wn - i // 64 for i in range(n))  # triangle words written
    n_pairs, n_kept = _graph_size(wl)
    # Algorithmic bytes: sort = read scores and boxes, write perm and sorted
    # boxes; resolve = read the pair list, the neighbour bitmap and perm of the
    # kept, write the int64 keep list.
    sort_bytes = n * (4 + 16 + 4 + 16)
    resolve_bytes = 4 * n_pairs + n // 8 + n_kept * (4 + 8)
    kernels = {"sort_gather_ms": sort_ms, "iou_mask_ms": mask_ms, "resolve_ms": resolve_ms,
               "iou_mask_isolated_ms": mask_iso_ms, "pairs_over_threshold": n_pairs,
               "note": ("stage durations from events recorded between the stages of nms_run_timed; each "
                        "includes the ~5 us launch delay an event between two kernels causes on this platform "
                        "(2.048 us steps); iou_mask_isolated_ms times the mask kernel after an L2 flush with no "
                        "event in between")}
    # The mask is the kernel the roofline reports: the largest stage with the
    # resolve (the two read alike, within the events' 2 us steps) and the
    # kernel whose fraction of its roof is the target.
    dominant = "iou_mask" if mask_ms >= 0.9 * max(resolve_ms, sort_ms) else \
        max(("resolve", resolve_ms), ("sort", sort_ms), key=lambda x: x[1])[0]
    mask_roof = {"kernel": "iou_mask_kernel", "bound": "alu", "achieved": mask_tops,
                 "peak": fp32_roof, "unit": "TFLOP/s", "frac": mask_tops / fp32_roof,
                 "traffic": _ncu_traffic("iou_mask"),
                 "frac_of_best_form": mask_tops / alu["best_form_tops"],
                 "duration_ms": mask_iso_ms,
                 "note": (f"FP32 ops, {OPS_PER_PAIR}/pair x {m_pairs} pairs over the mask kernel's duration "
                          f"after an L2 flush (nms_iou_mask, no event between kernels); peak of "
                          f"measured: the canonical test's {ALU_OPS_PER_PAIR} ALU-pipe + {FMA_OPS_PER_PAIR} "
                          f"FMA-pipe ops at the probed pipe rates ({alu['roof_bound']}-bound, "
                          f"{alu['roof_pairs_per_clk_per_sm']:.2f} pairs/clk/SM) x {alu['sm_count']} SMs x "
                          f"{alu['probe_mhz']:.0f} MHz; frac_of_best_form is against the fastest probed form "
                          f"({alu['best_form']}, {alu['best_form_tops']:.1f} Tops/s)")}
    if dominant == "iou_mask":
        roof = mask_roof
    else:
        name, ms, nbytes = (("resolve_single_kernel", resolve_ms, resolve_bytes) if dominant == "resolve"
                            else ("bucket_rank_kernel", sort_ms, sort_bytes))
        ach = nbytes / (ms / 1000) / 1e9
        note = f"algorithmic bytes {nbytes}; peak of {peak_kind} (HBM copy)"
        if dominant == "resolve":
            note += ("; the resolve runs on one SM by design (dependency rounds over the pair list in "
                     "shared memory), so its time is set by round latency, not by HBM")
        roof = {"kernel": name, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "traffic": _ncu_traffic(dominant), "note": note}

    per_config = fast_nms = matrix_nms = matrix_lin = front_end = lanes = None
    summary = None
    if not args.no_configs:
        per_config, fast_nms, matrix_nms, matrix_lin = {}, {}, {}, {}
        sections = set(args.sections.split(","))
        names = list(W.CONFIGS) if args.configs == "all" else args.configs.split(",")
        for name in names:
            wl_c = W.make(name, 0)
            if "greedy" in sections:
                per_config[name] = time_workload(g, torch, wl_c, dev, flush)
            if "fast" in sections:
                fast_nms[name] = time_workload(g, torch, wl_c, dev, flush, fast=True)
            if "matrix" in sections and wl_c.class_ids is None and wl_c.batch_offsets is None:
                matrix_nms[name] = time_matrix(g, torch, wl_c, dev, flush)
                matrix_lin[name] = time_matrix(g, torch, wl_c, dev, flush, decay=g.NMS_DECAY_LINEAR)
        if "front_end" in sections:
            front_end = time_front_end(g, torch, dev, flush)
        if "lanes" in sections:
            lanes = time_lanes(g, torch, dev, flush)
        summary = greedy_summary(per_config, fp32_roof, hbm)

    cpu = None
    cpu_all = None
    if not args.no_cpu_baseline:
        v, reps_cpu, secs = cpu_oracle_run(wl, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{reps_cpu} full runs of {wl.name} in {secs:.1f} s",
               "cpu_model": cpu_model(), "host_cores": os.cpu_count()}
        va, reps_a, secs_a, threads = cpu_all_cores_run(wl, min(args.cpu_seconds, 5.0))
        cpu_all = {"value": va, "unit": UNIT, "cores": threads, "kind": "all-core bitmask baseline (OpenMP)",
                   "sample": f"{reps_a} full runs of {wl.name} in {secs_a:.1f} s", "cpu_model": cpu_model(),
                   "host_cores": os.cpu_count()}

    alu_brief = {"sm_count": alu["sm_count"], "probe_mhz": round(alu["probe_mhz"], 1),
                 "roof_tops": round(fp32_roof, 3), "roof_bound": alu["roof_bound"],
                 "lane_ops_per_clk_per_sm": {k: round(v["lane_ops_per_clk_per_sm"], 1)
                                             for k, v in alu["forms"].items()}}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": bench_config(wl, world),
        "alu_peaks": alu,
        "fast_nms_per_config": fast_nms,
        "front_end": front_end,
        "lane_nms": lanes,
        "matrix_nms_per_config": matrix_nms,
        "matrix_nms_linear_per_config": matrix_lin,
        "per_config": per_config,
        "e2e_with_copies": {"value": n / (cp_ms / 1000), "unit": UNIT, "h2d_bytes_per_step": cp_h2d,
                            "d2h_bytes_per_step": cp_d2h, "ms_per_step": cp_ms, "host_ms_per_step": cp_host_ms},
        "kernels": kernels,
        "us_per_call": 1000 * ms_per_step,
        "gpairs_per_s": pairs / (ms_per_step / 1000) / 1e9,
        "mask_gpairs_per_s": m_pairs / (mask_iso_ms / 1000) / 1e9,
        "mask_gbs": mask_bytes / (mask_iso_ms / 1000) / 1e9,
        "mask_hbm_frac": mask_bytes / (mask_iso_ms / 1000) / 1e9 / hbm,
        "cpu_baseline": cpu,
        "e2e": {"value": n / (e2e_ms / 1000), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "host_ms_per_step": e2e_host_ms,
                "transfer": ("zero-copy: a copy kernel stages the pinned input into device memory in one "
                             "pass; the resolve writes the count and the kept indices into the pinned output"
                             if e2e_zc else "copies")},
        "gpu_launches": 3 * args.steps,  # sort, mask, resolve per call at this size
        "parity_vs_oracle": parity and e2e_parity,
        "peaks": {"hbm": peak_kind, "fp32": "measured (probe in this run)"},
        # Last, so that a reader keeping only the end of the line has them.
        "roofline": roof,
        "roofline_iou_mask": mask_roof,
        "alu_roof": alu_brief,
        "cpu_baseline_all_cores": cpu_all,
        "per_config_greedy": summary,
        "clocks": clocks,
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def greedy_summary(per_config, fp32_roof, hbm):
    """Compact per-workload table of nms_run: median us per call, M boxes/s,
    the stages' us (events between the stages: each carries the per-event
    launch delay), and for the mask the kernel's own us after an L2 flush
    (workloads without max_out; with max_out the first mask launch's stage
    time), its G pairs/s, fraction of the FP32 op roof and GB/s of written
    triangle words."""
    out = {}
    for name, r in per_config.items():
        row = {"us": round(r["us_median"], 1), "Mboxes_s": round(r["boxes_per_s"] / 1e6, 1)}
        st = r.get("stages_us")
        if st and "mask" in st:
            n = r["n"]
            m_us = r.get("mask_isolated_us", st["mask"])
            k = int(round((1 + math.sqrt(1 + 8 * r["mask_pairs"])) / 2))  # boxes of the first mask launch
            wn = (n + 63) // 64
            words = sum(wn - i // 64 for i in range(k))
            row.update({"sort_us": round(st["sort"], 1), "mask_stage_us": round(st["mask"], 1),
                        "mask_us": round(m_us, 1),
                        "mask_Gpairs_s": round(r["mask_pairs"] / m_us / 1e3, 1),
                        "mask_frac": round(OPS_PER_PAIR * r["mask_pairs"] / (m_us / 1e6) / 1e12 / fp32_roof, 3),
                        "mask_GBs": round(8 * words / m_us / 1e3, 1), "resolve_us": round(st["resolve"], 1)})
        elif st:
            row.update({k: round(v, 1) for k, v in st.items()})
        out[name] = row
    return out


def cpu_model():
    """The host CPU's model string (/proc/cpuinfo, or lscpu on Arm hosts whose
    cpuinfo has no model name)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


KERNEL_SOURCES = {"iou_mask": "k_mask.cu", "resolve": "k_resolve.cu", "sort": "k_sort.cu"}


def kernel_source_sha(kernel):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "greedy_iou_nms_gb300", "csrc")
    for name in (KERNEL_SOURCES[kernel], "common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _ncu_traffic(kernel):
    """DRAM bytes per launch of `kernel` (dram__bytes_read.sum + write.sum) from
    the committed ncu summary, or None when absent or when the kernel source
    changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("src_sha") != kernel_source_sha(kernel):
        return None
    return d.get("bytes_per_launch")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gbnms", choices=["gbnms", "reference"])
    ap.add_argument("--workload", default=W.HEADLINE)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config timing table")
    ap.add_argument("--configs", default="all",
                    help="comma-separated workload names for the per-config tables (default: all)")
    ap.add_argument("--sections", default="greedy,fast,matrix,front_end,lanes",
                    help="per-config tables to time: greedy, fast, matrix, front_end, lanes")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gbnms(args)


if __name__ == "__main__":
    sys.exit(main())
